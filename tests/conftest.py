import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity margins of this run: every comparison the GPU tests made against
    the oracle (tests/pathcheck.py), the tightest first; all of them as JSON in
    the file named by ULYSSES_PARITY_LOG when that variable is set."""
    pc = sys.modules.get("pathcheck")
    recs = list(getattr(pc, "RECORDS", []) or [])
    if not recs:
        return
    recs.sort(key=lambda r: -r["worst_frac_of_bound"])
    tr = terminalreporter
    tr.write_sep("-", f"parity margins ({len(recs)} comparisons; worst element as a fraction of its bound)")
    for r in recs[:12]:
        rel = "" if r["rel_l2"] is None else f" rel-L2 {r['rel_l2']:.2e}"
        tr.write_line(f"{r['worst_frac_of_bound']:.3f}  max-abs {r['max_abs']:.3e}{rel}  {r['kind']}  "
                      f"{r['what']}  {r['test']}")
    path = os.environ.get("ULYSSES_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            json.dump(recs, f, indent=1)
