"""bench.py's CPU legs, no GPU: the reference arm prints the contract's JSON
line (the fp64 oracle timed on the host), and the oracle leg runs the ring
hybrid's steps for a hybrid workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "C2",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] >= 3
    assert d["config"]["workload"] == "C2"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_oracle_leg_runs_the_ring_hybrid():
    sys.path.insert(0, ROOT)
    import bench
    from ulysses_sequence_attention_seq_gb300.synthetic import WORKLOADS
    w = WORKLOADS["C2"].with_(name="C2-ring", P=8, ring=2, n_head=16, n_kv_head=16)
    ob = bench.OracleBench(w, nthreads=2)
    t_full, n_rows, pairs, wall = ob.step(8)
    assert t_full > 0 and 0 < n_rows <= 8 and pairs > 0 and wall > 0
    assert "2 ring positions" in ob.describe(n_rows)


def test_pack_bytes_count_replicas_within_an_all_to_all_group():
    """K and V are written once per replica only when there are fewer
    kv-heads than ranks in one All-to-All group (P / ring ranks): the ring
    hybrid at P = 256 with 32 kv-heads replicates nothing, C4 with 4 kv-heads
    writes each kv-head to 2 ranks."""
    sys.path.insert(0, ROOT)
    import bench
    from ulysses_sequence_attention_seq_gb300.synthetic import EXTRA_WORKLOADS, WORKLOADS
    c4 = WORKLOADS["C4"]
    per_head = c4.B * c4.S * c4.head_dim * 2            # one bf16 head over the sequence
    assert bench.permute_bytes(c4, 2) == 6 * 32 * per_head
    assert bench.permute_bytes(EXTRA_WORKLOADS["C4-ring8"], 2) == 6 * 32 * per_head
    kv4 = EXTRA_WORKLOADS["C4-kv4"]
    assert bench.permute_bytes(kv4, 2) == per_head * (2 * 32 + 2 * 4 + 2 * 8)
