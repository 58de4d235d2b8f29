"""The range-checked build (-DULYSSES_CHECK_BOUNDS: every plain global load
and store checked against its buffer) runs the whole path without a single
failed check and gives bit for bit what the normal build gives: forward,
backward (two-kernel, dS-store, and dS-store in kv-head chunks), the workspace-free backward, the fp32 forward, replicated kv-heads,
the ring hybrid, the folded forward and backward and the two projections.  The checked library runs in a
child process (ULYSSES_LIB)."""
import os
import subprocess
import sys

import pytest
import torch

from ulysses_sequence_attention_seq_gb300 import build as B

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Runs every case with whichever library ULYSSES_LIB names; saves the outputs
# and the status words to the file given as argv[1].
CHILD = r'''
import os, sys
sys.path.insert(0, os.environ["ULYSSES_ROOT"]); sys.path.insert(0, os.path.join(os.environ["ULYSSES_ROOT"], "tests"))
import torch
from pathcheck import GpuRun
from test_gpu_forward import wl
from ulysses_sequence_attention_seq_gb300 import binding as U
cases = [wl(2, 1, 424, 4, 2, 128).with_(backward=True),
         wl(4, 2, 512, 8, 8, 64, causal=False).with_(backward=True),
         wl(8, 1, 1024, 8, 2, 128).with_(backward=True),
         wl(8, 1, 1024, 4, 4, 128).with_(ring=4, backward=True),
         wl(2, 1, 256, 4, 4, 32, "fp32", causal=False, rope=False)]
out = {}
for n, w in enumerate(cases):
    run = GpuRun(w, backward=w.backward, ds=w.backward)
    run.forward()
    names = ["o_seq", "lse"]
    if w.backward:
        run.backward()
        names += ["dq_seq", "dk_seq", "dv_seq"]
    for name in names:
        out[f"{n}/{name}"] = getattr(run.buf, name).cpu()
    out[f"{n}/status"] = torch.tensor(U.ulysses_read_status(run.buf.ws))
    if w.backward:  # the dS-store backward on the same buffers (its tile store written and read back)
        run.buf.backward_ds()
        for name in ("dq_seq", "dk_seq", "dv_seq"):
            out[f"{n}/ds/{name}"] = getattr(run.buf, name).cpu()
        out[f"{n}/ds/status"] = torch.tensor(U.ulysses_read_status(run.buf.ws))
        # and in kv-head chunks, one kv-head's tiles at a time (a phase-4 workspace)
        b = run.buf
        ws4 = torch.empty(U.ulysses_workspace_bytes(run.prob, 4), dtype=torch.uint8, device="cuda")
        U.ulysses_workspace_init(run.prob, ws4)
        U.ulysses_attn_bwd_ds(run.prob, b.q_head, b.k_head, b.v_head, b.o_head, b.lse, b.do_seq, b.dq_seq,
                              b.dk_seq, b.dv_seq, ws4)
        torch.cuda.synchronize()
        for name in ("dq_seq", "dk_seq", "dv_seq"):
            out[f"{n}/ds4/{name}"] = getattr(b, name).cpu()
        out[f"{n}/ds4/status"] = torch.tensor(U.ulysses_read_status(ws4))
    if n == 0:  # the workspace-free backward on the same buffers
        b = run.buf
        grads = [torch.empty_like(getattr(b, g)) for g in ("dq_seq", "dk_seq", "dv_seq")]
        U.ulysses_attn_bwd_noalloc(run.prob, b.q_head, b.k_head, b.v_head, b.o_head, b.lse, b.do_seq, *grads)
        for g, t in zip(("dq_seq", "dk_seq", "dv_seq"), grads):
            out[f"noalloc/{g}"] = t.cpu()
        out["noalloc/status"] = torch.tensor(U.ulysses_noalloc_read_status())
# the folded forward and backward (RoPE off, S/P = 256, kv-heads replicated)
w = wl(8, 1, 2048, 16, 2, 128, rope=False).with_(backward=True)
run = GpuRun(w, backward=True)
b = run.buf
U.ulysses_attn_fwd_folded(run.prob, b.q_seq, b.k_seq, b.v_seq, b.o_seq, b.lse, b.ws)
U.ulysses_attn_bwd_folded(run.prob, b.q_seq, b.k_seq, b.v_seq, b.o_seq, b.lse, b.do_seq,
                          b.dq_seq, b.dk_seq, b.dv_seq, b.ws)
torch.cuda.synchronize()
for name in ("o_seq", "lse", "dq_seq", "dk_seq", "dv_seq"):
    out[f"fold/{name}"] = getattr(b, name).cpu()
out["fold/status"] = torch.tensor(U.ulysses_read_status(b.ws))
# the projections (QKV with pack and RoPE; output with unpack)
w = wl(2, 1, 512, 4, 2, 128)
prob = U.Problem.from_workload(w)
g = torch.Generator(device="cuda").manual_seed(3)
x = torch.randn(w.P, w.B, w.Sl, w.hidden, generator=g, device="cuda").to(torch.bfloat16)
n_out = (w.n_head + 2 * w.n_kv_head) * w.head_dim
wq = (torch.randn(n_out, w.hidden, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
bq = torch.randn(n_out, generator=g, device="cuda").to(torch.bfloat16)
buf = U.Buffers(prob)
U.ulysses_workspace_init(prob, buf.ws)
U.ulysses_qkv_proj_pack(prob, x, wq, bq, buf.q_head, buf.k_head, buf.v_head, buf.ws)
wo = (torch.randn(w.hidden, w.hidden, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
y = torch.empty(w.P, w.B, w.Sl, w.hidden, dtype=torch.bfloat16, device="cuda")
U.ulysses_out_proj_unpack(prob, buf.q_head, wo, None, y, buf.ws)
torch.cuda.synchronize()
for name in ("q_head", "k_head", "v_head"):
    out[f"proj/{name}"] = getattr(buf, name).cpu()
out["proj/y"] = y.cpu()
out["proj/status"] = torch.tensor(U.ulysses_read_status(buf.ws))
torch.save(out, sys.argv[1])
'''


def _run(lib, path):
    env = dict(os.environ, ULYSSES_LIB=lib, ULYSSES_ROOT=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD, path], env=env, capture_output=True, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    return torch.load(path)


def test_checked_build_is_clean_and_identical(tmp_path):
    checked = B.build(checked=True)
    normal = B.build()
    got = _run(checked, str(tmp_path / "checked.pt"))
    want = _run(normal, str(tmp_path / "normal.pt"))
    assert got.keys() == want.keys()
    for k in got:
        if k.endswith("status"):
            assert int(got[k]) == 0, (k, int(got[k]))   # no failed range check, no timeout
        else:
            assert torch.equal(got[k], want[k]), k
