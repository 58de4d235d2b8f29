"""The workspace-free backward (ulysses_attn_bwd_noalloc), through the C ABI.

It serves callers that cannot allocate device memory (their allocator is owned
by someone else, or they must not call cudaMalloc on this path): its scratch
is the library's fixed 32 MiB device array.  Its results must match the
ordinary backward (which takes a caller workspace) on two calls in a row, and
a problem too large for the fixed array must be refused up front.  This file
sorts last so that a run stopping at the first failure has run everything else.
"""
import numpy as np
import pytest
import torch

from pathcheck import GpuRun, assert_close, to64
from test_gpu_forward import wl
from ulysses_sequence_attention_seq_gb300 import binding as U

pytestmark = pytest.mark.gpu


def _noalloc(run, outs):
    b = run.buf
    U.ulysses_attn_bwd_noalloc(run.prob, b.q_head, b.k_head, b.v_head, b.o_head, b.lse, b.do_seq, *outs)


@pytest.mark.parametrize("w", [wl(2, 1, 424, 4, 2, 128), wl(4, 1, 512, 8, 8, 64, causal=False)],
                         ids=["P2S424gqaD128", "P4S512D64nc"])
def test_noalloc_backward_matches_workspace_backward_twice(w):
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True)
    run.forward()
    run.backward()                       # the ordinary entry point, caller workspace
    ref = [to64(getattr(run.buf, n)) for n in ("dq_seq", "dk_seq", "dv_seq")]
    for _ in range(2):                   # two calls in a row share the fixed array
        outs = [torch.full_like(getattr(run.buf, n), float("nan")) for n in ("dq_seq", "dk_seq", "dv_seq")]
        _noalloc(run, outs)
        torch.cuda.synchronize()
        for got, want, name in zip(outs, ref, ("dq", "dk", "dv")):
            assert_close(to64(got), want, w, f"noalloc {name}")


def test_noalloc_refuses_problems_beyond_its_scratch():
    p = U.Problem(B=1, S=32768, hidden=4096, n_head=32, n_kv_head=32, head_dim=128, P=8)
    assert U.ulysses_workspace_bytes(p, 1) > 32 << 20
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(U.UlyssesError) as e:
        U.ulysses_attn_bwd_noalloc(p, dummy, dummy, dummy, dummy, lse, dummy, dummy, dummy, dummy)
    assert e.value.code == -7
