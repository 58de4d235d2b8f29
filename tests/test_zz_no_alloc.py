"""The workspace-free backward (ulysses_attn_bwd_noalloc), through the C ABI.

It serves callers that cannot allocate device memory (their allocator is owned
by someone else, or they must not call cudaMalloc on this path): its scratch
is the library's fixed 32 MiB device array.  It runs the very kernels of the
ordinary backward (which takes a caller workspace) on the same inputs, so its
gradients must equal that backward's bit for bit, on two calls in a row, with
the array's status word clear after each.  Problems the backward would refuse,
or too large for the fixed array, must be refused up front.  This file sorts
last so that a run stopping at the first failure has run everything else.
"""
import dataclasses

import pytest
import torch

from pathcheck import GpuRun
from test_gpu_forward import wl
from ulysses_sequence_attention_seq_gb300 import binding as U

pytestmark = pytest.mark.gpu

GRADS = ("dq_seq", "dk_seq", "dv_seq")


def _noalloc(run, outs):
    b = run.buf
    U.ulysses_attn_bwd_noalloc(run.prob, b.q_head, b.k_head, b.v_head, b.o_head, b.lse, b.do_seq, *outs)


@pytest.mark.parametrize("w", [wl(2, 1, 424, 4, 2, 128), wl(4, 1, 512, 8, 8, 64, causal=False),
                               wl(4, 1, 512, 8, 8, 64, causal=False, rope=False)],
                         ids=["P2S424gqaD128", "P4S512D64nc", "P4S512D64nc-norope"])
def test_noalloc_backward_equals_workspace_backward_twice(w):
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True)
    run.forward()
    run.backward()                       # the ordinary entry point, caller workspace
    ref = [getattr(run.buf, n).clone() for n in GRADS]
    for _ in range(2):                   # two calls in a row share the fixed array
        outs = [torch.full_like(getattr(run.buf, n), float("nan")) for n in GRADS]
        _noalloc(run, outs)
        assert U.ulysses_noalloc_read_status() == 0   # waits for the stream
        for got, want, name in zip(outs, ref, GRADS):
            assert torch.equal(got, want), f"noalloc {name} differs from the workspace backward"


def test_noalloc_refuses_problems_beyond_its_scratch():
    p = U.Problem(B=1, S=32768, hidden=4096, n_head=32, n_kv_head=32, head_dim=128, P=8)
    assert U.ulysses_workspace_bytes(p, 1) > 32 << 20
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(U.UlyssesError) as e:
        U.ulysses_attn_bwd_noalloc(p, dummy, dummy, dummy, dummy, lse, dummy, dummy, dummy, dummy)
    assert e.value.code == -7


def test_noalloc_refuses_what_the_backward_refuses():
    """An fp32 problem (no backward kernel) and aliased outputs are refused with
    the ordinary backward's codes, and the array is left as the last call left it."""
    w = wl(2, 1, 256, 4, 4, 64).with_(backward=True)
    run = GpuRun(w, backward=True)
    run.forward()
    b = run.buf
    outs = [torch.empty_like(getattr(b, n)) for n in GRADS]
    pf = dataclasses.replace(run.prob, dtype=U.FP32)
    with pytest.raises(U.UlyssesError) as e:
        U.ulysses_attn_bwd_noalloc(pf, b.q_head, b.k_head, b.v_head, b.o_head, b.lse, b.do_seq, *outs)
    assert e.value.code == -4
    with pytest.raises(U.UlyssesError) as e:   # dK written over dQ
        U.ulysses_attn_bwd_noalloc(run.prob, b.q_head, b.k_head, b.v_head, b.o_head, b.lse, b.do_seq,
                                   outs[0], outs[0], outs[2])
    assert e.value.code == -6
    _noalloc(run, outs)
    assert U.ulysses_noalloc_read_status() == 0
