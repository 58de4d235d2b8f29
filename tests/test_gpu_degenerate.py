"""The path's degenerate sizes on the GPU, against the fp64 oracle through the
C ABI: one token per rank (S = P), shards of an odd length (S not a multiple
of 4, so the backward's per-row delta / LSE rows are padded to 16 bytes in the
workspace), a shard length just past one tile, and a single token, where
attention has a closed form (O = V, LSE = the one score, dV = dO); the
backward in each of its three modes."""
import numpy as np
import pytest
import torch

import test_gpu_backward as BWD
import test_gpu_ds as DS
import test_gpu_forward as FWD
from pathcheck import GpuRun, to64
from test_gpu_forward import wl

pytestmark = pytest.mark.gpu

CASES = [wl(8, 1, 8, 8, 8, 64),                   # S = P: one token per rank
         wl(4, 2, 4, 8, 2, 128),                  # S = P, B = 2, kv-heads replicated (R = 2)
         wl(2, 1, 6, 4, 2, 128),                  # Sl = 3
         wl(2, 1, 202, 4, 4, 64, causal=False),   # Sl = 101, one ragged tile
         wl(3, 1, 387, 3, 3, 128)]                # Sl = 129, S = 3 tiles + 3 rows


@pytest.mark.parametrize("w", CASES, ids=BWD._ids)
def test_forward_at_degenerate_sizes(w):
    FWD.test_forward_matches_oracle(w)


@pytest.mark.parametrize("w", CASES, ids=BWD._ids)
def test_backward_at_degenerate_sizes(w):
    BWD.test_backward_matches_oracle(w)


@pytest.mark.parametrize("w", CASES, ids=BWD._ids)
def test_every_backward_mode_at_degenerate_sizes(w):
    """The two-kernel, dS-store and fused backwards against the oracle, dK and
    dV identical across the three."""
    DS.test_tiny_sequences_every_backward_mode(w)


def test_fp32_forward_one_token_per_rank():
    FWD.test_forward_matches_oracle(wl(2, 1, 2, 2, 2, 32, "fp32"))


def test_single_token_has_the_closed_form():
    """S = 1 (P = 1, one head): the softmax over one key is 1, so O = V and
    dV = dO bit for bit (a product by 1 + O(1e-7), rounded back to bf16), LSE
    is the scaled score q.k / sqrt(D) (RoPE at position 0 is the identity),
    and dS = P (dP - delta) vanishes up to rounding, and with it dQ and dK."""
    w = wl(1, 1, 1, 1, 1, 64).with_(backward=True)
    run = GpuRun(w, backward=True, ds=True, fused=True)
    run.forward()
    b = run.buf
    assert torch.equal(b.o_seq.flatten(), b.v_seq.flatten())
    q, k = to64(b.q_seq).reshape(-1), to64(b.k_seq).reshape(-1)
    want = float(q @ k) / np.sqrt(w.head_dim)
    assert abs(float(to64(b.lse).reshape(-1)[0]) - want) <= 1e-3 * (1 + abs(want))
    for call in (run.backward, run.backward_ds, run.backward_fused):
        for t in (b.dq_seq, b.dk_seq, b.dv_seq):
            t.fill_(float("nan"))
        call()
        assert torch.equal(b.dv_seq.flatten(), b.do_seq.flatten())
        assert b.dq_seq.float().abs().max() <= 1e-2 and b.dk_seq.float().abs().max() <= 1e-2
