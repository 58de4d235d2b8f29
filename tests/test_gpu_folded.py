"""Folded forward and backward (ulysses_attn_fwd_folded, ulysses_attn_bwd_folded):
the attention kernels read the sequence-sharded Q/K/V (and dO) directly and
write O (and dQ, dK, dV) in sequence layout, so every All-to-All becomes
addressing.  They must reproduce the packed path bit for bit, and the fp64
oracle within the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
from pathcheck import GpuRun, assert_close, assert_lse_close, oracle_inputs, oracle_problem, to64
from test_gpu_forward import wl
from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300.synthetic import WORKLOADS

pytestmark = pytest.mark.gpu

CASES = [wl(2, 1, 512, 4, 2, 128, rope=False),          # Sl = 256, GQA
         wl(4, 2, 1024, 8, 8, 64, rope=False),          # D = 64, B = 2
         wl(8, 1, 2048, 32, 8, 128, rope=False),        # the GQA workload's head layout
         wl(2, 1, 256, 4, 4, 128, causal=False, rope=False),   # Sl = 128, non-causal
         wl(4, 1, 1536, 4, 4, 128, rope=False)]         # odd number of 128-row tiles


def _folded(run):
    b = run.buf
    o = torch.full_like(b.o_seq, float("nan"))
    lse = torch.full_like(b.lse, float("nan"))
    U.ulysses_attn_fwd_folded(run.prob, b.q_seq, b.k_seq, b.v_seq, o, lse, b.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(b.ws) == 0
    return o, lse


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"P{w.P}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}{'c' if w.causal else 'n'}")
def test_folded_equals_pack_attend_unpack_bit_exact(w):
    run = GpuRun(w)
    run.forward()
    o, lse = _folded(run)
    assert torch.equal(o, run.buf.o_seq)
    assert torch.equal(lse, run.buf.lse)


def test_folded_matches_oracle():
    w = CASES[0]
    run = GpuRun(w)
    o, lse = _folded(run)
    x = oracle_inputs(run.inputs)
    want = oracle.forward(oracle_problem(w), x["q"], x["k"], x["v"])
    assert_close(to64(o), np.stack([a.reshape(w.B, w.Sl, -1) for a in want["o_seq"]]), w, "folded o_seq")
    assert_lse_close(to64(lse), np.stack(want["lse"]), w, "folded lse")


def test_folded_full_size_pages_sizing_without_rope():
    """The pages' sizing (P=8, S=32768, 32 heads, D=128) with pre-rotated q/k."""
    w = WORKLOADS["C4"].with_(use_rope=False)
    run = GpuRun(w)
    run.forward()
    o, lse = _folded(run)
    assert torch.equal(o, run.buf.o_seq)
    assert torch.equal(lse, run.buf.lse)


def test_folded_refuses_what_it_cannot_fold():
    run = GpuRun(wl(2, 1, 512, 4, 2, 128, rope=True))
    b = run.buf
    with pytest.raises(U.UlyssesError) as e:      # RoPE must be applied by the producer
        U.ulysses_attn_fwd_folded(run.prob, b.q_seq, b.k_seq, b.v_seq, b.o_seq, b.lse, b.ws)
    assert e.value.code == -4
    run = GpuRun(wl(2, 1, 200, 4, 2, 128, rope=False))   # Sl = 100: tiles would straddle ranks
    b = run.buf
    with pytest.raises(U.UlyssesError) as e:
        U.ulysses_attn_fwd_folded(run.prob, b.q_seq, b.k_seq, b.v_seq, b.o_seq, b.lse, b.ws)
    assert e.value.code == -4


def test_folded_with_replicated_kv_heads_equals_three_calls():
    """KV-head replication in the folded forward: rank r's K/V tiles come from
    kv-head r / R of the sequence-sharded buffers."""
    w = wl(8, 1, 2048, 16, 2, 128, rope=False)
    run = GpuRun(w)
    run.forward()
    o3, l3 = run.buf.o_seq.clone(), run.buf.lse.clone()
    run.buf.o_seq.zero_()
    b = run.buf
    U.ulysses_attn_fwd_folded(run.prob, b.q_seq, b.k_seq, b.v_seq, b.o_seq, b.lse, b.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(b.ws) == 0
    assert torch.equal(b.o_seq, o3) and torch.equal(b.lse, l3)


# ------------------------------------------------------------ folded backward

BWD_CASES = CASES + [wl(8, 1, 2048, 16, 2, 128, rope=False)]   # kv-heads replicated (R = 4)


def _folded_bwd(run):
    b = run.buf
    outs = {n: torch.full_like(getattr(b, n), float("nan")) for n in ("dq_seq", "dk_seq", "dv_seq")}
    U.ulysses_attn_bwd_folded(run.prob, b.q_seq, b.k_seq, b.v_seq, b.o_seq, b.lse, b.do_seq,
                              outs["dq_seq"], outs["dk_seq"], outs["dv_seq"], b.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(b.ws) == 0
    return outs


@pytest.mark.parametrize("w", BWD_CASES, ids=lambda w: f"P{w.P}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}{'c' if w.causal else 'n'}")
def test_folded_backward_equals_the_packed_backward_bit_exact(w):
    """The dK/dV and dQ kernels read the same tiles through the sequence-layout
    maps as through the packed buffers, and delta is formed from the same O and
    dO values in the same order: every gradient bit for bit."""
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True)
    run.forward()
    run.backward()
    outs = _folded_bwd(run)
    for n, t in outs.items():
        assert torch.equal(t, getattr(run.buf, n)), n


def test_folded_backward_matches_oracle():
    w = CASES[0].with_(backward=True)
    run = GpuRun(w, backward=True)
    o, lse = _folded(run)
    run.buf.o_seq.copy_(o)
    run.buf.lse.copy_(lse)
    outs = _folded_bwd(run)
    x = oracle_inputs(run.inputs)
    want = oracle.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"])
    for n in ("dq_seq", "dk_seq", "dv_seq"):
        assert_close(to64(outs[n]), np.stack(want[n]), w, "folded " + n)


def test_folded_backward_full_size_pages_sizing_without_rope():
    w = WORKLOADS["C4"].with_(use_rope=False, backward=True)
    run = GpuRun(w, backward=True)
    run.forward()
    run.backward()
    outs = _folded_bwd(run)
    for n, t in outs.items():
        assert torch.equal(t, getattr(run.buf, n)), n


@pytest.mark.parametrize("w", [wl(2, 1, 512, 4, 2, 128, rope=True),          # RoPE must be applied by the producer
                               wl(2, 1, 200, 4, 2, 128, rope=False),         # Sl = 100: tiles would straddle ranks
                               wl(8, 1, 1024, 4, 4, 128, rope=False).with_(ring=4)])   # no hybrid form
def test_folded_backward_refuses_what_it_cannot_fold(w):
    run = GpuRun(w.with_(backward=True), backward=True)
    b = run.buf
    with pytest.raises(U.UlyssesError) as e:
        U.ulysses_attn_bwd_folded(run.prob, b.q_seq, b.k_seq, b.v_seq, b.o_seq, b.lse, b.do_seq,
                                  b.dq_seq, b.dk_seq, b.dv_seq, b.ws)
    assert e.value.code == -4
