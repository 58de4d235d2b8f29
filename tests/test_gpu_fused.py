"""GPU parity of the fused backward (ulysses_attn_bwd_fused: dQ accumulated in
the dK/dV loop by reduce-adds into a float workspace accumulator) through the
C ABI: dQ against the fp64 oracle under the same bar as every other gradient;
dK and dV bit-identical to the two-kernel backward (the same products in the
same order); two calls in a row (each zeroes the accumulator first); the three
steps equal the composed call; the full-size workloads on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from pathcheck import GpuRun, assert_close, oracle_inputs, oracle_problem, to64
from test_gpu_backward import BWD_CASES, REP_BWD_CASES, _ids
from test_gpu_forward import sample_rows, wl
from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300.synthetic import EXTRA_WORKLOADS, WORKLOADS

pytestmark = pytest.mark.gpu

GRADS = ("dq_seq", "dk_seq", "dv_seq")
CASES = BWD_CASES + REP_BWD_CASES + [wl(8, 1, 1024, 8, 2, 128).with_(ring=2)]


def _fused_ids(w):
    return _ids(w) + (f"R{w.ring}" if w.ring > 1 else "")


@pytest.mark.parametrize("w", CASES, ids=_fused_ids)
def test_fused_backward_matches_oracle_and_two_kernel_backward(w):
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True, fused=True)
    run.forward()
    run.backward()                                   # the two-kernel backward
    ref = {n: getattr(run.buf, n).clone() for n in GRADS}
    x = oracle_inputs(run.inputs)
    if w.ring > 1:
        from oracle import ring as oracle_ring
        want = oracle_ring.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"])
    else:
        want = oracle.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"])
    for _ in range(2):                               # each call zeroes the accumulator before adding
        for n in GRADS:
            getattr(run.buf, n).fill_(float("nan"))
        run.backward_fused()
        assert torch.equal(run.buf.dk_seq, ref["dk_seq"]), "fused dK differs from the two-kernel backward"
        assert torch.equal(run.buf.dv_seq, ref["dv_seq"]), "fused dV differs from the two-kernel backward"
        assert_close(to64(run.buf.dq_seq), np.stack(want["dq_seq"]), w, "fused dq_seq")


def test_fused_steps_equal_composed_call():
    """prepare + dkdvq + dq_finish give what ulysses_attn_bwd_fused gives
    (dQ to float-summation order: within one bf16 ulp; dK, dV exactly)."""
    w = WORKLOADS["C3"].with_(S=1024)
    run = GpuRun(w, backward=True, fused=True)
    run.forward()
    run.backward_fused()
    b = run.buf
    ref = [t.clone() for t in (b.dq_seq, b.dk_seq, b.dv_seq)]
    for t in (b.dq_seq, b.dk_seq, b.dv_seq):
        t.zero_()
    U.ulysses_attn_bwd_prepare(run.prob, b.o_head, b.lse, b.do_seq, b.ws)
    U.ulysses_attn_bwd_dkdvq(run.prob, b.q_head, b.k_head, b.v_head, b.dk_seq, b.dv_seq, b.ws)
    U.ulysses_attn_bwd_dq_finish(run.prob, b.dq_seq, b.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(b.ws) == 0
    assert torch.equal(b.dk_seq, ref[1]) and torch.equal(b.dv_seq, ref[2])
    d = (b.dq_seq.float() - ref[0].float()).abs()
    ulp = torch.exp2(torch.floor(torch.log2(ref[0].float().abs().clamp_min(2.0 ** -126))) - 7)
    assert bool((d <= ulp).all()), "dQ of the steps differs from the composed call by more than one bf16 ulp"


def test_fused_backward_needs_a_phase2_workspace():
    w = wl(2, 1, 256, 4, 4, 64).with_(backward=True)
    run = GpuRun(w, backward=True)                   # phase-1 workspace
    run.forward()
    with pytest.raises(U.UlyssesError) as e:
        run.buf.backward_fused()
    assert e.value.code == -7


@pytest.mark.parametrize("name", ["C3", "C4", "C4-kv4"])
def test_fused_backward_workloads(name):
    """Full size, in the bench's launch configuration: dQ of every q-head on
    sampled rows (shard/tile boundaries and seeded random rows, each exact
    over its full key range) against the oracle; dK and dV equal to the
    two-kernel backward's."""
    w = WORKLOADS[name] if name in WORKLOADS else EXTRA_WORKLOADS[name]
    run = GpuRun(w, backward=True, fused=True)
    run.forward()
    run.backward()
    ref = {n: getattr(run.buf, n).clone() for n in ("dk_seq", "dv_seq")}
    run.backward_fused()
    assert torch.equal(run.buf.dk_seq, ref["dk_seq"]) and torch.equal(run.buf.dv_seq, ref["dv_seq"])
    x = oracle_inputs(run.inputs)
    rows = sample_rows(w, 8, seed=3)
    op = oracle_problem(w)
    # one (rank, kv-head) group at each end of the head range: their q-heads' dQ rows
    groups = [(0, 0, 0), (w.P - 1, w.B - 1, op.kvp - 1)]
    want = oracle.backward(op, x["q"], x["k"], x["v"], x["do"], groups=groups, q_rows=rows, kv_rows=[rows[0]])
    hp = w.n_head // w.P
    G = hp // op.kvp
    got = np.concatenate(list(to64(run.buf.dq_seq)), axis=1)      # [B][S][n_head][D] global
    want_dq = np.concatenate(list(want["dq_seq"]), axis=1)
    for b in sorted({g[1] for g in groups}):
        # the q-heads of the groups of batch b (the oracle computed no others)
        heads = [r * hp + kl * G + gi for (r, bb, kl) in groups if bb == b for gi in range(G)]
        assert_close(got[b][rows][:, heads], want_dq[b][rows][:, heads], w, f"fused dq_seq batch {b}")
