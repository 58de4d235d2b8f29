"""GPU parity of the dS-store backward (ulysses_attn_bwd_ds: the dK/dV kernel
writes every tile pair's bf16 dS to the workspace, a second kernel sums dQ
from those tiles) through the C ABI: dQ against the fp64 oracle under the same
bar as every other gradient; dK and dV bit-identical to the two-kernel
backward (the same kernel, which only also stores dS); dQ bit-identical from
call to call (no reduction whose order varies); the three steps equal the
composed call; the full-size workloads on sampled rows."""
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


def _ds_ids(w):
    return _ids(w) + (f"R{w.ring}" if w.ring > 1 else "")


@pytest.mark.parametrize("w", CASES, ids=_ds_ids)
def test_ds_backward_matches_oracle_and_two_kernel_backward(w):
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True, ds=True)
    run.forward()
    run.backward()                                   # the two-kernel backward
    ref = {n: getattr(run.buf, n).clone() for n in GRADS}
    x = oracle_inputs(run.inputs)
    if w.ring > 1:
        from oracle import ring as oracle_ring
        want = oracle_ring.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"])
    else:
        want = oracle.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"])
    first = None
    for _ in range(2):
        for n in GRADS:
            getattr(run.buf, n).fill_(float("nan"))
        run.backward_ds()
        assert torch.equal(run.buf.dk_seq, ref["dk_seq"]), "dS-store dK differs from the two-kernel backward"
        assert torch.equal(run.buf.dv_seq, ref["dv_seq"]), "dS-store dV differs from the two-kernel backward"
        if first is None:
            first = run.buf.dq_seq.clone()
            assert_close(to64(run.buf.dq_seq), np.stack(want["dq_seq"]), w, "dS-store dq_seq")
        else:
            assert torch.equal(run.buf.dq_seq, first), "dS-store dQ differs from one call to the next"


def test_ds_steps_equal_composed_call():
    """prepare + dkdv_ds + dq_ds give exactly what ulysses_attn_bwd_ds gives."""
    w = WORKLOADS["C3"].with_(S=1024)
    run = GpuRun(w, backward=True, ds=True)
    run.forward()
    run.backward_ds()
    b = run.buf
    ref = [t.clone() for t in (b.dq_seq, b.dk_seq, b.dv_seq)]
    for t in (b.dq_seq, b.dk_seq, b.dv_seq):
        t.zero_()
    U.ulysses_attn_bwd_prepare(run.prob, b.o_head, b.lse, b.do_seq, b.ws)
    U.ulysses_attn_bwd_dkdv_ds(run.prob, b.q_head, b.k_head, b.v_head, b.dk_seq, b.dv_seq, b.ws)
    U.ulysses_attn_bwd_dq_ds(run.prob, b.k_head, b.dq_seq, b.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(b.ws) == 0
    for got, want in zip((b.dq_seq, b.dk_seq, b.dv_seq), ref):
        assert torch.equal(got, want)


def test_ds_backward_needs_a_phase3_workspace():
    w = wl(2, 1, 256, 4, 4, 64).with_(backward=True)
    run = GpuRun(w, backward=True)                   # phase-1 workspace
    run.forward()
    with pytest.raises(U.UlyssesError) as e:
        run.buf.backward_ds()
    assert e.value.code == -7


@pytest.mark.parametrize("name", ["C2", "C3", "C4", "C4-kv4"])
def test_ds_backward_workloads(name):
    """Full size, in the bench's launch configuration: dQ of every q-head of
    two (rank, kv-head) groups on sampled rows (shard/tile boundaries and
    seeded random rows, each exact over its full key range) against the
    oracle; dK and dV equal to the two-kernel backward's.  C2 (head_dim 64,
    B = 2) is a forward workload; its shapes are run with a backward here."""
    w = WORKLOADS[name] if name in WORKLOADS else EXTRA_WORKLOADS[name]
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True, ds=True)
    run.forward()
    run.backward()
    ref = {n: getattr(run.buf, n).clone() for n in ("dk_seq", "dv_seq")}
    run.backward_ds()
    assert torch.equal(run.buf.dk_seq, ref["dk_seq"]) and torch.equal(run.buf.dv_seq, ref["dv_seq"])
    x = oracle_inputs(run.inputs)
    rows = sample_rows(w, 8, seed=3)
    op = oracle_problem(w)
    groups = [(0, 0, 0), (w.P - 1, w.B - 1, op.kvp - 1)]
    want = oracle.backward(op, x["q"], x["k"], x["v"], x["do"], groups=groups, q_rows=rows, kv_rows=[rows[0]])
    hp = w.n_head // w.P
    G = hp // op.kvp
    got = np.concatenate(list(to64(run.buf.dq_seq)), axis=1)      # [B][S][n_head][D] global
    want_dq = np.concatenate(list(want["dq_seq"]), axis=1)
    for b in sorted({g[1] for g in groups}):
        # the q-heads of the groups of batch b (the oracle computed no others)
        heads = [r * hp + kl * G + gi for (r, bb, kl) in groups if bb == b for gi in range(G)]
        assert_close(got[b][rows][:, heads], want_dq[b][rows][:, heads], w, f"dS-store dq_seq batch {b}")


TINY = [wl(2, 1, 96, 2, 2, 64),                    # one ragged 128-row tile
        wl(2, 1, 2, 4, 2, 128),                    # one token per rank
        wl(4, 1, 40, 4, 1, 64, causal=False),      # unmasked, replicated kv-head
        wl(1, 1, 129, 2, 1, 128)]                  # a full tile and one row


@pytest.mark.parametrize("w", TINY, ids=_ids)
def test_tiny_sequences_every_backward_mode(w):
    """Degenerate lengths (fewer rows than a tile, one token per rank, a tile
    and one row): the two-kernel, dS-store and fused backwards against the
    oracle, dK and dV identical across the three."""
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True, ds=True, fused=True)
    run.forward()
    x = oracle_inputs(run.inputs)
    want = oracle.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"])
    ref = None
    for name, call in (("two-kernel", run.backward), ("dS-store", run.backward_ds), ("fused", run.backward_fused)):
        for n in GRADS:
            getattr(run.buf, n).fill_(float("nan"))
        call()
        for n in GRADS:
            assert_close(to64(getattr(run.buf, n)), np.stack(want[n]), w, f"{name} {n}")
        if ref is None:
            ref = {n: getattr(run.buf, n).clone() for n in ("dk_seq", "dv_seq")}
        else:
            assert all(torch.equal(getattr(run.buf, n), ref[n]) for n in ref), f"{name} dK/dV differ"


@pytest.mark.parametrize("w", [wl(8, 1, 1024, 32, 8, 128),            # GQA: 4 q-heads a kv-head, 8 kv-heads
                               wl(8, 1, 1024, 8, 2, 128),             # kv-heads replicated over 4 ranks
                               wl(4, 2, 512, 8, 8, 64, causal=False)], ids=_ids)
def test_ds_backward_in_chunks_of_kv_heads(w):
    """A workspace smaller than phase 3 (down to phase 4: one kv-head's tiles)
    makes the dS-store backward run the kv-heads in chunks; every chunking
    gives the same bits as the whole-workspace call."""
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True, ds=True)
    run.forward()
    run.backward_ds()
    b, p = run.buf, run.prob
    ref = {n: getattr(b, n).clone() for n in GRADS}
    n1, n3, n4 = (U.ulysses_workspace_bytes(p, k) for k in (1, 3, 4))
    per_kv = n4 - n1
    for nbytes in (n4, n1 + 3 * per_kv, n3 - 256):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        U.ulysses_workspace_init(p, ws)
        for n in GRADS:
            getattr(b, n).fill_(float("nan"))
        U.ulysses_attn_bwd_ds(p, b.q_head, b.k_head, b.v_head, b.o_head, b.lse, b.do_seq, b.dq_seq, b.dk_seq,
                              b.dv_seq, ws)
        torch.cuda.synchronize()
        assert U.ulysses_read_status(ws) == 0
        for n in GRADS:
            assert torch.equal(getattr(b, n), ref[n]), (nbytes, n)
