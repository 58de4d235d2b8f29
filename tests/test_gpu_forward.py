"""GPU parity of the forward path (pack -> attention -> unpack) against the
fp64 oracle, through the C ABI.  Needs a GB300 and the built library."""
import numpy as np
import pytest
import torch

import oracle
from pathcheck import (GpuRun, assert_close, assert_lse_close, oracle_inputs,
                       oracle_problem, to64, ulp_bf16)
from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300.synthetic import WORKLOADS, Workload

pytestmark = pytest.mark.gpu


def wl(P, B, S, h, kv, D, dtype="bf16", causal=True, rope=True, seed=7):
    return Workload("t", P=P, B=B, S=S, hidden=h * D, n_head=h, n_kv_head=kv, head_dim=D,
                    dtype=dtype, causal=causal, use_rope=rope, rope_base=10000.0, sigma=1.0,
                    backward=False, seed=seed)


PERM_CASES = [wl(2, 1, 256, 4, 4, 32, "fp32"), wl(4, 2, 512, 16, 16, 64), wl(8, 1, 1024, 32, 8, 128),
              wl(2, 3, 424, 4, 2, 128), wl(1, 1, 96, 2, 1, 64), wl(4, 1, 64, 8, 4, 128, "fp32"),
              wl(32, 1, 2048, 32, 32, 128)]


def _pack(run):
    b = run.buf
    U.ulysses_pack_qkv(run.prob, b.q_seq, b.k_seq, b.v_seq, b.q_head, b.k_head, b.v_head, b.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(b.ws) == 0


@pytest.mark.parametrize("w", PERM_CASES, ids=lambda w: f"P{w.P}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}{w.dtype}")
def test_pack_is_bit_exact_permutation(w):
    """Without RoPE the seq->head pack is the pages' All-to-All, bit for bit."""
    w = w.with_(use_rope=False)
    run = GpuRun(w)
    _pack(run)
    x = oracle_inputs(run.inputs)
    for name, heads, got in (("q", w.n_head, run.buf.q_head), ("k", w.n_kv_head, run.buf.k_head),
                             ("v", w.n_kv_head, run.buf.v_head)):
        want, _, _ = oracle.a2a_seq_to_head(oracle.shard_sequence(x[name], w.P), heads)
        g = to64(got)
        for r in range(w.P):
            assert np.array_equal(g[r], want[r]), f"{name} rank {r}"


@pytest.mark.parametrize("w", PERM_CASES, ids=lambda w: f"P{w.P}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}{w.dtype}")
def test_pack_rope_within_one_ulp(w):
    run = GpuRun(w)
    _pack(run)
    x = oracle_inputs(run.inputs)
    half = w.head_dim // 2
    for name, heads, got, rope in (("q", w.n_head, run.buf.q_head, True), ("k", w.n_kv_head, run.buf.k_head, True),
                                   ("v", w.n_kv_head, run.buf.v_head, False)):
        seq = oracle.shard_sequence(x[name], w.P)
        rot = oracle.rope_seq(seq, float(np.float32(w.rope_base))) if rope else seq
        want, _, _ = oracle.a2a_seq_to_head(rot, heads)
        mag, _, _ = oracle.a2a_seq_to_head(
            [np.concatenate([np.abs(a[..., :half]) + np.abs(a[..., half:])] * 2, axis=-1) for a in seq], heads)
        g = to64(got)
        for r in range(w.P):
            if not rope:
                assert np.array_equal(g[r], want[r])
                continue
            err = np.abs(g[r] - want[r])
            if w.dtype == "bf16":
                tol = ulp_bf16(want[r]) + 2.0 ** -20 * mag[r]
            else:
                tol = 2.0 ** -20 * (np.abs(want[r]) + mag[r])
            bad = err > tol
            assert not bad.any(), f"{name} rank {r}: {bad.sum()} elements off, worst {err.max():.3e}"


@pytest.mark.parametrize("w", PERM_CASES[:5], ids=lambda w: f"P{w.P}B{w.B}S{w.S}h{w.n_head}D{w.head_dim}{w.dtype}")
def test_unpack_is_bit_exact_permutation(w):
    prob = U.Problem.from_workload(w)
    g = torch.Generator().manual_seed(5)
    o_head_cpu = torch.randn(w.P, w.B, w.S, w.n_head // w.P, w.head_dim, generator=g).to(prob.torch_dtype)
    o_head = o_head_cpu.cuda()
    o_seq = torch.empty(w.P, w.B, w.Sl, w.n_head * w.head_dim, dtype=prob.torch_dtype, device="cuda")
    U.ulysses_unpack_out(prob, o_head, o_seq)
    torch.cuda.synchronize()
    want, _, _ = oracle.a2a_head_to_seq([to64(o_head_cpu[r]) for r in range(w.P)], w.n_head)
    got = to64(o_seq)
    for r in range(w.P):
        assert np.array_equal(got[r], want[r].reshape(w.B, w.Sl, -1))


FWD_CASES = [wl(2, 1, 256, 4, 4, 32, "fp32", causal=False, rope=False),
             wl(2, 1, 256, 4, 2, 64, "fp32", causal=True, rope=True),
             wl(2, 1, 424, 4, 2, 128),            # ragged tail: 3 full tiles + 40 rows
             wl(4, 2, 512, 8, 8, 64),
             wl(2, 1, 320, 2, 2, 128, causal=False, rope=False),
             wl(1, 1, 640, 4, 1, 128, causal=True),
             wl(8, 1, 1024, 32, 8, 128),
             wl(2, 1, 130, 2, 2, 64, causal=False)]


@pytest.mark.parametrize("w", FWD_CASES, ids=lambda w: f"P{w.P}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}{w.dtype}{'c' if w.causal else 'n'}")
def test_forward_matches_oracle(w):
    run = GpuRun(w)
    run.forward()
    x = oracle_inputs(run.inputs)
    want = oracle.forward(oracle_problem(w), x["q"], x["k"], x["v"])
    got_o = to64(run.buf.o_seq)
    got_lse = to64(run.buf.lse)
    want_o = np.stack([a.reshape(w.B, w.Sl, -1) for a in want["o_seq"]])
    assert_close(got_o, want_o, w, "o_seq")
    want_lse = np.stack(want["lse"])
    assert_lse_close(got_lse, want_lse, w)
    # bit-exact consistency of the unpack with the kernel's own head-layout output
    o_head = to64(run.buf.o_head)
    hp = w.n_head // w.P
    for d in range(w.P):
        for s in range(w.P):
            blk = o_head[s][:, d * w.Sl:(d + 1) * w.Sl].reshape(w.B, w.Sl, hp * w.head_dim)
            assert np.array_equal(got_o[d][:, :, s * hp * w.head_dim:(s + 1) * hp * w.head_dim], blk)


def sample_rows(w, n_random, seed=0):
    rows = {0, 1, 127, 128, w.S - 1}
    for r in range(1, w.P):
        rows.update({r * w.Sl - 1, r * w.Sl, r * w.Sl + 1})
    rng = np.random.default_rng(seed)
    rows.update(int(x) for x in rng.integers(0, w.S, n_random))
    return sorted(x for x in rows if 0 <= x < w.S)


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4", "C5"])
def test_forward_workloads(name):
    """Each workload at full size, in the launch configuration the bench times;
    C1 is compared in full, the others on sampled query rows (all heads,
    every shard boundary +-1, tile boundaries and seeded random rows)."""
    w = WORKLOADS[name]
    run = GpuRun(w, backward=False)
    run.forward()
    x = oracle_inputs(run.inputs)
    rows = None if name == "C1" else sample_rows(w, 48 if w.S <= 8192 else 24)
    want = oracle.forward(oracle_problem(w), x["q"], x["k"], x["v"], rows=rows)
    got_h = to64(run.buf.o_head)
    got_lse = to64(run.buf.lse)
    sel = slice(None) if rows is None else rows
    want_h = np.stack(want["o_head"])[:, :, sel]
    assert_close(got_h[:, :, sel], want_h, w, f"{name} o_head")
    want_lse = np.stack(want["lse"])[..., sel]
    assert_lse_close(got_lse[..., sel], want_lse, w, f"{name} lse")
    # the unpack is the exact inverse permutation of what the kernel wrote
    o_seq = run.buf.o_seq
    o_head = run.buf.o_head
    hp = w.n_head // w.P
    for d in (0, w.P - 1):
        for s in (0, w.P // 2, w.P - 1):
            blk = o_head[s][:, d * w.Sl:(d + 1) * w.Sl].reshape(w.B, w.Sl, hp * w.head_dim)
            assert torch.equal(o_seq[d][:, :, s * hp * w.head_dim:(s + 1) * hp * w.head_dim], blk)


def test_forward_at_the_longest_sequence():
    """The pages' model at S = 131072 over P = 32 ranks (one head per rank; the
    largest sequence of the permutation sweep): sampled query rows of every
    head, each exact over its full key range, and the unpack inverting what the
    kernel wrote.  Exercises the index arithmetic at 4M (position, head) rows
    per tensor."""
    w = WORKLOADS["C5"].with_(name="C5-128K", S=131072, seed=1008)
    run = GpuRun(w, backward=False)
    run.forward()
    x = oracle_inputs(run.inputs)
    rows = sample_rows(w, 12, seed=4)
    want = oracle.forward(oracle_problem(w), x["q"], x["k"], x["v"], rows=rows)
    got_h = to64(run.buf.o_head)
    assert_close(got_h[:, :, rows], np.stack(want["o_head"])[:, :, rows], w, "C5-128K o_head")
    assert_lse_close(to64(run.buf.lse)[..., rows], np.stack(want["lse"])[..., rows], w)
    o_seq, o_head = run.buf.o_seq, run.buf.o_head
    for d in (0, w.P - 1):
        for s in (0, w.P - 1):
            blk = o_head[s][:, d * w.Sl:(d + 1) * w.Sl].reshape(w.B, w.Sl, w.head_dim)
            assert torch.equal(o_seq[d][:, :, s * w.head_dim:(s + 1) * w.head_dim], blk)


def test_forward_is_deterministic():
    w = wl(4, 1, 1024, 8, 4, 128)
    run = GpuRun(w)
    outs = []
    for _ in range(3):
        run.forward()
        outs.append((run.buf.o_seq.clone(), run.buf.lse.clone()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_stale_rope_table_is_flagged():
    """A workspace prepared for another problem is detected by the kernel and
    reported through the status word, not silently used."""
    w = wl(2, 1, 256, 4, 4, 64)
    run = GpuRun(w)
    other = U.Problem.from_workload(w.with_(rope_base=500.0))
    U.ulysses_workspace_init(other, run.buf.ws)
    b = run.buf
    U.ulysses_pack_qkv(run.prob, b.q_seq, b.k_seq, b.v_seq, b.q_head, b.k_head, b.v_head, b.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(b.ws) & U.STATUS_ROPE_TABLE


@pytest.mark.parametrize("slope", [1.25, -1.25])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_forward_moving_reference(slope, causal, D):
    """Scores that rise (or fall) by about 20 in the base-2 domain per 128-key
    tile: every query row's maximum moves far past the first tile's, so the
    kernel's reference must move (and O, l be rescaled) on nearly every tile;
    falling scores drive the later tiles' P to underflow.  Each head's query
    rows are one random vector x and key s is s * slope * x / |x|^2, so
    q.k = s * slope exactly up to the bf16 rounding both sides share."""
    w = wl(2, 1, 768, 4, 2, D, causal=causal, rope=False)
    g = torch.Generator().manual_seed(11)
    x = torch.randn(w.n_kv_head, D, generator=g)
    xq = x.repeat_interleave(w.n_head // w.n_kv_head, dim=0)          # query head j uses kv head j / group
    q = xq.expand(w.B, w.S, w.n_head, D).clone()
    pos = torch.arange(w.S, dtype=torch.float32).view(1, w.S, 1, 1)
    k = pos * slope * (x / (x * x).sum(-1, keepdim=True)).view(1, 1, w.n_kv_head, D)
    v = torch.randn(w.B, w.S, w.n_kv_head, D, generator=g)
    inputs = {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
    run = GpuRun(w, inputs=inputs)
    run.forward()
    xin = oracle_inputs(run.inputs)
    want = oracle.forward(oracle_problem(w), xin["q"], xin["k"], xin["v"])
    got_o = to64(run.buf.o_seq)
    want_o = np.stack([a.reshape(w.B, w.Sl, -1) for a in want["o_seq"]])
    assert_close(got_o, want_o, w, "o_seq")
    assert_lse_close(to64(run.buf.lse), np.stack(want["lse"]), w)


# KV-head replication: fewer kv-heads than ranks, each kv-head handed to the
# P / n_kv_head ranks whose q-heads read it.
REP_CASES = [wl(4, 1, 512, 8, 2, 128),                     # R = 2, GQA 4
             wl(8, 2, 1024, 8, 1, 64),                     # R = 8 (one kv-head: MQA), B = 2
             wl(8, 1, 648, 16, 4, 128, causal=False),      # R = 2, ragged tail
             wl(4, 1, 256, 4, 2, 32, "fp32", causal=False, rope=False)]


@pytest.mark.parametrize("w", REP_CASES, ids=lambda w: f"P{w.P}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}{w.dtype}")
def test_replicated_kv_pack_is_bit_exact(w):
    """Without RoPE the kv part of the pack is the oracle's replicating
    All-to-All bit for bit (and q's the plain one)."""
    w = w.with_(use_rope=False)
    run = GpuRun(w)
    _pack(run)
    x = oracle_inputs(run.inputs)
    want_q, _, _ = oracle.a2a_seq_to_head(oracle.shard_sequence(x["q"], w.P), w.n_head)
    g = to64(run.buf.q_head)
    for r in range(w.P):
        assert np.array_equal(g[r], want_q[r])
    for name, got in (("k", run.buf.k_head), ("v", run.buf.v_head)):
        want, _, _ = oracle.a2a_seq_to_head_replicated(oracle.shard_sequence(x[name], w.P), w.n_kv_head)
        g = to64(got)
        for r in range(w.P):
            assert np.array_equal(g[r], want[r]), f"{name} rank {r}"


@pytest.mark.parametrize("w", REP_CASES, ids=lambda w: f"P{w.P}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}{w.dtype}{'c' if w.causal else 'n'}")
def test_replicated_kv_forward_matches_oracle(w):
    run = GpuRun(w)
    run.forward()
    x = oracle_inputs(run.inputs)
    want = oracle.forward(oracle_problem(w), x["q"], x["k"], x["v"])
    got_o = to64(run.buf.o_seq)
    want_o = np.stack([a.reshape(w.B, w.Sl, -1) for a in want["o_seq"]])
    assert_close(got_o, want_o, w, "o_seq")
    assert_lse_close(to64(run.buf.lse), np.stack(want["lse"]), w)


def test_replicated_kv_forward_full_size_sampled():
    """The replicated workload at full size (the bench's launch configuration),
    on sampled query rows of every head."""
    from ulysses_sequence_attention_seq_gb300.synthetic import EXTRA_WORKLOADS
    w = EXTRA_WORKLOADS["C4-kv4"]
    run = GpuRun(w, backward=False)
    run.forward()
    x = oracle_inputs(run.inputs)
    rows = sample_rows(w, 24)
    want = oracle.forward(oracle_problem(w), x["q"], x["k"], x["v"], rows=rows)
    assert_close(to64(run.buf.o_head)[:, :, rows], np.stack(want["o_head"])[:, :, rows], w, "o_head")
    assert_lse_close(to64(run.buf.lse)[..., rows], np.stack(want["lse"])[..., rows], w)
