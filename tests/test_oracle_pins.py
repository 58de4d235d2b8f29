"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

No GPU.  Sources (page title, section):
  [SP2] "Sequence Parallelism II: DeepSpeed Ulysses and All-to-All Attention"
  [CMP] "Comparing Ulysses and Megatron Sequence Parallelism"
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def tagged_ranks(P, B, Sl, heads, D):
    """x_r[b][t][h][e] = 1000*r + 100*h + 10*t + e (seq shard r = rank r)."""
    out = []
    for r in range(P):
        a = np.zeros((B, Sl, heads, D))
        for t in range(Sl):
            for h in range(heads):
                for e in range(D):
                    a[:, t, h, e] = 1000 * r + 100 * h + 10 * t + e
        out.append(a)
    return out


# ---------------------------------------------------------------- permutation

def test_ownership_example_matches_page():
    """[SP2] §1: rank 0 goes from S0H0,S0H1,S0H2,S0H3 to S0H0,S1H0,S2H0,S3H0."""
    P, Sl, D = 4, 3, 2
    want = {}
    with open(os.path.join(GOLD, "ownership_p4_h4.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kind, rank, _src, *labels = line.split()
            want[(kind, int(rank))] = labels
    x = tagged_ranks(P, 1, Sl, 4, D)
    y, _, _ = oracle.a2a_seq_to_head(x, 4)
    for r in range(P):
        before = [f"S{int(x[r][0, 0, h, 0]) // 1000}H{(int(x[r][0, 0, h, 0]) // 100) % 10}"
                  for h in range(4)]
        assert before == want[("before", r)]
        after = []
        for blk in range(P):
            v = int(y[r][0, blk * Sl, 0, 0])
            after.append(f"S{v // 1000}H{(v // 100) % 10}")
            # inside a piece, token order and features are preserved
            for t in range(Sl):
                for e in range(D):
                    assert int(y[r][0, blk * Sl + t, 0, e]) % 100 == 10 * t + e
        assert after == want[("after", r)]


@pytest.mark.parametrize("P,B,Sl,heads,D", [(1, 1, 5, 3, 4), (2, 2, 3, 4, 2), (4, 1, 7, 8, 3),
                                           (8, 1, 2, 8, 5), (4, 3, 1, 4, 1)])
def test_pack_then_unpack_is_identity(P, B, Sl, heads, D):
    """[SP2] §2 fifth step: the second All-to-All returns the layout to
    sequence-major ownership; composed with the first it is the identity."""
    x = [rnd((B, Sl, heads, D), 10 * P + r) for r in range(P)]
    y, _, _ = oracle.a2a_seq_to_head(x, heads)
    z, _, _ = oracle.a2a_head_to_seq(y, heads)
    for r in range(P):
        assert np.array_equal(z[r], x[r])
        # [CMP] "DeepSpeed Attention costs": the layout change does not change
        # the number of elements held by a rank.
        assert y[r].size == x[r].size


@pytest.mark.parametrize("P,B,Sl,heads,D,eb", [(2, 1, 4, 2, 8, 2), (4, 2, 3, 8, 4, 2),
                                              (8, 1, 2, 8, 2, 4), (3, 1, 2, 6, 2, 2)])
def test_bytes_moved_match_page_formula(P, B, Sl, heads, D, eb):
    """[CMP] "DeepSpeed Attention costs": each rank sends and receives
    N*(P-1)/P^2 bytes per All-to-All of an N-byte global tensor."""
    N = B * Sl * P * heads * D * eb
    x = [rnd((B, Sl, heads, D), r) for r in range(P)]
    y, sent, recv = oracle.a2a_seq_to_head(x, heads, elem_bytes=eb)
    assert sent == [N * (P - 1) // (P * P)] * P == recv
    _, sent2, recv2 = oracle.a2a_head_to_seq(y, heads, elem_bytes=eb)
    assert sent2 == sent and recv2 == recv


def test_pages_sizing_volumes():
    """28MB per All-to-All per rank, 112MB forward, 224MB forward+backward at
    P=8, S=32768, 32 heads, D=128, bf16 ([CMP] "DeepSpeed Attention costs").
    The byte counts come from running the loop All-to-All at that size."""
    g = {}
    with open(os.path.join(GOLD, "a2a_volume_pages_sizing.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                g[k] = int(v)
    MB = 1 << 20
    P, B, S, H, D, eb = g["P"], g["B"], g["S"], g["n_head"], g["head_dim"], g["elem_bytes"]
    assert B * S * H * D * eb == g["global_tensor_MB"] * MB
    Sl = S // P
    x = [np.zeros((B, Sl, H, D)) for _ in range(P)]
    assert x[0].size * eb == g["per_rank_shard_MB"] * MB
    y, sent_s2h, recv_s2h = oracle.a2a_seq_to_head(x, H, elem_bytes=eb)
    del x
    _, sent_h2s, recv_h2s = oracle.a2a_head_to_seq(y, H, elem_bytes=eb)
    del y
    for r in range(P):
        assert sent_s2h[r] == recv_s2h[r] == g["per_a2a_per_rank_MB"] * MB
        # forward: Q, K, V seq->head and the context head->seq
        fwd = 3 * sent_s2h[r] + sent_h2s[r]
        assert fwd == g["forward_per_rank_MB"] * MB
        # backward: dO seq->head, dQ, dK, dV head->seq
        bwd = sent_s2h[r] + 3 * sent_h2s[r]
        assert fwd + bwd == g["forward_backward_per_rank_MB"] * MB


def test_lost_piece_is_detected():
    """A dropped All-to-All piece breaks both the identity and the volume."""
    P, B, Sl, heads, D = 4, 1, 3, 4, 2
    x = [rnd((B, Sl, heads, D), r) for r in range(P)]
    y, sent, _ = oracle.a2a_seq_to_head(x, heads, skip=(2, 1), fill=np.nan)
    z, _, _ = oracle.a2a_head_to_seq(y, heads)
    assert not all(np.array_equal(z[r], x[r]) for r in range(P))
    N = B * Sl * P * heads * D * 2
    assert sent[2] != N * (P - 1) // (P * P)


# ---------------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity_and_positions_are_global():
    P, B, Sl, H, D = 4, 1, 3, 2, 8
    x = [rnd((B, Sl, H, D), r) for r in range(P)]
    y = oracle.rope_seq(x, 10000.0)
    assert np.array_equal(y[0][:, 0], x[0][:, 0])            # p = 0
    assert not np.allclose(y[1][:, 0], x[1][:, 0])           # p = Sl, not 0
    # sharded rope == rope of the unsharded tensor, then sharded
    whole = oracle.rope_seq([oracle.unshard_sequence(x)], 10000.0)[0]
    for r, part in enumerate(oracle.shard_sequence(whole, P)):
        assert np.array_equal(part, y[r])


def test_rope_preserves_pair_norms_and_inverts():
    P, B, Sl, H, D = 2, 2, 5, 3, 16
    x = [rnd((B, Sl, H, D), 7 + r) for r in range(P)]
    y = oracle.rope_seq(x, 10000.0)
    half = D // 2
    for r in range(P):
        n0 = x[r][..., :half] ** 2 + x[r][..., half:] ** 2
        n1 = y[r][..., :half] ** 2 + y[r][..., half:] ** 2
        np.testing.assert_allclose(n1, n0, rtol=1e-13, atol=1e-13)
    z = oracle.rope_seq(y, 10000.0, -1)
    for r in range(P):
        np.testing.assert_allclose(z[r], x[r], rtol=0, atol=1e-13)


def test_rope_scores_depend_on_relative_position_only():
    D, S = 16, 64
    q, k = rnd(D, 1), rnd(D, 2)

    def score(pq, pk):
        X = np.zeros((1, S, 2, D))
        X[0, pq, 0] = q
        X[0, pk, 1] = k
        Y = oracle.rope_seq([X], 10000.0)[0]
        return float(Y[0, pq, 0] @ Y[0, pk, 1])

    for (a, b, c) in [(5, 3, 17), (0, 9, 40), (20, 20, 13), (31, 2, 30)]:
        assert abs(score(a, b) - score(a + c, b + c)) < 1e-11
    assert abs(score(5, 3) - score(5, 4)) > 1e-6


# ----------------------------------------------------------------- attention

def _prob(P, B, S, h, kv, D, causal, rope):
    return oracle.Problem(B=B, S=S, n_head=h, n_kv_head=kv, D=D, P=P, causal=causal,
                          use_rope=rope, rope_base=10000.0)


def _global_lse(prob, lse_ranks):
    return np.concatenate(lse_ranks, axis=1)  # rank r holds heads [r*hp, (r+1)*hp)


@pytest.mark.parametrize("P,B,S,h,kv,D,causal,rope", [
    (2, 1, 8, 2, 2, 4, True, True), (4, 1, 16, 4, 4, 4, True, True),
    (2, 2, 6, 4, 2, 6, False, True), (4, 1, 8, 8, 4, 2, True, False),
    (1, 1, 5, 2, 1, 4, True, True), (2, 1, 4, 2, 2, 2, False, False),
    # KV-head replication (n_kv_head < P): every kv-head held by P/n_kv ranks
    (4, 1, 8, 4, 2, 4, True, True), (4, 2, 8, 4, 1, 2, False, True), (8, 1, 16, 8, 2, 2, True, False)])
def test_oracle_matches_brute_force(P, B, S, h, kv, D, causal, rope):
    Q, K, V = rnd((B, S, h, D), 1), rnd((B, S, kv, D), 2), rnd((B, S, kv, D), 3)
    dO = rnd((B, S, h * D), 4)
    prob = _prob(P, B, S, h, kv, D, causal, rope)
    fw = oracle.forward(prob, Q, K, V)
    out = oracle.unshard_sequence(fw["o_seq"]).reshape(B, S, h * D)
    bo, blse = brute.forward(Q.tolist(), K.tolist(), V.tolist(), causal, prob.softmax_scale, rope, 10000.0)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(_global_lse(prob, fw["lse"]), np.array(blse), rtol=0, atol=1e-12)
    bw = oracle.backward(prob, Q, K, V, dO)
    bdq, bdk, bdv = brute.backward(Q.tolist(), K.tolist(), V.tolist(), dO.tolist(), causal,
                                   prob.softmax_scale, rope, 10000.0)
    for mine, ref in ((bw["dq_seq"], bdq), (bw["dk_seq"], bdk), (bw["dv_seq"], bdv)):
        np.testing.assert_allclose(oracle.unshard_sequence(mine), np.array(ref), rtol=0, atol=1e-11)


def test_brute_force_gradients_match_finite_differences():
    """Pins the written-out softmax chain rule (and the inverse rope on dq, dk)
    against central differences of the forward itself."""
    B, S, h, kv, D = 1, 5, 2, 1, 4
    Q, K, V = rnd((B, S, h, D), 11), rnd((B, S, kv, D), 12), rnd((B, S, kv, D), 13)
    dO = rnd((B, S, h * D), 14)
    for causal, rope in ((True, True), (False, False)):
        args = (causal, 0.4, rope, 10000.0)
        dq, dk, dv = brute.backward(Q.tolist(), K.tolist(), V.tolist(), dO.tolist(), *args)
        eps = 1e-5
        for name, T, G in (("q", Q, dq), ("k", K, dk), ("v", V, dv)):
            for idx in [(0, 0, 0, 0), (0, S - 1, T.shape[2] - 1, D - 1), (0, 2, 0, 1), (0, 3, 0, 3)]:
                Tp, Tm = T.copy(), T.copy()
                Tp[idx] += eps
                Tm[idx] -= eps
                ins_p = {"q": Q, "k": K, "v": V}
                ins_m = dict(ins_p)
                ins_p[name], ins_m[name] = Tp, Tm
                lp = brute.loss(ins_p["q"].tolist(), ins_p["k"].tolist(), ins_p["v"].tolist(), dO.tolist(), *args)
                lm = brute.loss(ins_m["q"].tolist(), ins_m["k"].tolist(), ins_m["v"].tolist(), dO.tolist(), *args)
                fd = (lp - lm) / (2 * eps)
                b, s, hh, e = idx
                assert abs(fd - G[b][s][hh][e]) < 1e-7, (name, idx, fd, G[b][s][hh][e])


@pytest.mark.parametrize("P,B,S,h,kv,D,causal,rope", [
    (4, 2, 64, 8, 4, 8, True, True), (2, 1, 96, 4, 2, 16, False, True),
    (8, 1, 64, 8, 8, 4, True, False),
    (4, 1, 64, 4, 2, 8, True, True), (8, 2, 64, 8, 1, 4, True, True), (8, 1, 96, 16, 4, 8, False, True)])
def test_ulysses_equals_unsharded_attention_bit_exact(P, B, S, h, kv, D, causal, rope):
    """[SP2] §1/§3: the transposes are a permutation of ownership, so the
    sharded pipeline must reproduce unsharded attention exactly in fp64."""
    Q, K, V = rnd((B, S, h, D), 21), rnd((B, S, kv, D), 22), rnd((B, S, kv, D), 23)
    prob = _prob(P, B, S, h, kv, D, causal, rope)
    fw = oracle.forward(prob, Q, K, V)
    o_glob, lse_glob = oracle.unsharded(prob, Q, K, V)
    assert np.array_equal(oracle.unshard_sequence(fw["o_seq"]), o_glob)
    assert np.array_equal(_global_lse(prob, fw["lse"]), lse_glob)


@pytest.mark.parametrize("causal", [True, False])
def test_single_rank_matches_torch_sdpa_and_autograd(causal):
    """At P=1 the path is plain scaled-dot-product attention: compare with
    torch's fp64 CPU SDPA and its autograd (grouped K/V heads expanded)."""
    B, S, h, kv, D = 2, 40, 4, 2, 16
    Q, K, V = rnd((B, S, h, D), 31), rnd((B, S, kv, D), 32), rnd((B, S, kv, D), 33)
    dO = rnd((B, S, h * D), 34)
    prob = _prob(1, B, S, h, kv, D, causal, False)
    fw = oracle.forward(prob, Q, K, V)
    bw = oracle.backward(prob, Q, K, V, dO)
    q = torch.tensor(Q).transpose(1, 2).requires_grad_(True)
    k = torch.tensor(K).transpose(1, 2).requires_grad_(True)
    v = torch.tensor(V).transpose(1, 2).requires_grad_(True)
    G = h // kv
    o = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1), is_causal=causal)
    o_bshd = o.transpose(1, 2)
    (o_bshd.reshape(B, S, h * D) * torch.tensor(dO)).sum().backward()
    np.testing.assert_allclose(fw["o_seq"][0], o_bshd.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(bw["dq_seq"][0], q.grad.transpose(1, 2).numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(bw["dk_seq"][0], k.grad.transpose(1, 2).numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(bw["dv_seq"][0], v.grad.transpose(1, 2).numpy(), rtol=0, atol=1e-11)


def test_closed_forms():
    P, B, S, h, D = 2, 1, 32, 2, 8
    V = rnd((B, S, h, D), 41)
    K = rnd((B, S, h, D), 42)
    # q = 0: uniform softmax; causal output is the prefix mean, lse = log(i+1)
    prob = _prob(P, B, S, h, h, D, True, True)
    fw = oracle.forward(prob, np.zeros((B, S, h, D)), K, V)
    o = oracle.unshard_sequence(fw["o_seq"])
    pref = np.cumsum(V, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    np.testing.assert_allclose(o, pref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(_global_lse(prob, fw["lse"]),
                               np.broadcast_to(np.log(np.arange(1, S + 1)), (B, h, S)), atol=1e-13)
    # non-causal q = 0: every row is the mean of v
    prob_nc = _prob(P, B, S, h, h, D, False, False)
    o_nc = oracle.unshard_sequence(oracle.forward(prob_nc, np.zeros((B, S, h, D)), K, V)["o_seq"])
    np.testing.assert_allclose(o_nc, np.broadcast_to(V.mean(axis=1, keepdims=True), o_nc.shape), atol=1e-13)
    # causal row 0 sees only key 0: output is v_0 exactly, whatever q and k are
    Q = rnd((B, S, h, D), 43)
    fw = oracle.forward(prob, Q, K, V)
    assert np.array_equal(fw["o_seq"][0][:, 0], V[:, 0])
    # one dominant key j: rows that can see it return v_j
    j = 3
    Kd = np.zeros((B, S, h, D))
    Kd[:, j, :, 0] = 30.0
    Qd = np.zeros((B, S, h, D))
    Qd[..., 0] = 2.0 * math.sqrt(D)  # scaled score 30*2*sqrt(D)/sqrt(D) = 60 for key j, 0 elsewhere
    od = oracle.unshard_sequence(oracle.forward(_prob(P, B, S, h, h, D, True, False), Qd, Kd, V)["o_seq"])
    np.testing.assert_allclose(od[:, j:], np.broadcast_to(V[:, j:j + 1], od[:, j:].shape), atol=10 * S * math.exp(-60) * np.abs(V).max())


def test_gqa_equals_mha_with_repeated_kv_heads():
    P, B, S, h, kv, D = 2, 1, 48, 8, 2, 8
    G = h // kv
    Q, K, V = rnd((B, S, h, D), 51), rnd((B, S, kv, D), 52), rnd((B, S, kv, D), 53)
    dO = rnd((B, S, h * D), 54)
    pg = _prob(P, B, S, h, kv, D, True, True)
    pm = _prob(P, B, S, h, h, D, True, True)
    Kr, Vr = np.repeat(K, G, axis=2), np.repeat(V, G, axis=2)
    og = oracle.unshard_sequence(oracle.forward(pg, Q, K, V)["o_seq"])
    om = oracle.unshard_sequence(oracle.forward(pm, Q, Kr, Vr)["o_seq"])
    assert np.array_equal(og, om)
    bg = oracle.backward(pg, Q, K, V, dO)
    bm = oracle.backward(pm, Q, Kr, Vr, dO)
    np.testing.assert_array_equal(oracle.unshard_sequence(bg["dq_seq"]), oracle.unshard_sequence(bm["dq_seq"]))
    dk_m = oracle.unshard_sequence(bm["dk_seq"]).reshape(B, S, kv, G, D).sum(axis=3)
    dv_m = oracle.unshard_sequence(bm["dv_seq"]).reshape(B, S, kv, G, D).sum(axis=3)
    np.testing.assert_allclose(oracle.unshard_sequence(bg["dk_seq"]), dk_m, rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.unshard_sequence(bg["dv_seq"]), dv_m, rtol=0, atol=1e-12)


def test_row_sampling_matches_full():
    P, B, S, h, kv, D = 4, 1, 64, 4, 4, 8
    Q, K, V = rnd((B, S, h, D), 61), rnd((B, S, kv, D), 62), rnd((B, S, kv, D), 63)
    dO = rnd((B, S, h * D), 64)
    prob = _prob(P, B, S, h, kv, D, True, True)
    full = oracle.forward(prob, Q, K, V)
    rows = [0, 15, 16, 17, 63]
    part = oracle.forward(prob, Q, K, V, rows=rows)
    for r in range(P):
        assert np.array_equal(part["o_head"][r][:, rows], full["o_head"][r][:, rows])
        assert np.array_equal(part["lse"][r][:, :, rows], full["lse"][r][:, :, rows])
    bf = oracle.backward(prob, Q, K, V, dO)
    bp = oracle.backward(prob, Q, K, V, dO, groups=[(1, 0, 0)], q_rows=rows, kv_rows=rows)
    for name in ("dq_head", "dk_head", "dv_head"):
        assert np.array_equal(bp[name][1][:, rows], bf[name][1][:, rows])


@pytest.mark.parametrize("P,B,Sl,kv,D", [(4, 1, 3, 2, 4), (8, 2, 2, 1, 3), (8, 1, 4, 4, 2)])
def test_replicated_reduce_is_the_adjoint_of_the_replicating_all_to_all(P, B, Sl, kv, D):
    """The kv All-to-All with replication copies each kv-head to P/kv ranks; the
    gradient step must be its exact transpose: <A(x), y> = <x, A^T(y)> for all
    x, y (a dropped replica, a wrong replica index or a wrong source row breaks
    the identity).  Also: identical replicas reduce to R times the value."""
    rng = np.random.default_rng(41)
    x = [rng.standard_normal((B, Sl, kv, D)) for _ in range(P)]
    y = [rng.standard_normal((B, Sl * P, 1, D)) for _ in range(P)]
    ax, _, _ = oracle.a2a_seq_to_head_replicated(x, kv, 8)
    aty, _, _ = oracle.reduce_head_to_seq_replicated(y, kv, 8)
    lhs = sum(float((a * b).sum()) for a, b in zip(ax, y))
    rhs = sum(float((a * b).sum()) for a, b in zip(x, aty))
    assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + 1.0)
    R = P // kv
    same, _, _ = oracle.reduce_head_to_seq_replicated(ax, kv, 8)
    for r in range(P):  # R-fold repeated addition rounds at 3x, 5x, ...: not bit-equal to R*x
        np.testing.assert_allclose(same[r], R * x[r], rtol=1e-15, atol=0)


@pytest.mark.parametrize("P,B,Sl,kv,D,eb", [(4, 1, 3, 2, 4, 2), (8, 2, 5, 1, 8, 2), (8, 1, 2, 4, 6, 4)])
def test_replicated_bytes_moved(P, B, Sl, kv, D, eb):
    """With replication every rank needs one kv-head over the full sequence,
    of which it holds 1/P itself: it receives (P-1)/P * B*S*D*eb bytes per
    tensor, and (every rank holding exactly one kv-head) sends as much; the
    gradient reduce moves the same amount the other way."""
    x = [np.zeros((B, Sl, kv, D)) for _ in range(P)]
    _, sent, recv = oracle.a2a_seq_to_head_replicated(x, kv, eb)
    want = (P - 1) * B * Sl * D * eb
    assert sent == [want] * P and recv == [want] * P
    y = [np.zeros((B, Sl * P, 1, D)) for _ in range(P)]
    _, sent, recv = oracle.reduce_head_to_seq_replicated(y, kv, eb)
    assert sent == [want] * P and recv == [want] * P


@pytest.mark.parametrize("P,B,S,h,kv,D,bias", [(2, 1, 6, 2, 1, 4, True), (4, 2, 8, 4, 2, 2, False), (4, 1, 8, 4, 1, 2, True)])
def test_qkv_projection_matches_brute_force(P, B, S, h, kv, D, bias):
    """The per-rank projection against plain loops over the unsharded tokens
    (x W^T + b), then split into q, k, v heads."""
    H = h * D
    x = rnd((B, S, H), 51)
    W = rnd(((h + 2 * kv) * D, H), 52)
    b = rnd(((h + 2 * kv) * D,), 53) if bias else None
    prob = _prob(P, B, S, h, kv, D, True, False)
    q, k, v = oracle.qkv_projection(prob, oracle.shard_sequence(x, P), W, b)
    y = np.array(brute.linear(x.tolist(), W.tolist(), None if b is None else b.tolist())).reshape(B, S, h + 2 * kv, D)
    np.testing.assert_allclose(oracle.unshard_sequence(q), y[:, :, :h], rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.unshard_sequence(k), y[:, :, h:h + kv], rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.unshard_sequence(v), y[:, :, h + kv:], rtol=0, atol=1e-12)


def test_qkv_projection_identity_weights_and_pack():
    """Identity blocks as weights: q is x itself viewed as heads and k, v its
    first n_kv_head heads; projecting and packing then equals packing x
    (rotated) directly -- the fused path's definition reduces to the plain one."""
    P, B, S, h, kv, D = 2, 2, 16, 4, 2, 8
    H = h * D
    x = rnd((B, S, H), 61)
    I = np.eye(H)
    W = np.concatenate([I, I[:kv * D], I[:kv * D]], axis=0)
    prob = _prob(P, B, S, h, kv, D, True, True)
    xs = oracle.shard_sequence(x, P)
    qh, kh, vh = oracle.project_and_pack(prob, xs, W)
    xq = [a.reshape(B, S // P, h, D) for a in xs]
    xk = [np.ascontiguousarray(a[:, :, :kv * D]).reshape(B, S // P, kv, D) for a in xs]
    want_q, _, _ = oracle.a2a_seq_to_head(oracle.rope_seq(xq, prob.rope_base, +1), h)
    want_k, _, _ = oracle.a2a_seq_to_head(oracle.rope_seq(xk, prob.rope_base, +1), kv)
    want_v, _, _ = oracle.a2a_seq_to_head(xk, kv)
    for r in range(P):
        assert np.array_equal(qh[r], want_q[r]) and np.array_equal(kh[r], want_k[r]) and np.array_equal(vh[r], want_v[r])


def test_rope_rows_equals_rope_seq():
    """rope_rows (arbitrary positions, used for sampled checks) is the same
    rotation as the pinned rope_seq, row for row."""
    P, B, Sl, h, D = 4, 2, 5, 3, 8
    xs = [rnd((B, Sl, h, D), 70 + r) for r in range(P)]
    want = oracle.rope_seq(xs, 10000.0, +1)
    rows, pos, ref = [], [], []
    for r in range(P):
        for b in range(B):
            for t in range(Sl):
                rows.append(xs[r][b, t]); pos.append(r * Sl + t); ref.append(want[r][b, t])
    got = oracle.rope_rows(np.stack(rows), pos, 10000.0)
    np.testing.assert_allclose(got, np.stack(ref), rtol=0, atol=1e-12)


@pytest.mark.parametrize("P,B,S,h,D,bias", [(2, 1, 6, 2, 4, True), (4, 2, 8, 4, 2, False)])
def test_unpack_and_project_matches_brute_force(P, B, S, h, D, bias):
    """Output projection after the inverse All-to-All, against plain loops
    over the unsharded attention output (the unpack is a permutation, so
    projecting per rank after it equals projecting the global tensor)."""
    H = h * D
    o = rnd((B, S, h, D), 81)
    W = rnd((H, H), 82)
    b = rnd((H,), 83) if bias else None
    prob = _prob(P, B, S, h, h, D, True, False)
    o_head, _, _ = oracle.a2a_seq_to_head(oracle.shard_sequence(o, P), h)
    y = oracle.unpack_and_project(prob, o_head, W, b)
    want = np.array(brute.linear(o.reshape(B, S, H).tolist(), W.tolist(), None if b is None else b.tolist()))
    np.testing.assert_allclose(oracle.unshard_sequence(y), want, rtol=0, atol=1e-12)


def test_unpack_and_project_identity_is_the_unpack():
    """With W = I and no bias the fused definition is the plain unpack."""
    P, B, S, h, D = 4, 2, 16, 4, 8
    o = rnd((B, S, h, D), 91)
    prob = _prob(P, B, S, h, h, D, True, False)
    o_head, _, _ = oracle.a2a_seq_to_head(oracle.shard_sequence(o, P), h)
    y = oracle.unpack_and_project(prob, o_head, np.eye(h * D))
    back, _, _ = oracle.a2a_head_to_seq(o_head, h)
    for r in range(P):
        assert np.array_equal(y[r], back[r].reshape(B, S // P, h * D))
