"""Pins of the Ulysses x ring hybrid oracle (oracle/ring.py), no GPU.

Sources (page title, section):
  [SP2] "Sequence Parallelism II: DeepSpeed Ulysses and All-to-All Attention",
        §1 (ownership example), §3 (the All-to-All), §4 (the head-count bound
        and another parallel dimension), §8 (Ring Attention circulates the
        key/value blocks around fixed query blocks).

What pins it (none of it re-types the oracle's own formulas):
  * the hybrid is a re-distribution of ownership plus an exact merge of
    partial softmaxes, so its output and gradients must equal plain attention
    on the unsharded tensors (the C oracle's, itself pinned against the
    brute force, torch SDPA/autograd and finite differences) to fp64 rounding;
  * the pure-Python brute force on tiny problems;
  * R = 1 is plain Ulysses: the same pieces as the C oracle's All-to-All,
    bit for bit;
  * ownership: a tagged input lands where the reading says (rank (r, u) holds
    chunk r of heads block u, pieces in source order);
  * pack then unpack is the identity; bytes moved per rank follow the pages'
    N(P-1)/P^2 for the group of Pu ranks;
  * the merge of two partial softmaxes is the softmax over the union.
A mutant battery at the end plants plausible slips in a copy of the module
and checks that one of these pins fails.
"""
import importlib.util
import os
import sys
import types

import numpy as np
import pytest

import oracle
from oracle import brute
from oracle import ring as RG

SRC = os.path.join(os.path.dirname(oracle.__file__), "ring.py")


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def prob(P, R, B, S, h, kv, D, causal=True, rope=True):
    return oracle.Problem(B=B, S=S, n_head=h, n_kv_head=kv, D=D, P=P, causal=causal, use_rope=rope, ring=R)


def plain_lse_to_ring(p, lse_glob):
    """The unsharded lse [B,h,S] in the hybrid's per-rank layout [B,hp,Cs]."""
    Pu, R, Cs, hp, _ = RG.dims(p)
    return [lse_glob[:, u * hp:(u + 1) * hp, r * Cs:(r + 1) * Cs] for r in range(R) for u in range(Pu)]


# ------------------------------------------------------------ pins (mod = RG)

CASES = [  # P, R, B, S, h, kv, D, causal, rope
    (4, 2, 1, 64, 4, 2, 8, True, True),
    (8, 4, 2, 64, 2, 2, 8, True, True),     # P > n_head: the case the hybrid exists for
    (8, 8, 1, 64, 4, 4, 4, True, False),    # pure ring (Pu = 1)
    (4, 2, 2, 48, 4, 4, 8, False, True),
    (6, 3, 1, 72, 4, 2, 8, True, True),     # three ring positions
    (8, 2, 1, 64, 8, 2, 4, True, True),     # kv-heads replicated inside a ring position (rep 2)
    (16, 4, 2, 64, 4, 1, 4, False, True),   # one kv-head for the 4 members of every position
]


def check_forward_equals_unsharded(mod, P, R, B, S, h, kv, D, causal, rope):
    Q, K, V = rnd((B, S, h, D), 1), rnd((B, S, kv, D), 2), rnd((B, S, kv, D), 3)
    p = prob(P, R, B, S, h, kv, D, causal, rope)
    fw = mod.forward(p, Q, K, V)
    o_glob, lse_glob = oracle.unsharded(p, Q, K, V)
    np.testing.assert_allclose(mod.unshard(fw["o_seq"]), o_glob, rtol=0, atol=1e-12)
    for mine, ref in zip(fw["lse"], plain_lse_to_ring(p, lse_glob)):
        np.testing.assert_allclose(mine, ref, rtol=0, atol=1e-12)


def check_backward_equals_plain(mod, P, R, B, S, h, kv, D, causal, rope):
    Q, K, V = rnd((B, S, h, D), 4), rnd((B, S, kv, D), 5), rnd((B, S, kv, D), 6)
    dO = rnd((B, S, h * D), 7)
    p = prob(P, R, B, S, h, kv, D, causal, rope)
    bw = mod.backward(p, Q, K, V, dO)
    plain = oracle.backward(prob(1, 1, B, S, h, kv, D, causal, rope), Q, K, V, dO)
    for name in ("dq_seq", "dk_seq", "dv_seq"):
        np.testing.assert_allclose(mod.unshard(bw[name]), oracle.unshard_sequence(plain[name]), rtol=0,
                                   atol=1e-11, err_msg=name)


@pytest.mark.parametrize("case", CASES)
def test_forward_equals_unsharded_attention(case):
    check_forward_equals_unsharded(RG, *case)


@pytest.mark.parametrize("case", CASES)
def test_backward_equals_plain_attention_backward(case):
    check_backward_equals_plain(RG, *case)


def test_matches_brute_force():
    P, R, B, S, h, kv, D = 4, 2, 1, 8, 2, 2, 4
    Q, K, V = rnd((B, S, h, D), 8), rnd((B, S, kv, D), 9), rnd((B, S, kv, D), 10)
    dO = rnd((B, S, h * D), 11)
    for causal in (True, False):
        p = prob(P, R, B, S, h, kv, D, causal, True)
        fw = RG.forward(p, Q, K, V)
        bo, _ = brute.forward(Q.tolist(), K.tolist(), V.tolist(), causal, p.softmax_scale, True, 10000.0)
        np.testing.assert_allclose(RG.unshard(fw["o_seq"]).reshape(B, S, h * D), np.array(bo), rtol=0, atol=1e-12)
        bw = RG.backward(p, Q, K, V, dO)
        bdq, bdk, bdv = brute.backward(Q.tolist(), K.tolist(), V.tolist(), dO.tolist(), causal,
                                       p.softmax_scale, True, 10000.0)
        for mine, ref in ((bw["dq_seq"], bdq), (bw["dk_seq"], bdk), (bw["dv_seq"], bdv)):
            np.testing.assert_allclose(RG.unshard(mine), np.array(ref), rtol=0, atol=1e-11)


def check_ring_one_is_ulysses(mod):
    """R = 1: the hybrid's All-to-All hands out exactly the C oracle's pieces,
    and its attention equals the Ulysses oracle's."""
    P, B, S, h, kv, D = 4, 2, 32, 8, 4, 4
    Q, K, V = rnd((B, S, h, D), 12), rnd((B, S, kv, D), 13), rnd((B, S, kv, D), 14)
    q_seq = oracle.shard_sequence(Q, P)
    mine, ms, _ = mod.a2a_seq_to_head(q_seq, h, 1)
    ref, rs, _ = oracle.a2a_seq_to_head(q_seq, h)
    assert all(np.array_equal(a, b) for a, b in zip(mine, ref)) and ms == rs
    p = prob(P, 1, B, S, h, kv, D)
    o1 = mod.unshard(mod.forward(p, Q, K, V)["o_seq"])
    o2 = oracle.unshard_sequence(oracle.forward(p, Q, K, V)["o_seq"])
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_ring_one_is_ulysses():
    check_ring_one_is_ulysses(RG)


def check_ownership(mod):
    """P = 4 ranks in 2 ring positions of 2, 2 heads: rank (r, u) must hold
    chunk r (tokens [r*Cs, (r+1)*Cs)) of head u, in sequence order."""
    P, R, B, Sl, h, D = 4, 2, 1, 2, 2, 1
    x = []
    for s in range(P):
        a = np.zeros((B, Sl, h, D))
        for t in range(Sl):
            for g in range(h):
                a[0, t, g, 0] = 100 * (s * Sl + t) + g   # global token * 100 + head
        x.append(a)
    y, _, _ = mod.a2a_seq_to_head(x, h, R)
    Cs = Sl * P // R
    for r in range(R):
        for u in range(P // R):
            got = y[r * (P // R) + u][0, :, 0, 0]
            want = [100 * (r * Cs + i) + u for i in range(Cs)]
            assert got.tolist() == want, (r, u, got)


def test_ownership():
    check_ownership(RG)


def check_identity_and_bytes(mod):
    P, R, B, Sl, h, D, eb = 8, 2, 2, 3, 8, 4, 2
    x = [rnd((B, Sl, h, D), 20 + s) for s in range(P)]
    y, sent, recv = mod.a2a_seq_to_head(x, h, R, eb)
    back, sent2, _ = mod.a2a_head_to_seq(y, h, R, eb)
    assert all(np.array_equal(a, b) for a, b in zip(back, x))
    # [CMP] "DeepSpeed Attention costs": N(P-1)/P^2 per rank, here for the Pu
    # ranks of one ring position and N = the bytes of that position's chunk
    Pu = P // R
    N_chunk = B * Sl * Pu * h * D * eb
    assert sent == recv == sent2 == [N_chunk * (Pu - 1) // (Pu * Pu)] * P


def test_pack_unpack_identity_and_bytes():
    check_identity_and_bytes(RG)


def test_merge_is_softmax_over_the_union():
    """Splitting the keys in two and merging the two partial results gives
    block_attention over all keys, and a fully masked part changes nothing."""
    q, k, v = rnd((5, 4), 30), rnd((9, 4), 31), rnd((9, 4), 32)
    pos_q, pos_k = np.arange(10, 15), np.arange(9)
    full = RG.block_attention(q, k, v, pos_q, pos_k, 0.7, False)
    a = RG.block_attention(q, k[:4], v[:4], pos_q, pos_k[:4], 0.7, False)
    b = RG.block_attention(q, k[4:], v[4:], pos_q, pos_k[4:], 0.7, False)
    o, l = RG.merge(*a, *b)
    np.testing.assert_allclose(o, full[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(l, full[1], rtol=0, atol=1e-14)
    masked = RG.block_attention(q, k, v, np.zeros(5, dtype=int), pos_k + 1, 0.7, True)
    assert np.all(masked[1] == -np.inf) and not masked[0].any()
    o2, l2 = RG.merge(*full, *masked)
    assert np.array_equal(o2, full[0]) and np.array_equal(l2, full[1])


# ------------------------------------------------------------------ mutants

MUTANTS = [
    ("a ring step dropped", "                    for step in range(R):\n                        c = (r - step) % R          # the block",
     "                    for step in range(R - 1):\n                        c = (r - step) % R          # the block"),
    ("merge keeps the larger lse", "new = np.logaddexp(lse, lse_k)", "new = np.maximum(lse, lse_k)"),
    ("causal mask on chunk-local key positions", "k_pos = c * Cs + np.arange(Cs)\n                        o_k",
     "k_pos = np.arange(Cs)\n                        o_k"),
    ("pieces in reverse source order", "y[r * Pu + dst][:, src * Sl:(src + 1) * Sl]",
     "y[r * Pu + dst][:, (Pu - 1 - src) * Sl:(Pu - src) * Sl]"),
    ("ring positions strided", "= x_ranks[r * Pu + src][:, :, dst * hp:(dst + 1) * hp]",
     "= x_ranks[src * ring + r][:, :, dst * hp:(dst + 1) * hp]"),
    ("dK stays on the query rank", "dk[owner][b][:, kl] += scale * (ds.T @ q)", "dk[me][b][:, kl] += scale * (ds.T @ q)"),
    ("backward drops delta", "ds = p * (dp - delta[:, None])", "ds = p * dp"),
    ("own piece counted as traffic", "dst * hp:(dst + 1) * hp]\n                if src != dst:",
     "dst * hp:(dst + 1) * hp]\n                if True:"),
    ("replica holds the wrong kv-head", "[:, src * Sl:(src + 1) * Sl, 0] = x_ranks[r * Pu + src][:, :, dst // rep]",
     "[:, src * Sl:(src + 1) * Sl, 0] = x_ranks[r * Pu + src][:, :, dst % heads]"),
    ("replica gradient dropped", "                for j in range(rep):\n                    src = kv * rep + j",
     "                for j in range(1, rep):\n                    src = kv * rep + j"),
    ("block lse misses the max", "lse = np.where(live, ms + np.log(np.where(live, l, 1.0)), -np.inf)",
     "lse = np.where(live, np.log(np.where(live, l, 1.0)), -np.inf)"),
]


def mutant_module(old: str, new: str) -> types.ModuleType:
    text = open(SRC).read()
    assert text.count(old) == 1, old
    spec = importlib.util.spec_from_loader("oracle._ring_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    sys.modules["oracle._ring_mutant"] = mod
    exec(compile(text.replace(old, new), SRC, "exec"), mod.__dict__)
    return mod


def battery(mod):
    cases = [
        ("fwd", lambda: check_forward_equals_unsharded(mod, *CASES[0])),
        ("fwd-P>h", lambda: check_forward_equals_unsharded(mod, *CASES[1])),
        ("bwd", lambda: check_backward_equals_plain(mod, *CASES[0])),
        ("bwd-three", lambda: check_backward_equals_plain(mod, *CASES[4])),
        ("bwd-replicated", lambda: check_backward_equals_plain(mod, *CASES[5])),
        ("ulysses", lambda: check_ring_one_is_ulysses(mod)),
        ("ownership", lambda: check_ownership(mod)),
        ("bytes", lambda: check_identity_and_bytes(mod)),
    ]
    failed = []
    for name, fn in cases:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_unmutated_module_passes_battery():
    assert battery(mutant_module("import numpy as np", "import numpy as np")) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    assert battery(mutant_module(old, new)), f"no pin caught: {name}"
