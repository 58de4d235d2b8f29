"""Pure-Python brute force for tiny problems (S <= 16), standard library only.

TEST INFRASTRUCTURE ONLY: it exists to pin the C oracle.  It works on the
global, unsharded tensors (no ranks, no All-to-All), so agreement with the
sharded C oracle also checks that the Ulysses transposes are a pure
permutation of ownership ("Sequence Parallelism II: DeepSpeed Ulysses and
All-to-All Attention", §1 and §3).  Nested Python lists, `math` only.

Shapes: q [B][S][n_head][D], k/v [B][S][n_kv][D], out/dout [B][S][n_head*D].
"""
from __future__ import annotations

import math


def zeros(*dims):
    if len(dims) == 1:
        return [0.0] * dims[0]
    return [zeros(*dims[1:]) for _ in range(dims[0])]


def rope(x, base, direction=1):
    """Rotate-half rope on global positions: for i < D/2, angle p*base^(-2i/D)."""
    B, S, H, D = len(x), len(x[0]), len(x[0][0]), len(x[0][0][0])
    half = D // 2
    y = zeros(B, S, H, D)
    for b in range(B):
        for p in range(S):
            for h in range(H):
                v = x[b][p][h]
                for i in range(half):
                    a = direction * p * base ** (-2.0 * i / D)
                    y[b][p][h][i] = v[i] * math.cos(a) - v[i + half] * math.sin(a)
                    y[b][p][h][i + half] = v[i + half] * math.cos(a) + v[i] * math.sin(a)
    return y


def attention(q, k, v, causal, scale):
    """Softmax attention per head; q-head g reads kv-head g // (n_head/n_kv).
    Returns (o [B][S][n_head][D], lse [B][n_head][S])."""
    B, S, H, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    KV = len(k[0][0])
    group = H // KV
    o = zeros(B, S, H, D)
    lse = zeros(B, H, S)
    for b in range(B):
        for g in range(H):
            c = g // group
            for i in range(S):
                keys = range(i + 1) if causal else range(S)
                s = [scale * sum(q[b][i][g][e] * k[b][j][c][e] for e in range(D)) for j in keys]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                tot = sum(w)
                for e in range(D):
                    o[b][i][g][e] = sum(w[n] * v[b][j][c][e] for n, j in enumerate(keys)) / tot
                lse[b][g][i] = m + math.log(tot)
    return o, lse


def forward(Q, K, V, causal, scale, use_rope, base):
    """Attention module output in [B][S][H] (H = n_head*D, feature g*D+e)."""
    q = rope(Q, base) if use_rope else Q
    k = rope(K, base) if use_rope else K
    o, lse = attention(q, k, V, causal, scale)
    B, S, H, D = len(o), len(o[0]), len(o[0][0]), len(o[0][0][0])
    out = [[[o[b][p][g][e] for g in range(H) for e in range(D)] for p in range(S)] for b in range(B)]
    return out, lse


def backward(Q, K, V, dOut, causal, scale, use_rope, base):
    """Gradients of sum(dOut * forward(...)) w.r.t. the pre-rope Q, K and V,
    from the softmax-attention chain rule written out element by element."""
    q = rope(Q, base) if use_rope else Q
    k = rope(K, base) if use_rope else K
    v = V
    B, S, H, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    KV = len(k[0][0])
    group = H // KV
    o, lse = attention(q, k, v, causal, scale)
    dq = zeros(B, S, H, D)
    dk = zeros(B, S, KV, D)
    dv = zeros(B, S, KV, D)
    for b in range(B):
        for g in range(H):
            c = g // group
            for i in range(S):
                do = [dOut[b][i][g * D + e] for e in range(D)]
                delta = sum(do[e] * o[b][i][g][e] for e in range(D))
                keys = range(i + 1) if causal else range(S)
                for j in keys:
                    s = scale * sum(q[b][i][g][e] * k[b][j][c][e] for e in range(D))
                    p = math.exp(s - lse[b][g][i])
                    dp = sum(do[e] * v[b][j][c][e] for e in range(D))
                    ds = p * (dp - delta)
                    for e in range(D):
                        dv[b][j][c][e] += p * do[e]
                        dq[b][i][g][e] += scale * ds * k[b][j][c][e]
                        dk[b][j][c][e] += scale * ds * q[b][i][g][e]
    if use_rope:
        dq = rope(dq, base, -1)
        dk = rope(dk, base, -1)
    return dq, dk, dv


def loss(Q, K, V, dOut, causal, scale, use_rope, base):
    out, _ = forward(Q, K, V, causal, scale, use_rope, base)
    return sum(out[b][p][f] * dOut[b][p][f]
               for b in range(len(out)) for p in range(len(out[0])) for f in range(len(out[0][0])))


def linear(x, W, bias=None):
    """y[b][t][o] = sum_i x[b][t][i] * W[o][i] (+ bias[o]), in plain loops
    (x: [B][S][H] nested lists, W: [out][H])."""
    out = []
    for xb in x:
        rows = []
        for xt in xb:
            row = []
            for o, wo in enumerate(W):
                acc = 0.0
                for xi, wi in zip(xt, wo):
                    acc += xi * wi
                if bias is not None:
                    acc += bias[o]
                row.append(acc)
            rows.append(row)
        out.append(rows)
    return out
