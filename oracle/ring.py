"""fp64 oracle of the Ulysses x ring (context-parallel) hybrid.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only the tests,
``__graft_entry__.smoke()`` and the CPU leg of ``bench.py`` use it.

Sources, cited by page title and section:

  [SP2] "Sequence Parallelism II: DeepSpeed Ulysses and All-to-All Attention",
        §4 (a head-sharded group cannot have more ranks than heads; going
        further needs another level of hierarchy or parallel dimension) and §8
        (Ring Attention keeps each rank's query block and circulates the
        key/value blocks, so one head's context may exceed one rank).

The pages name the combination but print no algorithm for it.  The reading
taken (the plainest one the rest of the pages supports):

  * P = Pu * R ranks.  Rank p = r*Pu + u sits at ring position r and is member
    u of that position's Ulysses group.  Token ownership is unchanged: rank p
    owns tokens [p*Sl, (p+1)*Sl), so the Pu ranks of ring position r together
    own chunk r = tokens [r*Cs, (r+1)*Cs), Cs = S/R.
  * The Ulysses All-to-All runs inside each ring position over its Pu ranks:
    rank (r, u) receives heads [u*hp, (u+1)*hp), hp = n_head/Pu (kv-heads
    likewise), of the whole chunk r, pieces in source order ([SP2] §1).  With
    fewer kv-heads than Pu (Pu a multiple of n_kv_head) each kv-head goes to
    the rep = Pu/n_kv_head members whose q-heads read it, member u holding
    kv-head u // rep, and a kv-head's gradient is the sum of its replicas'
    (the KV-head replication of plain Ulysses, inside each ring position).
  * Ring attention over the R ranks (0, u) ... (R-1, u) that hold the same
    heads: rank (r, u) keeps its query block (chunk r); at ring step k it
    works on the key/value block of chunk c = (r - k) mod R, the blocks moving
    one rank along the ring per step.  Each step's partial result (o_k,
    lse_k) over that block is merged into the running one with log-sum-exp
    weights.  Causal masking uses global positions: blocks of later chunks
    are entirely masked and contribute nothing, the own chunk (step 0) is
    masked on the diagonal.
  * Backward, with the final lse of every query row: at each ring step the
    query rank recomputes P for the visiting block, accumulates its dQ, and
    the block's dK, dV accumulate with the block and travel back to its owner.
  * The inverse Ulysses All-to-All inside each ring position returns O (and
    dQ, dK, dV, with the RoPE rotation undone on dQ, dK) to sequence layout.

Steps use numpy (matmul, exp, logaddexp) on per-rank arrays; the copies of the
All-to-All are explicit loops over (ring position, destination, source).
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np

from . import Problem, rope_seq, shard_sequence


def dims(prob: Problem):
    """(Pu, R, Cs, hp, kvp) of a hybrid problem; kvp = 1 with replicated kv-heads."""
    R = prob.ring
    assert R >= 1 and prob.P % R == 0 and prob.S % prob.P == 0
    Pu = prob.P // R
    kv = prob.n_kv_head
    assert prob.n_head % Pu == 0 and prob.n_head % kv == 0 and (kv % Pu == 0 or Pu % kv == 0)
    return Pu, R, prob.S // R, prob.n_head // Pu, kv // Pu if kv >= Pu else 1


def kv_replicas(prob: Problem) -> int:
    """Members of a ring position holding each kv-head (1 unless n_kv_head < Pu)."""
    Pu = prob.P // prob.ring
    return Pu // prob.n_kv_head if prob.n_kv_head < Pu else 1


def a2a_seq_to_head(x_ranks: Sequence[np.ndarray], heads: int, ring: int, elem_bytes: int = 2):
    """The Ulysses All-to-All of every ring position: per rank [B,Sl,heads,D]
    -> [B,Cs,heads/Pu,D].  Returns (y_ranks, sent_bytes[P], recv_bytes[P])."""
    P = len(x_ranks)
    Pu = P // ring
    B, Sl, h, D = x_ranks[0].shape
    assert h == heads and heads % Pu == 0
    hp = heads // Pu
    y = [np.zeros((B, Sl * Pu, hp, D)) for _ in range(P)]
    sent, recv = [0] * P, [0] * P
    piece = B * Sl * hp * D * elem_bytes
    for r in range(ring):
        for dst in range(Pu):
            for src in range(Pu):
                # rank (r, src) sends its tokens of heads [dst*hp, (dst+1)*hp) to
                # rank (r, dst), which stores them at sequence block src
                y[r * Pu + dst][:, src * Sl:(src + 1) * Sl] = x_ranks[r * Pu + src][:, :, dst * hp:(dst + 1) * hp]
                if src != dst:
                    sent[r * Pu + src] += piece
                    recv[r * Pu + dst] += piece
    return y, sent, recv


def a2a_seq_to_head_replicated(x_ranks: Sequence[np.ndarray], heads: int, ring: int, elem_bytes: int = 2):
    """The kv All-to-All of every ring position when heads < Pu: member u of
    ring position r receives kv-head u // rep (rep = Pu/heads) of chunk r.
    Per rank [B,Sl,heads,D] -> [B,Cs,1,D]."""
    P = len(x_ranks)
    Pu = P // ring
    B, Sl, h, D = x_ranks[0].shape
    assert h == heads and Pu % heads == 0
    rep = Pu // heads
    y = [np.zeros((B, Sl * Pu, 1, D)) for _ in range(P)]
    sent, recv = [0] * P, [0] * P
    piece = B * Sl * D * elem_bytes
    for r in range(ring):
        for dst in range(Pu):
            for src in range(Pu):
                y[r * Pu + dst][:, src * Sl:(src + 1) * Sl, 0] = x_ranks[r * Pu + src][:, :, dst // rep]
                if src != dst:
                    sent[r * Pu + src] += piece
                    recv[r * Pu + dst] += piece
    return y, sent, recv


def reduce_head_to_seq_replicated(y_ranks: Sequence[np.ndarray], heads: int, ring: int, elem_bytes: int = 2):
    """Adjoint of a2a_seq_to_head_replicated: kv-head kv of sequence rank
    (r, dst) = the sum over its rep replicas (members kv*rep + j, j in order)
    of their rows.  Per rank [B,Cs,1,D] -> [B,Sl,heads,D]."""
    P = len(y_ranks)
    Pu = P // ring
    B, Cs, one, D = y_ranks[0].shape
    assert one == 1 and Pu % heads == 0 and Cs % Pu == 0
    rep, Sl = Pu // heads, Cs // Pu
    x = [np.zeros((B, Sl, heads, D)) for _ in range(P)]
    sent, recv = [0] * P, [0] * P
    piece = B * Sl * D * elem_bytes
    for r in range(ring):
        for dst in range(Pu):
            for kv in range(heads):
                for j in range(rep):
                    src = kv * rep + j
                    x[r * Pu + dst][:, :, kv] += y_ranks[r * Pu + src][:, dst * Sl:(dst + 1) * Sl, 0]
                    if src != dst:
                        sent[r * Pu + src] += piece
                        recv[r * Pu + dst] += piece
    return x, sent, recv


def a2a_head_to_seq(y_ranks: Sequence[np.ndarray], heads: int, ring: int, elem_bytes: int = 2):
    """Inverse of a2a_seq_to_head: per rank [B,Cs,hp,D] -> [B,Sl,heads,D]."""
    P = len(y_ranks)
    Pu = P // ring
    B, Cs, hp, D = y_ranks[0].shape
    assert hp * Pu == heads and Cs % Pu == 0
    Sl = Cs // Pu
    x = [np.zeros((B, Sl, heads, D)) for _ in range(P)]
    sent, recv = [0] * P, [0] * P
    piece = B * Sl * hp * D * elem_bytes
    for r in range(ring):
        for dst in range(Pu):          # sequence side
            for src in range(Pu):      # head side
                x[r * Pu + dst][:, :, src * hp:(src + 1) * hp] = y_ranks[r * Pu + src][:, dst * Sl:(dst + 1) * Sl]
                if src != dst:
                    sent[r * Pu + src] += piece
                    recv[r * Pu + dst] += piece
    return x, sent, recv


def block_attention(q, k, v, q_pos, k_pos, scale: float, causal: bool):
    """Softmax attention of query rows q [n,D] over one key/value block k, v
    [m,D] at global positions q_pos [n], k_pos [m]: returns (o [n,D], lse [n]).
    Rows with every key masked get o = 0 and lse = -inf."""
    s = scale * (q @ k.T)
    if causal:
        s = np.where(k_pos[None, :] <= q_pos[:, None], s, -np.inf)
    m = s.max(axis=1)
    live = np.isfinite(m)
    ms = np.where(live, m, 0.0)
    w = np.exp(s - ms[:, None])
    l = w.sum(axis=1)
    o = np.zeros((q.shape[0], v.shape[1]))
    o[live] = (w[live] @ v) / l[live, None]
    lse = np.where(live, ms + np.log(np.where(live, l, 1.0)), -np.inf)
    return o, lse


def merge(o, lse, o_k, lse_k):
    """Merge a ring step's partial result into the running one: the combined
    softmax over the union of the key blocks is the lse-weighted mean."""
    new = np.logaddexp(lse, lse_k)
    fin = np.isfinite(new)
    safe = np.where(fin, new, 0.0)
    a = np.where(fin, np.exp(lse - safe), 0.0)
    b = np.where(fin, np.exp(lse_k - safe), 0.0)
    return a[:, None] * o + b[:, None] * o_k, new


def ring_attention_fwd(prob: Problem, q_head, k_head, v_head, rows: Optional[Sequence[int]] = None):
    """Ring attention on the hybrid's head layout.  q_head ranks [B,Cs,hp,D],
    k/v [B,Cs,kvp,D].  Returns (o_head [B,Cs,hp,D], lse [B,hp,Cs]) per rank;
    with `rows` (global positions) only those query rows, the rest NaN."""
    Pu, R, Cs, hp, kvp = dims(prob)
    B, D = prob.B, prob.D
    G = hp // kvp
    scale = prob.softmax_scale
    o = [np.full((B, Cs, hp, D), np.nan) for _ in range(prob.P)]
    lse = [np.full((B, hp, Cs), np.nan) for _ in range(prob.P)]
    for r in range(R):
        mine = np.arange(Cs) if rows is None else np.array(
            sorted(p - r * Cs for p in set(rows) if r * Cs <= p < (r + 1) * Cs), dtype=np.int64)
        if len(mine) == 0:
            continue
        q_pos = r * Cs + mine
        for u in range(Pu):
            me = r * Pu + u
            for b in range(B):
                for j in range(hp):
                    kl = j // G
                    acc_o = np.zeros((len(mine), D))
                    acc_l = np.full(len(mine), -np.inf)
                    for step in range(R):
                        c = (r - step) % R          # the block visiting at this step
                        owner = c * Pu + u
                        k_pos = c * Cs + np.arange(Cs)
                        o_k, l_k = block_attention(q_head[me][b][mine, j], k_head[owner][b][:, kl],
                                                   v_head[owner][b][:, kl], q_pos, k_pos, scale, prob.causal)
                        acc_o, acc_l = merge(acc_o, acc_l, o_k, l_k)
                    o[me][b][mine, j] = acc_o
                    lse[me][b][j, mine] = acc_l
    return o, lse


def ring_attention_bwd(prob: Problem, q_head, k_head, v_head, do_head, o_head, lse):
    """Backward of ring_attention_fwd (o_head, lse: its full results).
    Returns (dq, dk, dv) in the hybrid's head layout."""
    Pu, R, Cs, hp, kvp = dims(prob)
    B, D = prob.B, prob.D
    G = hp // kvp
    scale = prob.softmax_scale
    dq = [np.zeros((B, Cs, hp, D)) for _ in range(prob.P)]
    dk = [np.zeros((B, Cs, kvp, D)) for _ in range(prob.P)]
    dv = [np.zeros((B, Cs, kvp, D)) for _ in range(prob.P)]
    for r in range(R):
        q_pos = r * Cs + np.arange(Cs)
        for u in range(Pu):
            me = r * Pu + u
            for b in range(B):
                for j in range(hp):
                    kl = j // G
                    q = q_head[me][b][:, j]
                    do = do_head[me][b][:, j]
                    delta = np.sum(do * o_head[me][b][:, j], axis=1)
                    L = lse[me][b][j]
                    for step in range(R):
                        c = (r - step) % R
                        owner = c * Pu + u
                        k_pos = c * Cs + np.arange(Cs)
                        k = k_head[owner][b][:, kl]
                        v = v_head[owner][b][:, kl]
                        s = scale * (q @ k.T)
                        if prob.causal:
                            s = np.where(k_pos[None, :] <= q_pos[:, None], s, -np.inf)
                        p = np.exp(s - L[:, None])
                        dp = do @ v.T
                        ds = p * (dp - delta[:, None])
                        dq[me][b][:, j] += scale * (ds @ k)
                        # the visiting block's gradients travel back to its owner
                        dk[owner][b][:, kl] += scale * (ds.T @ q)
                        dv[owner][b][:, kl] += p.T @ do
    return dq, dk, dv


def forward(prob: Problem, Q, K, V, rows=None, elem_bytes: int = 2):
    """The hybrid forward in the pages' order: split by sequence, rope at global
    positions, Ulysses All-to-All inside each ring position, ring attention,
    inverse All-to-All.  Q [B,S,n_head,D], K/V [B,S,n_kv,D]."""
    P = prob.P
    q_seq, k_seq, v_seq = (shard_sequence(np.asarray(t, dtype=np.float64), P) for t in (Q, K, V))
    if prob.use_rope:
        q_seq = rope_seq(q_seq, prob.rope_base, +1)
        k_seq = rope_seq(k_seq, prob.rope_base, +1)
    q_head, sq, _ = a2a_seq_to_head(q_seq, prob.n_head, prob.ring, elem_bytes)
    kv_a2a = a2a_seq_to_head_replicated if kv_replicas(prob) > 1 else a2a_seq_to_head
    k_head, sk, _ = kv_a2a(k_seq, prob.n_kv_head, prob.ring, elem_bytes)
    v_head, sv, _ = kv_a2a(v_seq, prob.n_kv_head, prob.ring, elem_bytes)
    o_head, lse = ring_attention_fwd(prob, q_head, k_head, v_head, rows=rows)
    o_seq = a2a_head_to_seq(o_head, prob.n_head, prob.ring, elem_bytes)[0] if rows is None else None
    return dict(q_head=q_head, k_head=k_head, v_head=v_head, o_head=o_head, lse=lse, o_seq=o_seq,
                sent=dict(q=sq, k=sk, v=sv))


def backward(prob: Problem, Q, K, V, dO, elem_bytes: int = 2):
    """The hybrid backward: dO ([B,S,H]) split by sequence and All-to-All'd
    inside each ring position, ring backward, dQ/dK/dV back to sequence layout
    with the rope rotation undone on dQ and dK."""
    B, S, D = prob.B, prob.S, prob.D
    fw = forward(prob, Q, K, V, elem_bytes=elem_bytes)
    do_seq = shard_sequence(np.asarray(dO, dtype=np.float64).reshape(B, S, prob.n_head, D), prob.P)
    do_head = a2a_seq_to_head(do_seq, prob.n_head, prob.ring, elem_bytes)[0]
    dq_h, dk_h, dv_h = ring_attention_bwd(prob, fw["q_head"], fw["k_head"], fw["v_head"], do_head,
                                          fw["o_head"], fw["lse"])
    dq_seq = a2a_head_to_seq(dq_h, prob.n_head, prob.ring, elem_bytes)[0]
    kv_back = reduce_head_to_seq_replicated if kv_replicas(prob) > 1 else a2a_head_to_seq
    dk_seq = kv_back(dk_h, prob.n_kv_head, prob.ring, elem_bytes)[0]
    dv_seq = kv_back(dv_h, prob.n_kv_head, prob.ring, elem_bytes)[0]
    if prob.use_rope:
        dq_seq = rope_seq(dq_seq, prob.rope_base, -1)
        dk_seq = rope_seq(dk_seq, prob.rope_base, -1)
    return dict(dq_seq=dq_seq, dk_seq=dk_seq, dv_seq=dv_seq, dq_head=dq_h, dk_head=dk_h, dv_head=dv_h,
                o_head=fw["o_head"], lse=fw["lse"])


def unshard(xs: Sequence[np.ndarray]) -> np.ndarray:
    """Sequence-layout ranks [B,Sl,heads,D] -> the global [B,S,heads,D]."""
    return np.concatenate(list(xs), axis=1)


__all__: List[str] = ["dims", "kv_replicas", "a2a_seq_to_head", "a2a_seq_to_head_replicated",
                      "reduce_head_to_seq_replicated", "a2a_head_to_seq", "block_attention", "merge",
                      "ring_attention_fwd", "ring_attention_bwd", "forward", "backward", "unshard"]
