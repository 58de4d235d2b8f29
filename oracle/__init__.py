"""fp64 CPU oracle of the Ulysses attention path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.  The
CUDA library and its Python binding never import it, and it imports nothing
from them.

The arithmetic lives in ``ulysses_oracle.c`` (plain loops, double precision);
this module only builds that file with gcc, marshals numpy buffers and strings
the steps together in the order the pages give them:

  [SP2] "Sequence Parallelism II: DeepSpeed Ulysses and All-to-All Attention",
        §2 "Forward Pass in Slow Motion" (split by sequence, project, All-to-All
        Q/K/V, local attention, All-to-All the output back) and §6 "Backward
        Pass Intuition" (the same layout changes, reversed);
  [CMP] "Comparing Ulysses and Megatron Sequence Parallelism", "A simple
        attention skeleton" (rope before the transpose) and "DeepSpeed
        Attention" (per-rank shapes [B,S/P,heads,D] <-> [B,S,heads/P,D]).

Every virtual rank holds its own numpy array; the All-to-All is the C double
loop over (destination, source) that also counts the bytes crossing ranks.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ulysses_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags: the file must give the
    same results on x86-64 and aarch64, so no -march and no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Shape(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int), ("B", ctypes.c_int), ("S", ctypes.c_int),
                ("n_head", ctypes.c_int), ("n_kv_head", ctypes.c_int), ("D", ctypes.c_int),
                ("causal", ctypes.c_int), ("scale", ctypes.c_double)]


def lib():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def load_library(path: str):
    """Load a compiled oracle (the tests also load deliberately broken
    builds of the same source, to check that the pins catch them)."""
    L = ctypes.CDLL(path)
    pp = ctypes.POINTER(ctypes.c_void_p)
    ll = ctypes.POINTER(ctypes.c_longlong)
    L.oracle_a2a_seq_to_head.argtypes = [ctypes.c_int] * 6 + [pp, pp, ll, ll, ctypes.c_int, ctypes.c_int]
    L.oracle_a2a_head_to_seq.argtypes = [ctypes.c_int] * 6 + [pp, pp, ll, ll, ctypes.c_int, ctypes.c_int]
    if hasattr(L, "oracle_a2a_seq_to_head_rep"):
        L.oracle_a2a_seq_to_head_rep.argtypes = [ctypes.c_int] * 6 + [pp, pp, ll, ll]
        L.oracle_reduce_head_to_seq_rep.argtypes = [ctypes.c_int] * 6 + [pp, pp, ll, ll]
    L.oracle_rope_seq.argtypes = [ctypes.c_int] * 5 + [ctypes.c_double, ctypes.c_int, pp]
    L.oracle_rope_seq.restype = None
    ip = ctypes.POINTER(ctypes.c_int)
    L.oracle_attention_fwd.argtypes = [ctypes.POINTER(_Shape), pp, pp, pp, pp, pp, ip,
                                       ctypes.c_long, ctypes.c_int]
    L.oracle_attention_unsharded.argtypes = [ctypes.POINTER(_Shape)] + [ctypes.c_void_p] * 5 + [ctypes.c_int]
    L.oracle_attention_bwd_group.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, pp, pp, pp, pp, pp, pp, pp, ip,
                                             ctypes.c_long, ip, ctypes.c_long, ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_double)]
    return L


@dataclasses.dataclass
class Problem:
    """The pages' problem statement ([CMP] skeleton and "Megatron Attention
    costs" constants): batch B, sequence S, n_head, n_kv_head, head_dim D,
    group size P; plus the causal flag and the rope base."""
    B: int
    S: int
    n_head: int
    n_kv_head: int
    D: int
    P: int
    causal: bool = True
    use_rope: bool = True
    rope_base: float = 10000.0
    scale: Optional[float] = None
    ring: int = 1  # > 1: the Ulysses x ring hybrid of oracle/ring.py (P = (P/ring) * ring)

    @property
    def Sl(self) -> int:
        return self.S // self.P

    @property
    def kv_replicas(self) -> int:
        """R = P / n_kv_head ranks hold each kv-head when n_kv_head < P, else 1."""
        return self.P // self.n_kv_head if self.n_kv_head < self.P else 1

    @property
    def kvp(self) -> int:
        """kv-heads a rank holds in head layout."""
        return self.n_kv_head // self.P if self.n_kv_head >= self.P else 1

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    def shape(self) -> _Shape:
        return _Shape(self.P, self.B, self.S, self.n_head, self.n_kv_head, self.D,
                      1 if self.causal else 0, self.softmax_scale)


def _nthreads(n: Optional[int]) -> int:
    return n if n else (os.cpu_count() or 1)


def _ptrs(arrays: Sequence[np.ndarray]):
    for a in arrays:
        assert a.dtype == np.float64 and a.flags.c_contiguous
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


def shard_sequence(x: np.ndarray, P: int) -> List[np.ndarray]:
    """[SP2] §2 first step: split [B, S, ...] by sequence into P contiguous
    chunks; rank r gets tokens [r*S/P, (r+1)*S/P)."""
    S = x.shape[1]
    assert S % P == 0
    Sl = S // P
    return [np.ascontiguousarray(x[:, r * Sl:(r + 1) * Sl], dtype=np.float64) for r in range(P)]


def unshard_sequence(xs: Sequence[np.ndarray]) -> np.ndarray:
    return np.concatenate(list(xs), axis=1)


def a2a_seq_to_head(x_ranks: Sequence[np.ndarray], heads: int, elem_bytes: int = 2,
                    skip: Optional[tuple] = None, fill: float = 0.0):
    """Loop All-to-All, [B,Sl,heads,D] per rank -> [B,S,heads/P,D] per rank.
    Returns (y_ranks, sent_bytes[P], recv_bytes[P])."""
    P = len(x_ranks)
    B, Sl, h, D = x_ranks[0].shape
    assert h == heads
    y = [np.full((B, Sl * P, heads // P, D), fill, dtype=np.float64) for _ in range(P)]
    sent = (ctypes.c_longlong * P)()
    recv = (ctypes.c_longlong * P)()
    ss, sd = skip if skip else (-1, -1)
    rc = lib().oracle_a2a_seq_to_head(P, B, Sl, heads, D, elem_bytes, _ptrs(x_ranks), _ptrs(y),
                                      sent, recv, ss, sd)
    if rc != 0:
        raise ValueError("heads must be a multiple of P")
    return y, list(sent), list(recv)


def a2a_seq_to_head_replicated(x_ranks: Sequence[np.ndarray], heads: int, elem_bytes: int = 2):
    """The kv All-to-All when heads < P (KV-head replication): rank d gets
    kv-head d / (P/heads) over the full sequence, [B,S,1,D] per rank.
    Returns (y_ranks, sent_bytes[P], recv_bytes[P])."""
    P = len(x_ranks)
    B, Sl, h, D = x_ranks[0].shape
    assert h == heads
    y = [np.zeros((B, Sl * P, 1, D), dtype=np.float64) for _ in range(P)]
    sent = (ctypes.c_longlong * P)()
    recv = (ctypes.c_longlong * P)()
    rc = lib().oracle_a2a_seq_to_head_rep(P, B, Sl, heads, D, elem_bytes, _ptrs(x_ranks), _ptrs(y), sent, recv)
    if rc != 0:
        raise ValueError("heads must divide P")
    return y, list(sent), list(recv)


def reduce_head_to_seq_replicated(y_ranks: Sequence[np.ndarray], heads: int, elem_bytes: int = 2):
    """Gradients of replicated kv-heads back to sequence layout: each kv-head's
    gradient is the sum of its replicas' ([B,S,1,D] per rank ->
    [B,Sl,heads,D])."""
    P = len(y_ranks)
    B, S, one, D = y_ranks[0].shape
    assert one == 1 and S % P == 0
    Sl = S // P
    y_ranks = [np.ascontiguousarray(a, dtype=np.float64) for a in y_ranks]
    x = [np.zeros((B, Sl, heads, D), dtype=np.float64) for _ in range(P)]
    sent = (ctypes.c_longlong * P)()
    recv = (ctypes.c_longlong * P)()
    rc = lib().oracle_reduce_head_to_seq_rep(P, B, Sl, heads, D, elem_bytes, _ptrs(y_ranks), _ptrs(x), sent, recv)
    if rc != 0:
        raise ValueError("heads must divide P")
    return x, list(sent), list(recv)


def a2a_head_to_seq(y_ranks: Sequence[np.ndarray], heads: int, elem_bytes: int = 2,
                    skip: Optional[tuple] = None, fill: float = 0.0):
    """Inverse loop All-to-All, [B,S,heads/P,D] per rank -> [B,Sl,heads,D]."""
    P = len(y_ranks)
    B, S, hp, D = y_ranks[0].shape
    assert hp * P == heads and S % P == 0
    Sl = S // P
    x = [np.full((B, Sl, heads, D), fill, dtype=np.float64) for _ in range(P)]
    sent = (ctypes.c_longlong * P)()
    recv = (ctypes.c_longlong * P)()
    ss, sd = skip if skip else (-1, -1)
    rc = lib().oracle_a2a_head_to_seq(P, B, Sl, heads, D, elem_bytes, _ptrs(y_ranks), _ptrs(x),
                                      sent, recv, ss, sd)
    if rc != 0:
        raise ValueError("heads must be a multiple of P")
    return x, list(sent), list(recv)


def rope_seq(x_ranks: Sequence[np.ndarray], base: float, direction: int = 1) -> List[np.ndarray]:
    """Rotate copies of the per-rank [B,Sl,heads,D] buffers by global position
    (direction=-1: inverse rotation)."""
    out = [np.array(a, dtype=np.float64, copy=True) for a in x_ranks]
    P = len(out)
    B, Sl, h, D = out[0].shape
    lib().oracle_rope_seq(P, B, Sl, h, D, float(base), int(direction), _ptrs(out))
    return out


def rope_rows(x: np.ndarray, positions: Sequence[int], base: float) -> np.ndarray:
    """The rotation of rope_seq for rows at arbitrary global positions:
    x [n, heads, D], positions [n]; rotate-half, angle p * base^(-2i/D)."""
    x = np.asarray(x, dtype=np.float64)
    n, heads, D = x.shape
    half = D // 2
    i = np.arange(half, dtype=np.float64)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * np.power(float(base), -2.0 * i / D)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def attention_fwd(prob: Problem, q_head, k_head, v_head, rows=None, nthreads=None):
    """Per-rank attention over the full sequence for the rank's heads.
    Returns (o_head ranks [B,S,hp,D], lse ranks [B,hp,S]); rows not in `rows`
    stay NaN."""
    P, B, S, hp, D = prob.P, prob.B, prob.S, prob.n_head // prob.P, prob.D
    o = [np.full((B, S, hp, D), np.nan) for _ in range(P)]
    lse = [np.full((B, hp, S), np.nan) for _ in range(P)]
    sh = prob.shape()
    if rows is not None:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32)
        rp, nr = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), len(rows_arr)
    else:
        rows_arr, rp, nr = None, None, 0
    rc = lib().oracle_attention_fwd(ctypes.byref(sh), _ptrs(q_head), _ptrs(k_head), _ptrs(v_head),
                                    _ptrs(o), _ptrs(lse), rp, nr, _nthreads(nthreads))
    if rc != 0:
        raise ValueError("head counts do not divide")
    return o, lse


def attention_unsharded(prob: Problem, q, k, v, nthreads=None):
    """Plain attention on global [B,S,heads,D] tensors (no ranks at all)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    o = np.zeros_like(q)
    lse = np.zeros((prob.B, prob.n_head, prob.S))
    sh = prob.shape()
    rc = lib().oracle_attention_unsharded(ctypes.byref(sh), q.ctypes.data, k.ctypes.data,
                                          v.ctypes.data, o.ctypes.data, lse.ctypes.data,
                                          _nthreads(nthreads))
    if rc != 0:
        raise ValueError("head counts do not divide")
    return o, lse


def attention_bwd(prob: Problem, q_head, k_head, v_head, do_head, groups=None,
                  q_rows=None, kv_rows=None, nthreads=None, phase_seconds=None):
    """Backward on head-sharded buffers for the listed (rank, batch, local
    kv-head) groups (default: all).  Returns (dq, dk, dv) head-layout ranks;
    entries not computed stay NaN.  `phase_seconds` (a list, optional) gets
    the wall time of each group's three phases appended (timing only)."""
    P, B, S, D = prob.P, prob.B, prob.S, prob.D
    hp, kvp = prob.n_head // P, prob.kvp
    dq = [np.full((B, S, hp, D), np.nan) for _ in range(P)]
    dk = [np.full((B, S, kvp, D), np.nan) for _ in range(P)]
    dv = [np.full((B, S, kvp, D), np.nan) for _ in range(P)]
    if groups is None:
        groups = [(r, b, kl) for r in range(P) for b in range(B) for kl in range(kvp)]
    qa = np.ascontiguousarray(q_rows, dtype=np.int32) if q_rows is not None else None
    ka = np.ascontiguousarray(kv_rows, dtype=np.int32) if kv_rows is not None else None
    ip = ctypes.POINTER(ctypes.c_int)
    sh = prob.shape()
    ptrs = [_ptrs(x) for x in (q_head, k_head, v_head, do_head, dq, dk, dv)]
    for (r, b, kl) in groups:
        secs = (ctypes.c_double * 3)()
        rc = lib().oracle_attention_bwd_group(
            ctypes.byref(sh), r, b, kl, *ptrs,
            qa.ctypes.data_as(ip) if qa is not None else None, len(qa) if qa is not None else 0,
            ka.ctypes.data_as(ip) if ka is not None else None, len(ka) if ka is not None else 0,
            _nthreads(nthreads), secs)
        if rc != 0:
            raise ValueError(f"oracle backward failed ({rc})")
        if phase_seconds is not None:
            phase_seconds.append(tuple(secs))
    return dq, dk, dv


# --------------------------------------------------------------------------
# The whole path, in the pages' order.
# --------------------------------------------------------------------------

def forward(prob: Problem, Q, K, V, rows=None, elem_bytes=2, nthreads=None):
    """[SP2] §2: split by sequence; rope q, k at global positions ([CMP]
    skeleton); All-to-All Q, K, V (seq -> head); local attention; All-to-All
    the output back (head -> seq).  Q: [B,S,n_head,D], K/V: [B,S,n_kv,D]
    global arrays of the already-rounded input values.  Returns a dict with
    every intermediate, the output o_seq ranks [B,Sl,n_head,D] and the bytes
    each A2A moved."""
    P = prob.P
    q_seq, k_seq, v_seq = (shard_sequence(np.asarray(t, dtype=np.float64), P) for t in (Q, K, V))
    if prob.use_rope:
        q_seq = rope_seq(q_seq, prob.rope_base, +1)
        k_seq = rope_seq(k_seq, prob.rope_base, +1)
    q_head, sq, _ = a2a_seq_to_head(q_seq, prob.n_head, elem_bytes)
    # with fewer kv-heads than ranks each kv-head goes to the R ranks whose
    # q-heads read it (KV-head replication)
    kv_a2a = a2a_seq_to_head_replicated if prob.kv_replicas > 1 else a2a_seq_to_head
    k_head, sk, _ = kv_a2a(k_seq, prob.n_kv_head, elem_bytes)
    v_head, sv, _ = kv_a2a(v_seq, prob.n_kv_head, elem_bytes)
    o_head, lse = attention_fwd(prob, q_head, k_head, v_head, rows=rows, nthreads=nthreads)
    if rows is None:
        o_seq, so, _ = a2a_head_to_seq(o_head, prob.n_head, elem_bytes)
    else:
        o_seq, so = None, None
    return dict(q_seq_roped=q_seq, k_seq_roped=k_seq, q_head=q_head, k_head=k_head, v_head=v_head,
                o_head=o_head, lse=lse, o_seq=o_seq,
                sent=dict(q=sq, k=sk, v=sv, o=so))


def backward(prob: Problem, Q, K, V, dO, groups=None, q_rows=None, kv_rows=None,
             elem_bytes=2, nthreads=None):
    """[SP2] §6: the output gradient dO ([B,S,H] global, H = n_head*D) is
    split by sequence and All-to-All'd into head layout; per-head attention
    backward; dQ, dK, dV are All-to-All'd back to sequence layout; the rope
    rotation is undone on dQ and dK (gradients w.r.t. the pre-rope q, k).
    Returns dict with dq_seq/dk_seq/dv_seq ranks and the head-layout
    gradients."""
    P, B, S, D = prob.P, prob.B, prob.S, prob.D
    fw = forward(prob, Q, K, V, rows=[0], elem_bytes=elem_bytes, nthreads=nthreads)
    do_glob = np.asarray(dO, dtype=np.float64).reshape(B, S, prob.n_head, D)
    do_seq = shard_sequence(do_glob, P)
    do_head, sdo, _ = a2a_seq_to_head(do_seq, prob.n_head, elem_bytes)
    dq_h, dk_h, dv_h = attention_bwd(prob, fw["q_head"], fw["k_head"], fw["v_head"], do_head,
                                     groups=groups, q_rows=q_rows, kv_rows=kv_rows,
                                     nthreads=nthreads)
    dq_seq, sdq, _ = a2a_head_to_seq(dq_h, prob.n_head, elem_bytes, fill=np.nan)
    if prob.kv_replicas > 1:
        # each replica holds a partial dK, dV (its own q-heads' share): summed
        dk_seq, sdk, _ = reduce_head_to_seq_replicated(dk_h, prob.n_kv_head, elem_bytes)
        dv_seq, sdv, _ = reduce_head_to_seq_replicated(dv_h, prob.n_kv_head, elem_bytes)
    else:
        dk_seq, sdk, _ = a2a_head_to_seq(dk_h, prob.n_kv_head, elem_bytes, fill=np.nan)
        dv_seq, sdv, _ = a2a_head_to_seq(dv_h, prob.n_kv_head, elem_bytes, fill=np.nan)
    if prob.use_rope:
        dq_seq = rope_seq(dq_seq, prob.rope_base, -1)
        dk_seq = rope_seq(dk_seq, prob.rope_base, -1)
    return dict(dq_seq=dq_seq, dk_seq=dk_seq, dv_seq=dv_seq, dq_head=dq_h, dk_head=dk_h,
                dv_head=dv_h, do_head=do_head, q_head=fw["q_head"], k_head=fw["k_head"],
                v_head=fw["v_head"], sent=dict(do=sdo, dq=sdq, dk=sdk, dv=sdv))


def qkv_projection(prob: Problem, x_ranks: Sequence[np.ndarray], W: np.ndarray, bias=None):
    """[SP2] §2 second step ("run the QKV projections for the local sequence
    chunk"; the rank has the full projection weights) and [CMP] "A simple
    attention skeleton" (q/k/v projections of x, then view as heads): every
    rank applies the complete, replicated projection to its own tokens.
    x_r: [B, Sl, H] per rank; W: [(n_head + 2 n_kv_head) * D, H] -- the three
    projection weights stacked (q rows, then k, then v) in the Linear layout
    [out_features, in_features]; bias: [(n_head + 2 n_kv_head) * D] or None.
    Returns per-rank q [B,Sl,n_head,D], k and v [B,Sl,n_kv_head,D]:
    y = x W^T (+ b), the matrix product taken from numpy."""
    D, h, kv = prob.D, prob.n_head, prob.n_kv_head
    W = np.asarray(W, dtype=np.float64)
    assert W.shape[0] == (h + 2 * kv) * D
    q, k, v = [], [], []
    for x in x_ranks:
        x = np.asarray(x, dtype=np.float64)
        B, Sl, H = x.shape
        assert W.shape[1] == H
        y = x.reshape(B * Sl, H) @ W.T
        if bias is not None:
            y = y + np.asarray(bias, dtype=np.float64)[None, :]
        y = y.reshape(B, Sl, h + 2 * kv, D)
        q.append(np.ascontiguousarray(y[:, :, :h]))
        k.append(np.ascontiguousarray(y[:, :, h:h + kv]))
        v.append(np.ascontiguousarray(y[:, :, h + kv:]))
    return q, k, v


def project_and_pack(prob: Problem, x_ranks, W, bias=None, elem_bytes=2):
    """Projection, RoPE on q and k at global positions, and the seq -> head
    All-to-All ([CMP] skeleton order: project, rope, then transpose), with
    KV-head replication when n_kv_head < P.  Returns q_head, k_head, v_head."""
    q, k, v = qkv_projection(prob, x_ranks, W, bias)
    if prob.use_rope:
        q = rope_seq(q, prob.rope_base, +1)
        k = rope_seq(k, prob.rope_base, +1)
    q_head, _, _ = a2a_seq_to_head(q, prob.n_head, elem_bytes)
    kv_a2a = a2a_seq_to_head_replicated if prob.kv_replicas > 1 else a2a_seq_to_head
    k_head, _, _ = kv_a2a(k, prob.n_kv_head, elem_bytes)
    v_head, _, _ = kv_a2a(v, prob.n_kv_head, elem_bytes)
    return q_head, k_head, v_head


def unpack_and_project(prob: Problem, o_head, W: np.ndarray, bias=None, elem_bytes=2):
    """[SP2] §2 fifth step and [CMP] "DeepSpeed Attention": the head -> seq
    All-to-All restores [B, S/P, H] on every rank, which then applies the
    complete (replicated) output projection to its own tokens ([CMP]
    skeleton: y = output_proj(y)).  o_head ranks [B,S,hp,D]; W [hidden,
    n_head*D] in the Linear layout [out, in]; bias [hidden] or None.
    Returns y ranks [B, Sl, hidden]: y = o W^T (+ b), numpy's matrix product."""
    o_seq, _, _ = a2a_head_to_seq(o_head, prob.n_head, elem_bytes)
    W = np.asarray(W, dtype=np.float64)
    out = []
    for o in o_seq:
        B, Sl, h, D = o.shape
        y = o.reshape(B * Sl, h * D) @ W.T
        if bias is not None:
            y = y + np.asarray(bias, dtype=np.float64)[None, :]
        out.append(y.reshape(B, Sl, W.shape[0]))
    return out


def unsharded(prob: Problem, Q, K, V, nthreads=None):
    """The same attention with no ranks: rope on global positions (one rank
    holding everything), then plain attention on [B,S,heads,D]."""
    q = np.asarray(Q, dtype=np.float64)
    k = np.asarray(K, dtype=np.float64)
    if prob.use_rope:
        q = rope_seq([q], prob.rope_base, +1)[0]
        k = rope_seq([k], prob.rope_base, +1)[0]
    return attention_unsharded(prob, q, k, np.asarray(V, dtype=np.float64), nthreads=nthreads)
