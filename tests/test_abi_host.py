"""The C-ABI library without a GPU: it loads, exports every entry point that
include/ulysses.h declares, and its host-side validation returns the
documented codes.  Every call here fails validation before any launch (the
pointers are fake addresses that are never dereferenced)."""
import ctypes
import os
import re

import pytest

from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ulysses.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(U.LIB_PATH):
        B.build()
    return U.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(ulysses_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_entry_point(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(U.EXPORTS) <= set(names)


def prob(**kw):
    base = dict(B=1, S=4096, hidden=4096, n_head=32, n_kv_head=8, head_dim=128, P=8, causal=True,
                dtype=U.BF16, use_rope=True, rope_base=10000.0)
    base.update(kw)
    return U.Problem(**base)


@pytest.mark.parametrize("kw,code", [
    ({}, 0),
    (dict(B=0), -1), (dict(S=-4), -1), (dict(P=0), -1), (dict(rope_base=0.0), -1),
    (dict(rope_base=0.0, use_rope=False), 0), (dict(softmax_scale=-1.0), -1),
    (dict(S=4100), -2),                        # S % P
    (dict(n_head=36, hidden=36 * 128), -2),    # n_head % P
    (dict(n_kv_head=4), 0),                    # n_kv_head < P, P a multiple: kv-heads replicated (R = 2)
    (dict(n_kv_head=1), 0),                    # one kv-head on every rank (R = 8)
    (dict(n_head=48, hidden=48 * 128, n_kv_head=12), -2),  # neither of n_kv_head, P divides the other
    (dict(P=64, S=4096 * 64), -2),             # P > n_head: the head-count bound
    (dict(n_kv_head=24), -2),                  # n_head % n_kv_head
    (dict(hidden=1024), -3),
    (dict(head_dim=96, hidden=32 * 96), -4), (dict(dtype=7), -4),
    (dict(dtype=U.FP32, head_dim=32, hidden=1024), 0),
    # Ulysses x ring hybrid: the head-count bound applies to the Pu = P/ring ranks of a ring position
    (dict(P=64, S=4096 * 64, n_kv_head=32, ring=2), 0),  # P = 64 > 32 heads: 2 ring positions of 32
    (dict(P=256, S=32768, n_kv_head=32, ring=8), 0),     # the pages' 32 heads over 256 ranks
    (dict(ring=8), 0),                         # pure ring: one rank per position
    (dict(P=64, S=4096 * 64, ring=3), -2),     # P % ring
    (dict(ring=-1), -1),
    (dict(ring=2, dtype=U.FP32), -4),          # the hybrid runs on the bf16 tensor-core kernels only
    (dict(ring=2, head_dim=32, hidden=32 * 32), -4),
    (dict(S=8 * 96, ring=4), -4),              # chunk S/ring = 192 is not a multiple of 128
    (dict(ring=2, n_kv_head=2), 0),            # kv-head replication inside a ring position (Pu = 4)
    (dict(ring=2, n_kv_head=3, n_head=24, hidden=24 * 128), -2),  # neither of n_kv_head, Pu divides the other
])
def test_validate_codes(lib, kw, code):
    assert U.ulysses_validate(prob(**kw)) == code


def test_workspace_sizes(lib):
    p = prob()
    f, b = U.ulysses_workspace_bytes(p, 0), U.ulysses_workspace_bytes(p, 1)
    assert f >= 256 + p.S * p.head_dim * 4 and f % 256 == 0
    # backward adds delta [B][n_head][S] fp32 and dO in head layout
    assert b >= f + p.B * p.n_head * p.S * 4 + p.B * p.S * p.n_head * p.head_dim * 2
    assert U.ulysses_workspace_bytes(prob(use_rope=False), 0) == 256
    # replicated kv-heads: the backward also holds every rank's float partial dK and dV
    pr = prob(n_kv_head=2)
    assert U.ulysses_workspace_bytes(pr, 1) >= b + 2 * pr.P * pr.B * pr.S * pr.head_dim * 4
    assert U.ulysses_workspace_bytes(prob(B=0), 0) == 0
    assert U.ulysses_workspace_bytes(p, 5) == 0 and U.ulysses_workspace_bytes(p, -1) == 0
    # the hybrid regroups the same rows: the same workspace
    assert U.ulysses_workspace_bytes(prob(ring=2), 1) == b
    # S = 4098 over P = 2: the delta and base-2 LSE rows (one per batch and
    # head, 4098 floats) are padded to 4100 floats so each starts on 16 bytes
    po = prob(P=2, S=4098)
    fo, bo = U.ulysses_workspace_bytes(po, 0), U.ulysses_workspace_bytes(po, 1)
    assert bo - fo >= 2 * po.B * po.n_head * 4100 * 4 + po.B * po.S * po.n_head * po.head_dim * 2


def test_ds_store_workspace(lib):
    """Phase 3 is phase 1 followed by one bf16 128 x 128 dS tile per causal
    (key tile, query tile) pair of every (batch, q-head), or every pair
    without the mask; S = 4098 has 33 tiles, the last one ragged."""
    for kw, n, pairs in ((dict(), 32, 32 * 33 // 2), (dict(causal=False), 32, 32 * 32),
                         (dict(P=2, S=4098), 33, 33 * 34 // 2)):
        p = prob(**kw)
        assert p.S == n * 128 or (p.S + 127) // 128 == n
        b, d = U.ulysses_workspace_bytes(p, 1), U.ulysses_workspace_bytes(p, 3)
        assert d == b + ((p.B * p.n_head * pairs * 128 * 128 * 2 + 255) // 256) * 256


def test_ds_store_least_workspace(lib):
    """Phase 4 is phase 1 followed by the tiles of one kv-head's q-heads on
    one rank (n_head / n_kv_head of them; with replicated kv-heads, all of a
    rank's n_head / P)."""
    for kw, per_kv in ((dict(), 32 // 8), (dict(n_kv_head=2), 32 // 8), (dict(n_kv_head=32), 1)):
        p = prob(**kw)
        tiles = 32 * 33 // 2
        b, m = U.ulysses_workspace_bytes(p, 1), U.ulysses_workspace_bytes(p, 4)
        assert m == b + ((per_kv * tiles * 128 * 128 * 2 + 255) // 256) * 256
        assert m < U.ulysses_workspace_bytes(p, 3)


def test_ds_store_refusals(lib):
    """The dS-store backward refuses a workspace smaller than phase 4, and its
    steps one smaller than phase 3, before any launch."""
    vp = ctypes.c_void_p
    ptrs = [vp((1 << 40) + i * (1 << 30)) for i in range(10)]
    p = prob()
    n3, n4 = U.ulysses_workspace_bytes(p, 3), U.ulysses_workspace_bytes(p, 4)
    assert lib.ulysses_attn_bwd_ds(ctypes.byref(p.c()), *ptrs[:9], vp(1 << 46), n4 - 256, vp(0)) == -7
    assert lib.ulysses_attn_bwd_dq_ds(ctypes.byref(p.c()), ptrs[1], ptrs[6], vp(1 << 46), n3 - 256, vp(0)) == -7
    assert lib.ulysses_attn_bwd_dkdv_ds(ctypes.byref(p.c()), *ptrs[:5], vp(1 << 46), n3 - 256, vp(0)) == -7


def test_ring_is_refused_where_no_kernel_takes_it(lib):
    """The folded forward and the two projections have no hybrid mode; they
    refuse ring > 1 on the host (fake pointers, never dereferenced)."""
    vp = ctypes.c_void_p
    p = prob(ring=2)
    nws = U.ulysses_workspace_bytes(p, 0)
    a = [vp((1 << 40) + i * (1 << 34)) for i in range(8)]
    assert lib.ulysses_attn_fwd_folded(ctypes.byref(p.c()), a[0], a[1], a[2], a[3], a[4], a[5], nws, vp(0)) == -4
    assert lib.ulysses_qkv_proj_pack(ctypes.byref(p.c()), a[0], a[1], None, a[2], a[3], a[4], a[5], nws,
                                     vp(0)) == -4
    assert lib.ulysses_out_proj_unpack(ctypes.byref(p.c()), a[0], a[1], None, a[2], a[5], nws, vp(0)) == -4


@pytest.mark.parametrize("kw", [dict(use_rope=True), dict(use_rope=False, S=800, P=8),   # RoPE; Sl = 100
                                dict(use_rope=False, ring=2), dict(use_rope=False, dtype=U.FP32)])
def test_folded_backward_refusals(lib, kw):
    """The folded backward needs RoPE off, S/P a multiple of 128, plain
    Ulysses and bf16; anything else is ERR_UNSUPPORTED before a launch (fake
    pointers, never dereferenced)."""
    vp = ctypes.c_void_p
    p = prob(**kw)
    nws = U.ulysses_workspace_bytes(p, 1)
    a = [vp((1 << 40) + i * (1 << 34)) for i in range(11)]
    assert lib.ulysses_attn_bwd_folded(ctypes.byref(p.c()), *a[:10], nws, vp(0)) == -4


def test_folded_backward_pointer_checks(lib):
    """A foldable problem with a NULL, a misaligned or an overlapping buffer is
    refused before anything is enqueued (fake addresses, never dereferenced)."""
    vp = ctypes.c_void_p
    p = prob(S=1024, use_rope=False)
    nws = U.ulysses_workspace_bytes(p, 1)
    nq = p.B * p.S * p.n_head * p.head_dim * 2
    base = 1 << 40
    bufs = [base + i * 4 * nq for i in range(10)]          # q k v o lse do dq dk dv ws, far apart

    def call(b, n=nws):
        return lib.ulysses_attn_bwd_folded(ctypes.byref(p.c()), *[vp(x) for x in b], n, vp(0))
    for i in range(10):
        b = list(bufs)
        b[i] = 0
        assert call(b) == (-7 if i == 9 else -1), i       # NULL (the workspace: ERR_WORKSPACE)
    b = list(bufs)
    b[0] += 8
    assert call(b) == -5                                      # misaligned q
    b = list(bufs)
    b[6] = bufs[0]
    assert call(b) == -6                                      # dQ written over q
    assert call(bufs, nws - 256) == -7                        # workspace too small


def test_status_strings(lib):
    for code in range(0, -9, -1):
        s = lib.ulysses_status_string(code)
        assert s and b"unknown" not in s
    assert b"unknown" in lib.ulysses_status_string(-99)


def _call_pack(lib, p, q, k, v, qh, kh, vh, ws, nws):
    vp = ctypes.c_void_p
    return lib.ulysses_pack_qkv(ctypes.byref(p.c()), vp(q), vp(k), vp(v), vp(qh), vp(kh), vp(vh),
                                vp(ws), nws, vp(0))


def test_pointer_checks_fail_before_launch(lib):
    p = prob(S=1024)
    nq = p.B * p.S * p.n_head * p.head_dim * 2
    nk = p.B * p.S * p.n_kv_head * p.head_dim * 2
    nws = U.ulysses_workspace_bytes(p, 0)
    base = 1 << 40
    q, k, v = base, base + nq, base + nq + nk
    qh, kh, vh = base + 4 * nq, base + 5 * nq, base + 6 * nq
    ws = base + 8 * nq
    assert _call_pack(lib, p, 0, k, v, qh, kh, vh, ws, nws) == -1          # NULL input
    assert _call_pack(lib, p, q + 8, k, v, qh, kh, vh, ws, nws) == -5      # misaligned
    assert _call_pack(lib, p, q, k, v, q + 16, kh, vh, ws, nws) == -6      # output overlaps input
    assert _call_pack(lib, p, q, k, v, qh, qh + 16, vh, ws, nws) == -6     # outputs overlap
    assert _call_pack(lib, p, q, k, v, qh, kh, vh, ws, nws - 1) == -7      # workspace too small
    assert _call_pack(lib, p, q, k, v, qh, kh, vh, 0, nws) == -7           # no workspace
    bad = prob(S=1024, n_kv_head=3)
    assert _call_pack(lib, bad, q, k, v, qh, kh, vh, ws, nws) == -2
    vp = ctypes.c_void_p
    # the tensor-core forward has no kernel for head_dim 32 in bf16
    p32 = prob(head_dim=32, hidden=32 * 32, S=1024)
    assert lib.ulysses_attn_fwd(ctypes.byref(p32.c()), vp(q), vp(k), vp(v), vp(qh), vp(kh), vp(ws), nws,
                                vp(0)) == -4
    # the backward has no fp32 kernel
    pf = prob(dtype=U.FP32, S=1024)
    assert lib.ulysses_attn_bwd(ctypes.byref(pf.c()), *[vp(base + i * nq) for i in range(10)], nws, vp(0)) == -4


def test_read_status_argument_checks(lib):
    vp = ctypes.c_void_p
    assert lib.ulysses_read_status_async(vp(0), vp(0x10000), vp(0)) == -1
    assert lib.ulysses_read_status_async(vp(0x10000), vp(0), vp(0)) == -1


def test_selftest_ex2_rate_argument_checks(lib):
    vp = ctypes.c_void_p
    fn = lib.ulysses_selftest_ex2_rate
    n, sms = ctypes.c_longlong(0), ctypes.c_int(0)
    assert fn(vp(0), 8, ctypes.byref(n), ctypes.byref(sms), vp(0)) == -1          # NULL buffer
    assert fn(vp(0x10000), 4, ctypes.byref(n), ctypes.byref(sms), vp(0)) == -1    # too small
    assert fn(vp(0x10000), 8, None, ctypes.byref(sms), vp(0)) == -1               # NULL count
    assert fn(vp(0x10004), 8, ctypes.byref(n), ctypes.byref(sms), vp(0)) == -5    # misaligned


def test_selftest_wait_timeout_argument_checks(lib):
    """The timeout self-test refuses bad arguments on the host, before any launch."""
    vp = ctypes.c_void_p
    fn = lib.ulysses_selftest_wait_timeout
    assert fn(vp(0), 4096, 1000000, vp(0)) == -1            # NULL workspace
    assert fn(vp(0x10000), 128, 1000000, vp(0)) == -1       # smaller than the status block
    assert fn(vp(0x10000), 4096, 0, vp(0)) == -1            # no limit
    assert fn(vp(0x10000), 4096, 3000000000, vp(0)) == -1   # above 2 s
    assert fn(vp(0x10008), 4096, 1000000, vp(0)) == -5      # misaligned


def test_noalloc_refusals_before_any_device_call(lib):
    """The workspace-free backward refuses an fp32 problem, and a problem whose
    backward scratch exceeds its fixed 32 MiB array, before it touches the GPU;
    its status reader refuses a NULL destination."""
    vp = ctypes.c_void_p
    ptrs = [vp((1 << 40) + i * (1 << 30)) for i in range(9)]
    pf = prob(dtype=U.FP32, S=1024)
    assert lib.ulysses_attn_bwd_noalloc(ctypes.byref(pf.c()), *ptrs, vp(0)) == -4
    big = prob(S=32768, n_kv_head=32)
    assert U.ulysses_workspace_bytes(big, 1) > 32 << 20
    assert lib.ulysses_attn_bwd_noalloc(ctypes.byref(big.c()), *ptrs, vp(0)) == -7
    assert lib.ulysses_noalloc_read_status(None, vp(0)) == -1
