"""ctypes binding of libulysses.so (include/ulysses.h): argument marshalling only.

Every function here has the name of the C entry point it calls and takes
torch tensors in place of raw pointers.  Nothing here computes: every step of
the path runs in the library's CUDA kernels.  If the library is missing the
first call raises; there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# ULYSSES_LIB selects another build of the library (the range-checked one).
LIB_PATH = os.environ.get("ULYSSES_LIB") or os.path.join(_HERE, "_build", "libulysses.so")
_lib = None

BF16, FP32 = 0, 1
OK = 0
STATUS_FWD_TIMEOUT, STATUS_BWD_TIMEOUT, STATUS_ROPE_TABLE, STATUS_SMEM_ALIGN, STATUS_BOUNDS = 1, 2, 4, 8, 16

EXPORTS = ("ulysses_validate", "ulysses_workspace_bytes", "ulysses_workspace_init",
           "ulysses_read_status", "ulysses_pack_qkv", "ulysses_attn_fwd", "ulysses_unpack_out",
           "ulysses_attn_bwd", "ulysses_attn_fwd_folded", "ulysses_attn_bwd_folded", "ulysses_status_string")


class UlyssesError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed with {code}: {lib().ulysses_status_string(code).decode()}")


class CProblem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("S", ctypes.c_int), ("hidden", ctypes.c_int),
                ("n_head", ctypes.c_int), ("n_kv_head", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("P", ctypes.c_int), ("causal", ctypes.c_int), ("dtype", ctypes.c_int),
                ("use_rope", ctypes.c_int), ("rope_base", ctypes.c_float),
                ("softmax_scale", ctypes.c_float), ("ring", ctypes.c_int)]


@dataclasses.dataclass(frozen=True)
class Problem:
    """Mirror of ``ulysses_problem``."""
    B: int
    S: int
    hidden: int
    n_head: int
    n_kv_head: int
    head_dim: int
    P: int
    causal: bool = True
    dtype: int = BF16
    use_rope: bool = True
    rope_base: float = 10000.0
    softmax_scale: float = 0.0
    ring: int = 1  # ring positions of the Ulysses x ring hybrid (1: plain Ulysses)

    @classmethod
    def from_workload(cls, w) -> "Problem":
        return cls(B=w.B, S=w.S, hidden=w.hidden, n_head=w.n_head, n_kv_head=w.n_kv_head,
                   head_dim=w.head_dim, P=w.P, causal=w.causal,
                   dtype=BF16 if w.dtype == "bf16" else FP32, use_rope=w.use_rope,
                   rope_base=w.rope_base, ring=getattr(w, "ring", 1))

    def c(self) -> CProblem:
        return CProblem(self.B, self.S, self.hidden, self.n_head, self.n_kv_head, self.head_dim,
                        self.P, int(self.causal), self.dtype, int(self.use_rope),
                        float(self.rope_base), float(self.softmax_scale), int(self.ring))

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == BF16 else torch.float32

    @property
    def Sl(self):
        return self.S // self.P

    @property
    def Pu(self):
        """Ranks of one ring position (the All-to-All group): P / ring."""
        return self.P // max(self.ring, 1)

    @property
    def Cs(self):
        """Tokens a head-layout buffer holds: S / ring (S for plain Ulysses)."""
        return self.S // max(self.ring, 1)

    @property
    def hp(self):
        return self.n_head // self.Pu

    @property
    def kvp(self):
        """kv-heads a rank holds in head layout: n_kv_head / Pu, or one when
        n_kv_head < Pu (each kv-head then replicated to Pu / n_kv_head ranks)."""
        return self.n_kv_head // self.Pu if self.n_kv_head >= self.Pu else 1

    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale > 0 else 1.0 / math.sqrt(self.head_dim)


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() first "
                               "(the library has no non-CUDA fallback)")
        L = ctypes.CDLL(LIB_PATH)
        vp, P, sz = ctypes.c_void_p, ctypes.POINTER(CProblem), ctypes.c_size_t
        L.ulysses_validate.argtypes = [P]
        L.ulysses_workspace_bytes.argtypes = [P, ctypes.c_int]
        L.ulysses_workspace_bytes.restype = sz
        L.ulysses_workspace_init.argtypes = [P, vp, sz, vp]
        L.ulysses_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        L.ulysses_read_status_async.argtypes = [vp, vp, vp]
        L.ulysses_pack_qkv.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_attn_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_unpack_out.argtypes = [P, vp, vp, vp]
        L.ulysses_attn_fwd_folded.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_attn_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_attn_bwd_folded.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_attn_bwd_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.ulysses_noalloc_read_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
        L.ulysses_attn_bwd_prepare.argtypes = [P, vp, vp, vp, vp, sz, vp]
        L.ulysses_qkv_proj_pack.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_out_proj_unpack.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_selftest_wait_timeout.argtypes = [vp, sz, ctypes.c_ulonglong, vp]
        L.ulysses_selftest_ex2_rate.argtypes = [vp, sz, ctypes.POINTER(ctypes.c_longlong),
                                                ctypes.POINTER(ctypes.c_int), vp]
        L.ulysses_attn_bwd_dkdv.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_attn_bwd_dq.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_attn_bwd_fused.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_attn_bwd_dkdvq.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_attn_bwd_dq_finish.argtypes = [P, vp, vp, sz, vp]
        L.ulysses_attn_bwd_ds.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_attn_bwd_dkdv_ds.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp]
        L.ulysses_attn_bwd_dq_ds.argtypes = [P, vp, vp, vp, sz, vp]
        L.ulysses_status_string.argtypes = [ctypes.c_int]
        L.ulysses_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libulysses must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, rc: int):
    if rc != OK:
        raise UlyssesError(fn, rc)


def ulysses_validate(prob: Problem) -> int:
    return lib().ulysses_validate(ctypes.byref(prob.c()))


def ulysses_workspace_bytes(prob: Problem, phase: int) -> int:
    return lib().ulysses_workspace_bytes(ctypes.byref(prob.c()), phase)


def ulysses_workspace_init(prob: Problem, ws: torch.Tensor, stream=None):
    _check("ulysses_workspace_init",
           lib().ulysses_workspace_init(ctypes.byref(prob.c()), _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream)))


def ulysses_read_status(ws: torch.Tensor, stream=None) -> int:
    out = ctypes.c_uint32(0)
    _check("ulysses_read_status", lib().ulysses_read_status(_ptr(ws), ctypes.byref(out), _stream(stream)))
    return out.value


def ulysses_read_status_async(ws: torch.Tensor, out: torch.Tensor, stream=None):
    """Enqueue a copy of the status word into `out` (a pinned uint32/int32
    host tensor of at least one element) on the stream; no synchronisation."""
    if out.device.type != "cpu" or out.element_size() != 4 or out.numel() < 1:
        raise ValueError("out must be a 4-byte host tensor")
    _check("ulysses_read_status_async", lib().ulysses_read_status_async(_ptr(ws), _ptr(out), _stream(stream)))


def ulysses_pack_qkv(prob, q_seq, k_seq, v_seq, q_head, k_head, v_head, ws, stream=None):
    _check("ulysses_pack_qkv", lib().ulysses_pack_qkv(
        ctypes.byref(prob.c()), _ptr(q_seq), _ptr(k_seq), _ptr(v_seq), _ptr(q_head), _ptr(k_head),
        _ptr(v_head), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_attn_fwd(prob, q_head, k_head, v_head, o_head, lse, ws, stream=None):
    _check("ulysses_attn_fwd", lib().ulysses_attn_fwd(
        ctypes.byref(prob.c()), _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(o_head), _ptr(lse),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_attn_fwd_folded(prob, q_seq, k_seq, v_seq, o_seq, lse, ws, stream=None):
    _check("ulysses_attn_fwd_folded", lib().ulysses_attn_fwd_folded(
        ctypes.byref(prob.c()), _ptr(q_seq), _ptr(k_seq), _ptr(v_seq), _ptr(o_seq), _ptr(lse),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_attn_bwd_folded(prob, q_seq, k_seq, v_seq, o_seq, lse, do_seq, dq_seq, dk_seq, dv_seq, ws,
                            stream=None):
    """The folded backward: q, k, v, O and dO read in sequence layout, the
    gradients written in sequence layout (RoPE off, S/P % 128 == 0)."""
    _check("ulysses_attn_bwd_folded", lib().ulysses_attn_bwd_folded(
        ctypes.byref(prob.c()), _ptr(q_seq), _ptr(k_seq), _ptr(v_seq), _ptr(o_seq), _ptr(lse), _ptr(do_seq),
        _ptr(dq_seq), _ptr(dk_seq), _ptr(dv_seq), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_unpack_out(prob, o_head, o_seq, stream=None):
    _check("ulysses_unpack_out", lib().ulysses_unpack_out(
        ctypes.byref(prob.c()), _ptr(o_head), _ptr(o_seq), _stream(stream)))


def ulysses_attn_bwd(prob, q_head, k_head, v_head, o_head, lse, do_seq, dq_seq, dk_seq, dv_seq, ws,
                     stream=None):
    _check("ulysses_attn_bwd", lib().ulysses_attn_bwd(
        ctypes.byref(prob.c()), _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(o_head), _ptr(lse),
        _ptr(do_seq), _ptr(dq_seq), _ptr(dk_seq), _ptr(dv_seq), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def ulysses_attn_bwd_prepare(prob, o_head, lse, do_seq, ws, stream=None):
    """Step 1 of the backward: dO seq -> head, delta and the rescaled LSE into ws."""
    _check("ulysses_attn_bwd_prepare", lib().ulysses_attn_bwd_prepare(
        ctypes.byref(prob.c()), _ptr(o_head), _ptr(lse), _ptr(do_seq), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_attn_bwd_dkdv(prob, q_head, k_head, v_head, dk_seq, dv_seq, ws, stream=None):
    """Step 2 of the backward: dK, dV and their head -> seq All-to-All."""
    _check("ulysses_attn_bwd_dkdv", lib().ulysses_attn_bwd_dkdv(
        ctypes.byref(prob.c()), _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(dk_seq), _ptr(dv_seq),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_attn_bwd_dq(prob, q_head, k_head, v_head, dq_seq, ws, stream=None):
    """Step 3 of the backward: dQ and its head -> seq All-to-All."""
    _check("ulysses_attn_bwd_dq", lib().ulysses_attn_bwd_dq(
        ctypes.byref(prob.c()), _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(dq_seq), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_attn_bwd_fused(prob, q_head, k_head, v_head, o_head, lse, do_seq, dq_seq, dk_seq, dv_seq, ws,
                           stream=None):
    """The backward with dQ accumulated in the dK/dV loop (phase-2 workspace)."""
    _check("ulysses_attn_bwd_fused", lib().ulysses_attn_bwd_fused(
        ctypes.byref(prob.c()), _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(o_head), _ptr(lse),
        _ptr(do_seq), _ptr(dq_seq), _ptr(dk_seq), _ptr(dv_seq), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def ulysses_attn_bwd_dkdvq(prob, q_head, k_head, v_head, dk_seq, dv_seq, ws, stream=None):
    """Fused step 2: dK, dV and the dQ shares added into the workspace accumulator."""
    _check("ulysses_attn_bwd_dkdvq", lib().ulysses_attn_bwd_dkdvq(
        ctypes.byref(prob.c()), _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(dk_seq), _ptr(dv_seq),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_attn_bwd_dq_finish(prob, dq_seq, ws, stream=None):
    """Fused step 3: dQ from the accumulator into sequence layout (accumulator re-zeroed)."""
    _check("ulysses_attn_bwd_dq_finish", lib().ulysses_attn_bwd_dq_finish(
        ctypes.byref(prob.c()), _ptr(dq_seq), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_attn_bwd_ds(prob, q_head, k_head, v_head, o_head, lse, do_seq, dq_seq, dk_seq, dv_seq, ws,
                        stream=None):
    """The backward with every tile pair's dS stored and dQ read back from it
    (phase-3 workspace)."""
    _check("ulysses_attn_bwd_ds", lib().ulysses_attn_bwd_ds(
        ctypes.byref(prob.c()), _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(o_head), _ptr(lse),
        _ptr(do_seq), _ptr(dq_seq), _ptr(dk_seq), _ptr(dv_seq), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def ulysses_attn_bwd_dkdv_ds(prob, q_head, k_head, v_head, dk_seq, dv_seq, ws, stream=None):
    """dS-store step 2: dK, dV, and every tile pair's dS into the workspace."""
    _check("ulysses_attn_bwd_dkdv_ds", lib().ulysses_attn_bwd_dkdv_ds(
        ctypes.byref(prob.c()), _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(dk_seq), _ptr(dv_seq),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_attn_bwd_dq_ds(prob, k_head, dq_seq, ws, stream=None):
    """dS-store step 3: dQ from the stored dS tiles and K, in sequence layout."""
    _check("ulysses_attn_bwd_dq_ds", lib().ulysses_attn_bwd_dq_ds(
        ctypes.byref(prob.c()), _ptr(k_head), _ptr(dq_seq), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def ulysses_qkv_proj_pack(prob, x_seq, w_qkv, b_qkv, q_head, k_head, v_head, ws, stream=None):
    """QKV projection of the sequence-sharded activations with the pack and
    RoPE fused (b_qkv may be None)."""
    _check("ulysses_qkv_proj_pack", lib().ulysses_qkv_proj_pack(
        ctypes.byref(prob.c()), _ptr(x_seq), _ptr(w_qkv), None if b_qkv is None else _ptr(b_qkv),
        _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_out_proj_unpack(prob, o_head, w_o, b_o, y_seq, ws, stream=None):
    """Output projection of the head-layout attention output with the unpack
    folded into its loads (b_o may be None)."""
    _check("ulysses_out_proj_unpack", lib().ulysses_out_proj_unpack(
        ctypes.byref(prob.c()), _ptr(o_head), _ptr(w_o), None if b_o is None else _ptr(b_o), _ptr(y_seq),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def ulysses_selftest_wait_timeout(ws, limit_ns, stream=None):
    """A bounded wait that is made to run out: sets the forward-timeout bit of
    the workspace status word after limit_ns, without any fault."""
    _check("ulysses_selftest_wait_timeout", lib().ulysses_selftest_wait_timeout(
        _ptr(ws), ws.numel() * ws.element_size(), int(limit_ns), _stream(stream)))


def ulysses_selftest_ex2_rate(stream=None) -> float:
    """Measured base-2 exponentials per SM per cycle (synchronizes)."""
    cyc = torch.zeros(1, dtype=torch.int64, device="cuda")
    n, sms = ctypes.c_longlong(0), ctypes.c_int(0)
    _check("ulysses_selftest_ex2_rate", lib().ulysses_selftest_ex2_rate(
        _ptr(cyc), 8, ctypes.byref(n), ctypes.byref(sms), _stream(stream)))
    torch.cuda.synchronize()
    return n.value / (sms.value * float(cyc.item()))


def ulysses_attn_bwd_noalloc(prob, q_head, k_head, v_head, o_head, lse, do_seq, dq_seq, dk_seq,
                             dv_seq, stream=None):
    """The backward without a workspace (for callers that cannot allocate):
    scratch comes from the library's fixed 32 MiB device array."""
    _check("ulysses_attn_bwd_noalloc", lib().ulysses_attn_bwd_noalloc(
        ctypes.byref(prob.c()), _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(o_head), _ptr(lse),
        _ptr(do_seq), _ptr(dq_seq), _ptr(dk_seq), _ptr(dv_seq), _stream(stream)))


def ulysses_noalloc_read_status(stream=None) -> int:
    """Status word of the noalloc backward's scratch array (waits for the stream)."""
    out = ctypes.c_uint32(0)
    _check("ulysses_noalloc_read_status", lib().ulysses_noalloc_read_status(ctypes.byref(out), _stream(stream)))
    return out.value


# ---------------------------------------------------------------- buffers

def seq_layout(x: torch.Tensor, P: int) -> torch.Tensor:
    """Global [B, S, ...] -> rank-major sequence shards [P, B, S/P, ...]
    (rank r holds tokens [r*S/P, (r+1)*S/P)); a layout copy, no arithmetic."""
    B, S = x.shape[0], x.shape[1]
    return x.reshape(B, P, S // P, *x.shape[2:]).transpose(0, 1).contiguous()


class Buffers:
    """Device buffers for one problem: sequence-sharded inputs, head-sharded
    intermediates, outputs and the workspace (allocated by torch, owned by
    the caller, as the C ABI requires)."""

    def __init__(self, prob: Problem, device="cuda", backward: bool = False, fused: bool = False,
                 ds: bool = False):
        dt, p = prob.torch_dtype, prob
        D = p.head_dim
        e = lambda *s, d=dt: torch.empty(*s, dtype=d, device=device)
        self.q_seq = e(p.P, p.B, p.Sl, p.n_head, D)
        self.k_seq = e(p.P, p.B, p.Sl, p.n_kv_head, D)
        self.v_seq = e(p.P, p.B, p.Sl, p.n_kv_head, D)
        self.q_head = e(p.P, p.B, p.Cs, p.hp, D)
        self.k_head = e(p.P, p.B, p.Cs, p.kvp, D)
        self.v_head = e(p.P, p.B, p.Cs, p.kvp, D)
        self.o_head = e(p.P, p.B, p.Cs, p.hp, D)
        self.lse = e(p.P, p.B, p.hp, p.Cs, d=torch.float32)
        self.o_seq = e(p.P, p.B, p.Sl, p.n_head * D)
        if backward:
            self.do_seq = e(p.P, p.B, p.Sl, p.n_head * D)
            self.dq_seq = e(p.P, p.B, p.Sl, p.n_head, D)
            self.dk_seq = e(p.P, p.B, p.Sl, p.n_kv_head, D)
            self.dv_seq = e(p.P, p.B, p.Sl, p.n_kv_head, D)
        # phase 2 (the fused backward's dQ accumulator) and phase 3 (the dS
        # store) when asked for
        phases = [1] + [2] * fused + [3] * ds if backward else [0]
        nbytes = max(ulysses_workspace_bytes(prob, ph) for ph in phases)
        if nbytes == 0:
            raise UlyssesError("ulysses_workspace_bytes", ulysses_validate(prob))
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.prob = prob

    def forward(self, stream=None):
        p = self.prob
        ulysses_pack_qkv(p, self.q_seq, self.k_seq, self.v_seq, self.q_head, self.k_head,
                         self.v_head, self.ws, stream)
        ulysses_attn_fwd(p, self.q_head, self.k_head, self.v_head, self.o_head, self.lse, self.ws,
                         stream)
        ulysses_unpack_out(p, self.o_head, self.o_seq, stream)

    def backward(self, stream=None):
        ulysses_attn_bwd(self.prob, self.q_head, self.k_head, self.v_head, self.o_head, self.lse,
                         self.do_seq, self.dq_seq, self.dk_seq, self.dv_seq, self.ws, stream)

    def backward_fused(self, stream=None):
        ulysses_attn_bwd_fused(self.prob, self.q_head, self.k_head, self.v_head, self.o_head, self.lse,
                               self.do_seq, self.dq_seq, self.dk_seq, self.dv_seq, self.ws, stream)

    def backward_ds(self, stream=None):
        ulysses_attn_bwd_ds(self.prob, self.q_head, self.k_head, self.v_head, self.o_head, self.lse,
                            self.do_seq, self.dq_seq, self.dk_seq, self.dv_seq, self.ws, stream)
