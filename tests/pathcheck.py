"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare it with the fp64 oracle on the same seeded inputs.

Tolerances.  bf16 attention outputs and gradients: every element within
2e-2 + ulp_bf16(ref)/2 of the fp64 reference, and rel-L2 within 1e-2.  The
stated bar is max-abs 2e-2 / rel-L2 1e-2; the half ulp added to it is the
output format's own rounding floor: the kernels write bf16, and rounding even
the exact value to bf16 moves it by up to half a bf16 spacing (1/256 of its
binade), which alone exceeds 2e-2 once |ref| >= 8.  For |ref| < 2 the extra
term is at most 2^-8 = 0.0039.  fp32 workload: max-abs 1e-4.  LSE: max-abs
5e-2 for bf16, derived from the bf16 rounding of the rotated q and k the
kernel reads (|d s| <= 2 * 2^-9 * scale * sum_e |q_e k_e|, about 3e-2 at
D = 128 for unit-variance inputs), 1e-4 for fp32.  The permutation without
RoPE must be bit-exact; with RoPE each element must be within one bf16 ulp of
the fp64 rotation plus the float-arithmetic bound 2^-20 * (|x| + |y|) of the
pair.

Every comparison is recorded (worst absolute error, worst error as a fraction
of its per-element bound, rel-L2); tests/conftest.py prints the tightest
margins at the end of the run and writes them all as JSON to the file named by
the environment variable ULYSSES_PARITY_LOG, when it is set.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300.synthetic import Workload, make_inputs

BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 1e-2
FP32_MAX_ABS = 1e-4
LSE_BF16_MAX_ABS = 5e-2

# One entry per comparison made in this process (see tests/conftest.py).
RECORDS: list = []


def _record(what, kind, max_abs, worst_frac, rel_l2, n):
    RECORDS.append(dict(test=os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], what=what, kind=kind,
                        max_abs=max_abs, worst_frac_of_bound=worst_frac, rel_l2=rel_l2, n=int(n)))


def oracle_problem(w: Workload) -> oracle.Problem:
    return oracle.Problem(B=w.B, S=w.S, n_head=w.n_head, n_kv_head=w.n_kv_head, D=w.head_dim, P=w.P,
                          causal=w.causal, use_rope=w.use_rope, rope_base=float(np.float32(w.rope_base)),
                          ring=w.ring)


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    _, e = np.frexp(np.abs(x))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def bf16_bound(want: np.ndarray) -> np.ndarray:
    """Per-element max-abs bound of a bf16 result: 2e-2 plus half a bf16 ulp of
    the reference (the rounding of the output format itself)."""
    return BF16_MAX_ABS + 0.5 * ulp_bf16(want)


def errors(got: np.ndarray, want: np.ndarray, mask=None, bf16: bool = True):
    """(max-abs, worst |got - want| / per-element bound, rel-L2)."""
    if mask is not None:
        got, want = got[mask], want[mask]
    diff = np.abs(got - want)
    max_abs = float(diff.max()) if diff.size else 0.0
    bound = bf16_bound(want) if bf16 else FP32_MAX_ABS
    frac = float((diff / bound).max()) if diff.size else 0.0
    rel_l2 = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))
    return max_abs, frac, rel_l2


def assert_close(got, want, w: Workload, what: str, mask=None):
    assert np.all(np.isfinite(got[mask] if mask is not None else got)), f"{what}: non-finite output"
    bf16 = w.dtype != "fp32"
    max_abs, frac, rel = errors(got, want, mask, bf16=bf16)
    n = (got[mask] if mask is not None else got).size
    _record(what, "bf16" if bf16 else "fp32", max_abs, frac, rel, n)
    if not bf16:
        assert max_abs <= FP32_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {FP32_MAX_ABS}"
    else:
        assert frac <= 1.0, \
            f"{what}: max-abs {max_abs:.3e}; worst element at {frac:.3f} of its bound 2e-2 + ulp_bf16(ref)/2"
        assert rel <= BF16_REL_L2, f"{what}: rel-L2 {rel:.3e} > {BF16_REL_L2}"
    return max_abs, frac, rel


def assert_lse_close(got, want, w: Workload, what: str = "lse"):
    """LSE rows against the oracle's: max-abs 5e-2 (bf16) or 1e-4 (fp32)."""
    tol = FP32_MAX_ABS if w.dtype == "fp32" else LSE_BF16_MAX_ABS
    diff = np.abs(np.asarray(got) - np.asarray(want))
    max_abs = float(diff.max()) if diff.size else 0.0
    _record(what, "lse-" + ("fp32" if w.dtype == "fp32" else "bf16"), max_abs, max_abs / tol, None, diff.size)
    assert max_abs <= tol, f"{what}: max-abs {max_abs:.3e} > {tol}"
    return max_abs


class GpuRun:
    """Inputs on the device in the sequence-sharded layout, workspace prepared,
    forward (and optionally backward) run through the C ABI."""

    def __init__(self, w: Workload, backward: bool = False, inputs=None, fused: bool = False, ds: bool = False):
        self.w = w
        self.prob = U.Problem.from_workload(w)
        self.inputs = inputs if inputs is not None else make_inputs(w, with_grad=backward)
        self.buf = U.Buffers(self.prob, backward=backward, fused=fused, ds=ds)
        P = w.P
        self.buf.q_seq.copy_(U.seq_layout(self.inputs["q"], P))
        self.buf.k_seq.copy_(U.seq_layout(self.inputs["k"], P))
        self.buf.v_seq.copy_(U.seq_layout(self.inputs["v"], P))
        if backward:
            self.buf.do_seq.copy_(U.seq_layout(self.inputs["do"], P))
        U.ulysses_workspace_init(self.prob, self.buf.ws)

    def forward(self):
        self.buf.forward()
        torch.cuda.synchronize()
        assert U.ulysses_read_status(self.buf.ws) == 0

    def backward(self):
        self.buf.backward()
        torch.cuda.synchronize()
        assert U.ulysses_read_status(self.buf.ws) == 0

    def backward_fused(self):
        self.buf.backward_fused()
        torch.cuda.synchronize()
        assert U.ulysses_read_status(self.buf.ws) == 0

    def backward_ds(self):
        self.buf.backward_ds()
        torch.cuda.synchronize()
        assert U.ulysses_read_status(self.buf.ws) == 0


def oracle_inputs(inputs):
    return {k: to64(v) for k, v in inputs.items()}
