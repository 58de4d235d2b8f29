"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare it with the fp64 oracle on the same seeded inputs.

Tolerances (bf16): max-abs 2e-2 and rel-L2 1e-2 for attention outputs and
gradients (the stated bar); fp32 workload: max-abs 1e-4.  The max-abs bound is
read in units of max(1, |reference|): bf16 keeps 8 significant bits, so at
|x| >= 8 rounding the exact value to bf16 alone can move it by 2^-5 > 2e-2,
and no bf16 result could meet an absolute 2e-2 there.  For |x| <= 1 the bound
is exactly the stated 2e-2; rel-L2 is scale-free and applies unchanged.  LSE: max-abs 5e-2
for bf16, derived from the bf16 rounding of the rotated q and k the kernel
reads (|d s| <= 2 * 2^-9 * scale * sum_e |q_e k_e|, about 3e-2 at D = 128 for
unit-variance inputs), 1e-4 for fp32.  The permutation without RoPE must be
bit-exact; with RoPE each element must be within one bf16 ulp of the fp64
rotation plus the float-arithmetic bound 2^-20 * (|x| + |y|) of the pair.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300.synthetic import Workload, make_inputs

BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 1e-2
FP32_MAX_ABS = 1e-4
LSE_BF16_MAX_ABS = 5e-2


def oracle_problem(w: Workload) -> oracle.Problem:
    return oracle.Problem(B=w.B, S=w.S, n_head=w.n_head, n_kv_head=w.n_kv_head, D=w.head_dim, P=w.P,
                          causal=w.causal, use_rope=w.use_rope, rope_base=float(np.float32(w.rope_base)),
                          ring=w.ring)


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def errors(got: np.ndarray, want: np.ndarray, mask=None):
    """(max-abs, max-abs in units of max(1, |want|), rel-L2)."""
    if mask is not None:
        got, want = got[mask], want[mask]
    diff = np.abs(got - want)
    max_abs = float(diff.max()) if diff.size else 0.0
    scaled = float((diff / np.maximum(1.0, np.abs(want))).max()) if diff.size else 0.0
    rel_l2 = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))
    return max_abs, scaled, rel_l2


def assert_close(got, want, w: Workload, what: str, mask=None):
    assert np.all(np.isfinite(got[mask] if mask is not None else got)), f"{what}: non-finite output"
    max_abs, scaled, rel = errors(got, want, mask)
    if w.dtype == "fp32":
        assert max_abs <= FP32_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {FP32_MAX_ABS}"
    else:
        assert scaled <= BF16_MAX_ABS, \
            f"{what}: max-abs {max_abs:.3e} ({scaled:.3e} in units of max(1,|ref|)) > {BF16_MAX_ABS}"
        assert rel <= BF16_REL_L2, f"{what}: rel-L2 {rel:.3e} > {BF16_REL_L2}"
    return max_abs, scaled, rel


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    _, e = np.frexp(np.abs(x))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


class GpuRun:
    """Inputs on the device in the sequence-sharded layout, workspace prepared,
    forward (and optionally backward) run through the C ABI."""

    def __init__(self, w: Workload, backward: bool = False, inputs=None):
        self.w = w
        self.prob = U.Problem.from_workload(w)
        self.inputs = inputs if inputs is not None else make_inputs(w, with_grad=backward)
        self.buf = U.Buffers(self.prob, backward=backward)
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


def oracle_inputs(inputs):
    return {k: to64(v) for k, v in inputs.items()}
