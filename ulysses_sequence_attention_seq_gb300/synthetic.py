"""Seeded synthetic inputs and the workload table.

This module only draws random numbers and names shapes; it holds none of the
method's arithmetic.  Both the CUDA path (through the tests and the bench) and
the CPU oracle read the same rounded values from the tensors it returns.

Recipe: a CPU ``torch.Generator`` seeded with ``1000 + n`` for workload ``Cn``;
draws in the order Q [B,S,n_head,D], K [B,S,n_kv,D], V [B,S,n_kv,D] and (only
when asked) dO [B,S,n_head*D], each fp32 normal(0, sigma); then one rounding
to the workload dtype (round-to-nearest-even for bf16).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    P: int
    B: int
    S: int
    hidden: int
    n_head: int
    n_kv_head: int
    head_dim: int
    dtype: str            # "bf16" | "fp32"
    causal: bool
    use_rope: bool
    rope_base: float
    sigma: float
    backward: bool
    seed: int
    ring: int = 1         # ring positions of the Ulysses x ring hybrid (1: plain Ulysses)

    @property
    def Sl(self) -> int:
        return self.S // self.P

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: the pages' sizing ("Comparing Ulysses and Megatron
# Sequence Parallelism", "Megatron Attention costs": P=8, S=32768, H=4096,
# 32 heads, D=128, bf16) is C4; the others bracket it.
WORKLOADS: Dict[str, Workload] = {
    "C1": Workload("C1", P=2, B=1, S=256, hidden=128, n_head=4, n_kv_head=4, head_dim=32,
                   dtype="fp32", causal=False, use_rope=False, rope_base=10000.0, sigma=1.0,
                   backward=False, seed=1001),
    "C2": Workload("C2", P=4, B=2, S=4096, hidden=1024, n_head=16, n_kv_head=16, head_dim=64,
                   dtype="bf16", causal=True, use_rope=True, rope_base=10000.0, sigma=1.0,
                   backward=False, seed=1002),
    "C3": Workload("C3", P=8, B=1, S=8192, hidden=4096, n_head=32, n_kv_head=8, head_dim=128,
                   dtype="bf16", causal=True, use_rope=True, rope_base=10000.0, sigma=1.0,
                   backward=True, seed=1003),
    "C4": Workload("C4", P=8, B=1, S=32768, hidden=4096, n_head=32, n_kv_head=32, head_dim=128,
                   dtype="bf16", causal=True, use_rope=True, rope_base=10000.0, sigma=0.5,
                   backward=True, seed=1004),
    "C5": Workload("C5", P=32, B=1, S=65536, hidden=4096, n_head=32, n_kv_head=32, head_dim=128,
                   dtype="bf16", causal=True, use_rope=True, rope_base=10000.0, sigma=1.0,
                   backward=False, seed=1005),
}

# Beyond the five: the pages' sizing with fewer kv-heads than ranks (4 kv-heads
# over P=8, so each kv-head is replicated to 2 ranks), for the KV-head
# replication path.
EXTRA_WORKLOADS: Dict[str, Workload] = {
    "C4-kv4": WORKLOADS["C4"].with_(name="C4-kv4", n_kv_head=4, seed=1006),
    # The pages' example of the head-count bound ("Sequence Parallelism II",
    # §4: 32 heads cannot be spread over 256 ranks by heads alone), run as the
    # Ulysses x ring hybrid: 8 ring positions of 32 ranks on C4's model.
    "C4-ring8": WORKLOADS["C4"].with_(name="C4-ring8", P=256, ring=8, seed=1007),
}

# The permute-only sweep at the head-count bound (P=32, one head per rank).
SWEEP_S = (4096, 8192, 16384, 32768, 65536, 131072)


def torch_dtype(w: Workload) -> torch.dtype:
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def make_inputs(w: Workload, with_grad: Optional[bool] = None, seed: Optional[int] = None):
    """Global tensors (CPU, workload dtype): q, k, v and, if requested, do."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    dt = torch_dtype(w)
    out = {}
    shapes = [("q", (w.B, w.S, w.n_head, w.head_dim)),
              ("k", (w.B, w.S, w.n_kv_head, w.head_dim)),
              ("v", (w.B, w.S, w.n_kv_head, w.head_dim))]
    if w.backward if with_grad is None else with_grad:
        shapes.append(("do", (w.B, w.S, w.n_head * w.head_dim)))
    for name, shape in shapes:
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if w.sigma != 1.0:
            x.mul_(w.sigma)
        out[name] = x.to(dt)
    return out
