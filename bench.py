"""Benchmark of the Ulysses attention path on GB300 (one JSON line on stdout).

A step is one pass of the whole path over one batch of seeded synthetic input
in HBM: seq->head pack with RoPE, tensor-core attention forward, head->seq
unpack and, for workloads with a backward, the backward with its reverse
All-to-Alls.  Default workload: the pages' sizing (P=8 virtual ranks, B=1,
S=32768, 32 heads, D=128, bf16, causal, RoPE).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload C4] [--impl ulysses|reference]

N > 1 runs N independent replicas (one per GPU, launched by torchrun): the
path has no data exchange between GPUs once its P virtual ranks share one
HBM, so the job is weak-scaled and the only cross-GPU traffic is the timing
reduction.  `--impl reference` times the fp64 CPU oracle on the host cores on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from ulysses_sequence_attention_seq_gb300.synthetic import EXTRA_WORKLOADS, WORKLOADS, make_inputs  # noqa: E402

METRIC = "tokens/s + attn TFLOP/s (S=32K, 32 heads, P=8 virtual); seq↔head permute GB/s"


# ------------------------------------------------------------------ helpers

# DRAM bytes (read + write) per launch of a kernel on a workload, from ncu
# captures of this build: one kernel per capture, the mean of its two launches
# in the bench's timed steps (`-k regex:<kernel> -s 3 -c 2` on `bench.py
# --workload <w> --steps 2 --warmup 3 --no-cpu-baseline`; profiles/ gives the
# commands and tables); a kernel changed since its capture has no entry.
TRAFFIC = {
    ("attn_fwd", "C4"): 1062845312,
    ("bwd_dkdv", "C4"): 1627353472,
    ("bwd_dq", "C4"): 1359185920,
    ("bwd_dkdv_ds", "C4"): 36864050432,
    ("bwd_dq_ds", "C4"): 35416766208,
    ("attn_fwd", "C4-ring8"): 1077393792,
    ("bwd_dkdv", "C4-ring8"): 1636954368,
    ("bwd_dq", "C4-ring8"): 1360104576,
    ("bwd_dkdv_ds", "C4-ring8"): 36822935168,
    ("bwd_dq_ds", "C4-ring8"): 35417668224,
    ("attn_fwd", "C4-kv4"): 640970624,
    ("bwd_dkdv_ds", "C4-kv4"): 40575356032,
    ("bwd_dq_ds", "C4-kv4"): 35152657664,
}


SM_MAX_MHZ_FALLBACK = 2070.0  # GB300's maximum SM clock, when nvidia-smi gave none


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# The backward's tensor-core kernels: (kernel, algorithmic FLOPs, executed
# FLOPs) as functions of the forward's algorithmic FLOPs.  The method's
# products are the forward's S and PV and the backward's dV, dP, dQ, dK, each
# half a forward; the two-kernel backward's kernels both recompute S and the
# dQ kernel dP as well; the dS-store dK/dV kernel is the dK/dV kernel that
# also writes dS (its dQ step is a plain sum of products over stored tiles,
# bound by HBM); the fused kernel adds each pair's dQ share.
BWD_TC = {
    "bwd_dkdv": lambda fl: ("dkdv_kernel", 1.5 * fl, 2.0 * fl),
    "bwd_dq": lambda fl: ("dq_kernel", 0.5 * fl, 1.5 * fl),
    "bwd_dkdv_ds": lambda fl: ("dkdv_kernel", 1.5 * fl, 2.0 * fl),
    "bwd_dkdvq": lambda fl: ("dkdvq_kernel", 2.0 * fl, 2.5 * fl),
}
BWD_NOTES = {
    "two_kernel": "ulysses_attn_bwd: dK/dV kernel, then the dQ kernel recomputing S and dP; 7 products per tile "
                  "pair; bit-reproducible",
    "ds_store": "ulysses_attn_bwd_ds: the dK/dV kernel also stores every tile pair's bf16 dS (32 KB a pair), dQ "
                "is summed from the stored tiles; 5 products per tile pair; bit-reproducible",
    "fused": "ulysses_attn_bwd_fused: dQ shares reduce-added into a float accumulator inside the dK/dV loop; 5 "
             "products per tile pair; dQ reproducible to float rounding",
}


def ds_tiles(w):
    """(key tile, query tile) pairs of one head the dS store holds."""
    n = (w.S + 127) // 128
    return n * (n + 1) // 2 if w.causal else n * n


def dq_ds_bytes(w, es):
    """Bytes the dQ-from-dS step moves at the least: every stored 128 x 128
    bf16 dS tile, K (the kv-heads over the sequence) and dQ, once each."""
    return (w.B * w.n_head * ds_tiles(w) * 128 * 128 * 2 + w.B * w.S * w.n_kv_head * w.head_dim * es
            + w.B * w.S * w.n_head * w.head_dim * es)


def attn_fwd_flops(w):
    """Algorithmic FLOPs of the attention forward: two matmuls (QK^T and PV),
    2*D flops per (query, key) pair each; causal counts S(S+1)/2 pairs."""
    pairs = w.S * (w.S + 1) / 2 if w.causal else float(w.S) * w.S
    return 4.0 * w.B * w.n_head * w.head_dim * pairs


def permute_bytes(w, es):
    """Bytes read + written by the seq->head pack of Q, K, V: each tensor read
    once and written once, K and V written once per replica when there are
    fewer kv-heads than ranks in an All-to-All group (each kv-head then goes to
    Pu / n_kv_head ranks; Pu = P / ring is the group's size)."""
    pu = w.P // getattr(w, "ring", 1)
    kv_written = w.n_kv_head if w.n_kv_head >= pu else pu
    return float(w.B * w.S * w.head_dim * es) * (2 * w.n_head + 2 * w.n_kv_head + 2 * kv_written)


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ our CUDA path

def run_ulysses(args, w, rank, world):
    from ulysses_sequence_attention_seq_gb300 import binding as U

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    prob = U.Problem.from_workload(w)
    backward = w.backward and not args.fwd_only
    ins = make_inputs(w, with_grad=backward)
    # a workspace for every backward mode: the fused one's dQ accumulator
    # (phase 2) and the dS-store one's tiles (phase 3); the modes not on the
    # headline are timed beside it
    buf = U.Buffers(prob, device=dev, backward=backward, fused=backward, ds=backward)
    host = {"q": U.seq_layout(ins["q"], w.P).pin_memory(), "k": U.seq_layout(ins["k"], w.P).pin_memory(),
            "v": U.seq_layout(ins["v"], w.P).pin_memory()}
    if backward:
        host["do"] = U.seq_layout(ins["do"], w.P).pin_memory()
    buf.q_seq.copy_(host["q"])
    buf.k_seq.copy_(host["k"])
    buf.v_seq.copy_(host["v"])
    if backward:
        buf.do_seq.copy_(host["do"])
    stream = torch.cuda.current_stream()
    U.ulysses_workspace_init(prob, buf.ws)
    torch.cuda.synchronize()

    # Each backward mode as the entry points that make up its composed call
    # (ulysses_attn_bwd, ulysses_attn_bwd_ds, ulysses_attn_bwd_fused), so
    # that each kernel gets its own events.
    b = buf
    bwd_steps = {
        "two_kernel": (
            ("bwd_prepare", lambda: U.ulysses_attn_bwd_prepare(prob, b.o_head, b.lse, b.do_seq, b.ws)),
            ("bwd_dkdv", lambda: U.ulysses_attn_bwd_dkdv(prob, b.q_head, b.k_head, b.v_head, b.dk_seq, b.dv_seq,
                                                         b.ws)),
            ("bwd_dq", lambda: U.ulysses_attn_bwd_dq(prob, b.q_head, b.k_head, b.v_head, b.dq_seq, b.ws))),
        "ds_store": (
            ("bwd_prepare", lambda: U.ulysses_attn_bwd_prepare(prob, b.o_head, b.lse, b.do_seq, b.ws)),
            ("bwd_dkdv_ds", lambda: U.ulysses_attn_bwd_dkdv_ds(prob, b.q_head, b.k_head, b.v_head, b.dk_seq,
                                                               b.dv_seq, b.ws)),
            ("bwd_dq_ds", lambda: U.ulysses_attn_bwd_dq_ds(prob, b.k_head, b.dq_seq, b.ws))),
        "fused": (
            ("bwd_prepare", lambda: U.ulysses_attn_bwd_prepare(prob, b.o_head, b.lse, b.do_seq, b.ws)),
            ("bwd_dkdvq", lambda: U.ulysses_attn_bwd_dkdvq(prob, b.q_head, b.k_head, b.v_head, b.dk_seq, b.dv_seq,
                                                           b.ws)),
            ("bwd_dq_finish", lambda: U.ulysses_attn_bwd_dq_finish(prob, b.dq_seq, b.ws))),
    }
    mode = args.bwd_mode if backward else None
    names = ["pack_qkv", "attn_fwd", "unpack_out"] + ([n for n, _ in bwd_steps[mode]] if backward else [])
    # pack, forward, unpack; prepare, dK/dV (+ the replica sum when kv-heads are
    # replicated), dQ
    launches_per_step = 3 + ((4 if w.n_kv_head < w.P // w.ring else 3) if backward else 0)

    def step(evs=None):
        """One pass of the whole path: pack, attention, unpack, and the
        backward of the headline mode."""
        def mark(i):
            if evs is not None:
                evs[i].record(stream)
        mark(0)
        U.ulysses_pack_qkv(prob, buf.q_seq, buf.k_seq, buf.v_seq, buf.q_head, buf.k_head, buf.v_head, buf.ws)
        mark(1)
        U.ulysses_attn_fwd(prob, buf.q_head, buf.k_head, buf.v_head, buf.o_head, buf.lse, buf.ws)
        mark(2)
        U.ulysses_unpack_out(prob, buf.o_head, buf.o_seq)
        mark(3)
        if backward:
            for i, (_, fn) in enumerate(bwd_steps[mode]):
                fn()
                mark(4 + i)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if U.ulysses_read_status(buf.ws) != 0:
        raise RuntimeError("device status word set during warm-up")

    # ---- device-resident timing: K steps, per-kernel events on the stream
    nev = len(names) + 1
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    total_ms = t0.elapsed_time(t1)
    per = {n: [evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps)] for i, n in enumerate(names)}

    # ---- the other backward modes: the same K steps' backward through each
    # one's entry points, each kernel timed
    alt_per = {}
    for m in (sorted(bwd_steps) if backward else []):
        if m == mode:
            continue

        def alt_bwd(ev=None, m=m):
            if ev is not None:
                ev[0].record(stream)
            for i, (_, fn) in enumerate(bwd_steps[m]):
                fn()
                if ev is not None:
                    ev[i + 1].record(stream)

        for _ in range(2):
            alt_bwd()
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        torch.cuda.synchronize()
        for k in range(args.steps):
            alt_bwd(fev[k])
        torch.cuda.synchronize()
        alt_per[m] = {n: [fev[k][i].elapsed_time(fev[k][i + 1]) for k in range(args.steps)]
                      for i, (n, _) in enumerate(bwd_steps[m])}
        if U.ulysses_read_status(buf.ws) != 0:
            raise RuntimeError(f"device status word set during the {m} backward steps")

    # ---- end to end through the public API with host buffers: every step
    # uploads its inputs from pinned host memory and downloads its results
    # (O, and dQ, dK, dV with a backward); the streamed path overlaps step k's
    # compute with step k+1's upload and step k-1's download.
    from ulysses_sequence_attention_seq_gb300.streamed import StreamedPath
    sp = StreamedPath(prob, backward=backward, device=dev, bwd_mode=mode or "two_kernel")
    host_in = {"q_seq": host["q"], "k_seq": host["k"], "v_seq": host["v"]}
    if backward:
        host_in["do_seq"] = host["do"]
    host_out = {n: torch.empty(getattr(sp.sets[0], n).shape, dtype=getattr(sp.sets[0], n).dtype, pin_memory=True)
                for n in sp.out_names()}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    sp.run(host_in, host_out, 2)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    sp.run(host_in, host_out, args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if sp.status() != 0:
        raise RuntimeError("device status word set during the end-to-end steps")
    del sp
    # the host link's copy rate on this machine (the q input, up and then down,
    # each copy alone): what bounds the end-to-end leg's first upload and last
    # download, the copies the compute cannot hide
    link = {}
    up = torch.empty_like(host["q"], device=dev)
    down = torch.empty(host["q"].shape, dtype=host["q"].dtype, pin_memory=True)
    for name, fn in (("h2d_gbs", lambda: up.copy_(host["q"], non_blocking=True)),
                     ("d2h_gbs", lambda: down.copy_(up, non_blocking=True))):
        fn()
        torch.cuda.synchronize()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(3):
            fn()
        z.record(stream)
        torch.cuda.synchronize()
        link[name] = 3 * up.numel() * up.element_size() / (a.elapsed_time(z) * 1e-3) / 1e9
    # and both directions at once, as the end-to-end leg runs them (an upload
    # and a download on two streams): each direction's rate while the other runs
    src_dev = up.clone()
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    ev = {n: torch.cuda.Event(enable_timing=True) for n in ("u0", "u1", "d0", "d1")}
    with torch.cuda.stream(s_up):
        ev["u0"].record(s_up)
        for _ in range(3):
            up.copy_(host["q"], non_blocking=True)
        ev["u1"].record(s_up)
    with torch.cuda.stream(s_down):
        ev["d0"].record(s_down)
        for _ in range(3):
            down.copy_(src_dev, non_blocking=True)
        ev["d1"].record(s_down)
    torch.cuda.synchronize()
    nb = 3 * up.numel() * up.element_size()
    link["h2d_gbs_both_ways"] = nb / (ev["u0"].elapsed_time(ev["u1"]) * 1e-3) / 1e9
    link["d2h_gbs_both_ways"] = nb / (ev["d0"].elapsed_time(ev["d1"]) * 1e-3) / 1e9
    del up, down, src_dev
    # ---- folded forward (pack + attention + unpack in one kernel) vs the three
    # calls, same shapes with RoPE off (the folded path needs pre-rotated q, k)
    folded = None
    if w.dtype == "bf16" and w.Sl % 128 == 0 and w.ring == 1:  # the folded mode has no hybrid form
        import dataclasses
        pf = dataclasses.replace(prob, use_rope=False)

        def three():
            U.ulysses_pack_qkv(pf, buf.q_seq, buf.k_seq, buf.v_seq, buf.q_head, buf.k_head, buf.v_head, buf.ws)
            U.ulysses_attn_fwd(pf, buf.q_head, buf.k_head, buf.v_head, buf.o_head, buf.lse, buf.ws)
            U.ulysses_unpack_out(pf, buf.o_head, buf.o_seq)

        def fold():
            U.ulysses_attn_fwd_folded(pf, buf.q_seq, buf.k_seq, buf.v_seq, buf.o_seq, buf.lse, buf.ws)

        # the backward on the packed buffers (dO pack + delta, dK/dV, dQ) vs the
        # folded backward (delta from O and dO in place, the same two kernels
        # reading the sequence-sharded buffers)
        def bwd_packed():
            U.ulysses_attn_bwd(pf, buf.q_head, buf.k_head, buf.v_head, buf.o_head, buf.lse, buf.do_seq,
                               buf.dq_seq, buf.dk_seq, buf.dv_seq, buf.ws)

        def bwd_fold():
            U.ulysses_attn_bwd_folded(pf, buf.q_seq, buf.k_seq, buf.v_seq, buf.o_seq, buf.lse, buf.do_seq,
                                      buf.dq_seq, buf.dk_seq, buf.dv_seq, buf.ws)

        def timed(fn):
            for _ in range(2):
                fn()
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.steps):
                fn()
            b2.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b2) / args.steps

        label = f"{w.name} shapes, RoPE off (q and k rotated by their producer)"
        folded = {"fwd": dict(unfolded_ms=timed(three), ms=timed(fold), workload=label)}
        if backward:
            folded["bwd"] = dict(unfolded_ms=timed(bwd_packed), ms=timed(bwd_fold), workload=label)
    status = U.ulysses_read_status(buf.ws)
    # the MUFU unit's exponential throughput on this GPU (the softmax's secondary bound)
    ex2_rate = U.ulysses_selftest_ex2_rate()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return dict(total_ms=total_ms, per=per, alt_per=alt_per, bwd_mode=mode, clocks=clk, e2e_ms=e2e_ms, h2d=h2d,
                d2h=d2h, link=link, launches=launches_per_step * args.steps, status=status, backward=backward,
                folded=folded, ex2_rate=ex2_rate, sms=sms)


def line_config(w, passes, l2, parallelism):
    """The `config` of a JSON line: the same keys on the GPU arm and the reference arm."""
    return {"workload": w.name, "P": w.P, "ring": w.ring, "B": w.B, "S": w.S, "n_head": w.n_head,
            "n_kv_head": w.n_kv_head, "head_dim": w.head_dim, "causal": w.causal, "rope": w.use_rope,
            "passes": passes, "l2": l2, "parallelism": parallelism}


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world):
    """The slowest rank's time: every replica processed its units within it."""
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, seconds_max, world):
    """Whole-job rate: the units all replicas processed over the max-over-ranks time."""
    return units_per_rank * world / seconds_max


# ---------------------------------------------------------- the CPU oracle

class OracleBench:
    """Times the fp64 oracle, as it stands, on a bounded sample of a workload.

    One sampled step runs the oracle's steps in the path's order.  Forward:
    split by sequence, RoPE and the three loop All-to-Alls of Q, K, V in full;
    attention for `n_rows` random query rows of every head; the inverse
    All-to-All in full.  Backward (workloads with one, plain Ulysses): the
    All-to-All of dO in full; the attention backward of one (rank, batch,
    kv-head) group, whose statistics phase (lse and delta of every row of the
    group) runs in full and whose dQ and dK/dV phases run for `n_bwd_rows`
    random query rows and key rows; the inverse All-to-Alls of dQ, dK, dV and
    the inverse RoPE in full.  The full step's time is estimated as the layout
    time + each attention phase's time x (query-key pairs of the full workload
    / pairs sampled), the backward's groups being alike."""

    def __init__(self, w, nthreads=None, backward=None):
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        import oracle
        from oracle import ring as oracle_ring
        self.oracle = oracle
        self.ring = oracle_ring
        self.w = w
        self.nthreads = nthreads or (os.cpu_count() or 1)
        # the ring hybrid's oracle backward has no row sampling: forward only there
        self.backward = (w.backward if backward is None else backward) and w.ring == 1
        ins = make_inputs(w, with_grad=self.backward)
        self.x = {k: v.to(torch.float64).numpy() for k, v in ins.items()}
        del ins
        self.op = oracle.Problem(B=w.B, S=w.S, n_head=w.n_head, n_kv_head=w.n_kv_head, D=w.head_dim,
                                 P=w.P, causal=w.causal, use_rope=w.use_rope,
                                 rope_base=float(np.float32(w.rope_base)), ring=w.ring)
        self.rng = np.random.default_rng(0)

    @property
    def passes(self):
        return "fwd+bwd" if self.backward else "fwd"

    def _full_pairs(self):
        w = self.w
        return w.S * (w.S + 1) / 2 if w.causal else float(w.S) * w.S

    def step(self, n_rows, n_bwd_rows=None):
        """One sampled step.  Returns (estimated full-step seconds, query rows
        sampled in the forward, forward pairs sampled, wall seconds)."""
        o, w, x = self.oracle, self.w, self.x
        t0 = time.perf_counter()
        q, k, v = (o.shard_sequence(x[n], w.P) for n in ("q", "k", "v"))
        if w.use_rope:
            q, k = o.rope_seq(q, self.op.rope_base), o.rope_seq(k, self.op.rope_base)
        rows = sorted(set(int(r) for r in self.rng.integers(0, w.S, n_rows)))
        if w.ring > 1:  # the Ulysses x ring hybrid: All-to-All per ring position, ring attention
            rg = self.ring
            qh, kh, vh = (rg.a2a_seq_to_head(t, hh, w.ring)[0]
                          for t, hh in ((q, w.n_head), (k, w.n_kv_head), (v, w.n_kv_head)))
            t1 = time.perf_counter()
            oh, _ = rg.ring_attention_fwd(self.op, qh, kh, vh, rows=rows)
            t2 = time.perf_counter()
            rg.a2a_head_to_seq(oh, w.n_head, w.ring)
        else:
            qh, _, _ = o.a2a_seq_to_head(q, w.n_head)
            kv_a2a = o.a2a_seq_to_head_replicated if self.op.kv_replicas > 1 else o.a2a_seq_to_head
            kh, _, _ = kv_a2a(k, w.n_kv_head)
            vh, _, _ = kv_a2a(v, w.n_kv_head)
            t1 = time.perf_counter()
            oh, _ = o.attention_fwd(self.op, qh, kh, vh, rows=rows, nthreads=self.nthreads)
            t2 = time.perf_counter()
            o.a2a_head_to_seq(oh, w.n_head)
        t3 = time.perf_counter()
        pairs = sum((r + 1) if w.causal else w.S for r in rows)
        full = self._full_pairs()
        t_full = (t1 - t0) + (t3 - t2) + (t2 - t1) * full / pairs
        self.last = {"fwd_s": t_full}
        if self.backward:
            t_bwd = self._backward(qh, kh, vh, n_bwd_rows or self.bwd_rows_for(n_rows))
            t_full += t_bwd
            self.last["bwd_s"] = t_bwd
        return t_full, len(rows), pairs, time.perf_counter() - t0

    def bwd_rows_for(self, n_rows):
        """Backward rows giving the dQ and dK/dV phases about as much work as the
        forward's sampled attention: that covers all n_head heads, the backward
        sample one group of G heads at about 3.5 forward products per pair."""
        w = self.w
        G = (w.n_head // w.P) // self.op.kvp
        return int(min(w.S, max(16, n_rows * (w.n_head // G) // 4)))

    def _backward(self, qh, kh, vh, n_bwd_rows):
        o, w, x, op = self.oracle, self.w, self.x, self.op
        D, hp, kvp = w.head_dim, w.n_head // w.P, op.kvp
        G = hp // kvp
        tb0 = time.perf_counter()
        do_seq = o.shard_sequence(x["do"].reshape(w.B, w.S, w.n_head, D), w.P)
        doh, _, _ = o.a2a_seq_to_head(do_seq, w.n_head)
        tb1 = time.perf_counter()
        q_rows = sorted(set(int(r) for r in self.rng.integers(0, w.S, n_bwd_rows)))
        kv_rows = sorted(set(int(r) for r in self.rng.integers(0, w.S, n_bwd_rows)))
        ph = []
        dqh, dkh, dvh = o.attention_bwd(op, qh, kh, vh, doh, groups=[(0, 0, 0)], q_rows=q_rows, kv_rows=kv_rows,
                                        nthreads=self.nthreads, phase_seconds=ph)
        tb2 = time.perf_counter()
        dq_seq, _, _ = o.a2a_head_to_seq(dqh, w.n_head, fill=np.nan)
        if op.kv_replicas > 1:
            dk_seq, _, _ = o.reduce_head_to_seq_replicated(dkh, w.n_kv_head)
            o.reduce_head_to_seq_replicated(dvh, w.n_kv_head)
        else:
            dk_seq, _, _ = o.a2a_head_to_seq(dkh, w.n_kv_head, fill=np.nan)
            o.a2a_head_to_seq(dvh, w.n_kv_head, fill=np.nan)
        if w.use_rope:
            o.rope_seq(dq_seq, op.rope_base, -1)
            o.rope_seq(dk_seq, op.rope_base, -1)
        tb3 = time.perf_counter()
        t_stat, t_dq, t_dkdv = ph[0]
        full = G * self._full_pairs()
        pairs_dq = G * sum((i + 1) if w.causal else w.S for i in q_rows)
        pairs_dkdv = G * sum((w.S - kk) if w.causal else w.S for kk in kv_rows)
        t_group = t_stat + t_dq * full / pairs_dq + t_dkdv * full / pairs_dkdv
        n_groups = w.P * w.B * kvp
        self.last.update(bwd_rows=n_bwd_rows, bwd_groups=n_groups,
                         bwd_sampled_s=tb3 - tb0)
        return (tb1 - tb0) + (tb3 - tb2) + n_groups * t_group

    def calibrate(self, attn_budget_s):
        """Row count whose forward attention takes about `attn_budget_s` seconds
        (forward only: the backward sample is sized from it)."""
        n = 16
        bwd, self.backward = self.backward, False
        try:
            while True:
                _, nr, pairs, wall = self.step(n)
                if wall > attn_budget_s or n >= self.w.S:
                    return n
                n = min(self.w.S, n * 4)
        finally:
            self.backward = bwd

    def describe(self, n_rows):
        w = self.w
        ring = f", {w.ring} ring positions" if w.ring > 1 else ""
        text = (f"{w.name} (P={w.P}{ring}, S={w.S}, {w.n_head} heads, D={w.head_dim}): split, RoPE and the 4 loop "
                f"all-to-alls in full; attention for {n_rows} random query rows of all {w.n_head} heads, "
                f"scaled to the full causal triangle by query-key pairs")
        if self.backward:
            G = (w.n_head // w.P) // self.op.kvp
            text += (f"; backward: dO all-to-all, the inverse all-to-alls of dQ, dK, dV and the inverse RoPE in "
                     f"full; the attention backward of 1 of {w.P * w.B * self.op.kvp} (rank, batch, kv-head) "
                     f"groups ({G} q-head(s)) with its statistics phase in full and its dQ and dK/dV phases for "
                     f"{self.bwd_rows_for(n_rows)} random query and key rows, scaled by query-key pairs and "
                     f"by the number of groups")
        else:
            text += "; forward only"
        return text


def run_sweep(args):
    """Permutation alone at the head-count bound (P=32, one head per virtual
    rank, 32 heads, D=128, bf16), S = 4K..128K, RoPE on and off: median time
    of the seq->head pack of Q, K, V and of the head->seq unpack of O, with a
    512 MiB L2 flush before every timed launch.  Prints one JSON line."""
    from ulysses_sequence_attention_seq_gb300 import binding as U
    from ulysses_sequence_attention_seq_gb300.synthetic import SWEEP_S
    hbm = load_peaks()[0]
    dev = torch.device("cuda", 0)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1005)
    out = []
    for S in SWEEP_S:
        for rope in (True, False):
            prob = U.Problem(B=1, S=S, hidden=4096, n_head=32, n_kv_head=32, head_dim=128, P=32,
                             use_rope=rope)
            buf = U.Buffers(prob, device=dev)
            for t in (buf.q_seq, buf.k_seq, buf.v_seq, buf.o_head):
                t.copy_(torch.randn(t.shape, generator=gen, device=dev, dtype=torch.float32))
            U.ulysses_workspace_init(prob, buf.ws)
            res = {}
            for name, fn in (("pack", lambda: U.ulysses_pack_qkv(prob, buf.q_seq, buf.k_seq, buf.v_seq, buf.q_head,
                                                                 buf.k_head, buf.v_head, buf.ws)),
                             ("unpack", lambda: U.ulysses_unpack_out(prob, buf.o_head, buf.o_seq))):
                if name == "unpack" and not rope:
                    continue  # the unpack has no RoPE; timed once per S
                ts = []
                for it in range(args.warmup + args.steps):
                    flush.fill_(it & 255)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    fn()
                    b.record()
                    torch.cuda.synchronize()
                    if it >= args.warmup:
                        ts.append(a.elapsed_time(b))
                ms = statistics.median(ts)
                nbytes = (3 if name == "pack" else 1) * 2 * S * 4096 * 2
                res[name] = {"ms": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9, "frac_of_measured_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm,
                             "bytes": nbytes}
            assert U.ulysses_read_status(buf.ws) == 0
            out.append({"S": S, "rope": rope, **res})
            del buf
    print(json.dumps({"sweep": "permute P=32 B=1 heads=32 D=128 bf16", "hbm_peak_GBs": hbm, "results": out}))


def run_proj(args, w):
    """The QKV projection with the pack and RoPE fused (ulysses_qkv_proj_pack) on
    the workload's shapes with synthetic weights: X [P*B*Sl, hidden] times
    W^T [hidden, (n_head + 2 n_kv_head) D], plus bias.  One JSON line."""
    from ulysses_sequence_attention_seq_gb300 import binding as U
    dev = torch.device("cuda", 0)
    prob = U.Problem.from_workload(w)
    buf = U.Buffers(prob, device=dev, backward=False)
    H, N = w.hidden, (w.n_head + 2 * w.n_kv_head) * w.head_dim
    g = torch.Generator().manual_seed(77)
    x = U.seq_layout(torch.randn(w.B, w.S, H, generator=g).to(torch.bfloat16), w.P).to(dev)
    W = (torch.randn(N, H, generator=g) / H ** 0.5).to(torch.bfloat16).to(dev)
    b = (0.1 * torch.randn(N, generator=g)).to(torch.bfloat16).to(dev)
    U.ulysses_workspace_init(prob, buf.ws)
    stream = torch.cuda.current_stream()

    def step():
        U.ulysses_qkv_proj_pack(prob, x, W, b, buf.q_head, buf.k_head, buf.v_head, buf.ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if U.ulysses_read_status(buf.ws) != 0:
        raise RuntimeError("device status word set during warm-up")
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / args.steps
    hbm, tf_burst, tf_sust, peak_src = load_peaks()
    flops = 2.0 * w.B * w.S * N * H
    tf = flops / (ms * 1e-3) / 1e12
    # the output projection with the unpack folded into its loads (S/P % 128 == 0)
    out = None
    if w.Sl % 128 == 0:
        Wo = (torch.randn(H, H, generator=g) / H ** 0.5).to(torch.bfloat16).to(dev)
        bo = (0.1 * torch.randn(H, generator=g)).to(torch.bfloat16).to(dev)
        y = torch.empty(w.P, w.B, w.Sl, H, dtype=torch.bfloat16, device=dev)

        def ostep():
            U.ulysses_out_proj_unpack(prob, buf.q_head, Wo, bo, y, buf.ws)

        for _ in range(args.warmup):
            ostep()
        a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            ostep()
        b2.record(stream)
        torch.cuda.synchronize()
        oms = a.elapsed_time(b2) / args.steps
        otf = 2.0 * w.B * w.S * H * (w.n_head * w.head_dim) / (oms * 1e-3) / 1e12
        out = {"kernel": f"qkv_proj_kernel<{w.head_dim}, out>", "ms": oms, "achieved_tflops": otf,
               "frac": otf / tf_sust, "M_tokens": w.B * w.S, "N_features": H, "K_features": w.n_head * w.head_dim}

        # the whole attention layer forward: projection + pack + RoPE, attention,
        # output projection + unpack
        def lstep():
            step()
            U.ulysses_attn_fwd(prob, buf.q_head, buf.k_head, buf.v_head, buf.o_head, buf.lse, buf.ws)
            ostep()

        for _ in range(args.warmup):
            lstep()
        a.record(stream)
        for _ in range(args.steps):
            lstep()
        b2.record(stream)
        torch.cuda.synchronize()
        lms = a.elapsed_time(b2) / args.steps
        out["layer_fwd"] = {"ms": lms, "tokens_per_s": w.B * w.S / (lms * 1e-3),
                            "calls": "ulysses_qkv_proj_pack + ulysses_attn_fwd + ulysses_out_proj_unpack"}
    print(json.dumps({
        "metric": "QKV projection + seq->head pack + RoPE (fused) TFLOP/s", "value": tf, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic (seeded normal activations and weights)",
        "config": {"workload": w.name, "M_tokens": w.B * w.S, "N_features": N, "K_hidden": H,
                   "kv_replicas": w.P // w.n_kv_head if w.n_kv_head < w.P else 1},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": tf_sust, "unit": "TFLOP/s", "frac": tf / tf_sust,
                     "peak_source": f"{peak_src} bf16 sustained", "kernel": f"qkv_proj_kernel<{w.head_dim}>"},
        "out_proj_unpack": out,
        "clocks": clk, "gpu_launches": args.steps, "device_status": U.ulysses_read_status(buf.ws)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="C4", choices=sorted(WORKLOADS) + sorted(EXTRA_WORKLOADS))
    ap.add_argument("--impl", default="ulysses", choices=["ulysses", "reference"])
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--bwd-mode", default="ds_store", choices=["ds_store", "two_kernel", "fused"],
                    help="the backward on the headline step (the other modes are timed beside it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="time the permutation alone over S = 4K..128K")
    ap.add_argument("--proj", action="store_true",
                    help="time the fused QKV projection + pack + RoPE on the workload's shapes")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.sweep:
        run_sweep(args)
        return
    if args.proj:
        run_proj(args, WORKLOADS[args.workload] if args.workload in WORKLOADS else EXTRA_WORKLOADS[args.workload])
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    w = WORKLOADS[args.workload] if args.workload in WORKLOADS else EXTRA_WORKLOADS[args.workload]
    hbm, tf_burst, tf_sust, peak_src = load_peaks()
    tokens = w.B * w.S

    if args.impl == "reference":
        if rank != 0:
            return
        ob = OracleBench(w, backward=w.backward and not args.fwd_only)
        per_step_budget = max(2.0, 150.0 / max(args.steps + args.warmup, 1))
        n_rows = ob.calibrate(per_step_budget / 4)
        times, walls = [], []
        for _ in range(args.steps):
            t_full, _, _, wall = ob.step(n_rows)
            times.append(t_full)
            walls.append(wall)
        t = statistics.median(times)
        value = tokens / t
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
                "ms_per_step_kind": "extrapolated_from_sample",
                "sample_wall_ms_per_step": statistics.median(walls) * 1e3,
                "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": line_config(w, ob.passes, "n/a (host cores)", "host cores, P virtual ranks (oracle)"),
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": ob.nthreads, "kind": "oracle",
                                 "sample": ob.describe(n_rows)},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    r = run_ulysses(args, w, rank, world)
    ms = max_over_ranks(r["total_ms"], world) / args.steps
    e2e_ms = max_over_ranks(r["e2e_ms"], world) / args.steps
    per = {k: statistics.mean(v) for k, v in r["per"].items()}
    fl = attn_fwd_flops(w)
    es = 2 if w.dtype == "bf16" else 4
    attn_ms = per["attn_fwd"]
    bwd_parts = tuple(k for k in per if k.startswith("bwd_"))
    bwd_ms = sum(per[k] for k in bwd_parts) if bwd_parts else None
    bwd_tflops = 2.0 * fl / (bwd_ms * 1e-3) / 1e12 if bwd_ms else None
    attn_tflops = fl / (attn_ms * 1e-3) / 1e12
    pack_gbs = permute_bytes(w, es) / (per["pack_qkv"] * 1e-3) / 1e9
    unpack_gbs = 2.0 * w.B * w.S * w.n_head * w.head_dim * es / (per["unpack_out"] * 1e-3) / 1e9
    # Tensor-core kernels: algorithmic FLOPs per launch (the products the
    # method defines: forward S and PV; backward dV, dP, dQ, dK, each half a
    # forward) and the FLOPs each kernel executes (dK/dV and dQ both recompute
    # S, dQ also dP).
    # The fp32 workload's forward runs on the CUDA cores (fp32 FMA): its peak
    # is derived, SMs x 128 fp32 lanes x 2 FLOP per FMA x the maximum SM clock.
    fp32 = w.dtype != "bf16"
    sm_max = r["clocks"].get("sm_max_mhz") or SM_MAX_MHZ_FALLBACK
    alu_peak = r["sms"] * 128 * 2 * sm_max * 1e6 / 1e12
    peak_k = alu_peak if fp32 else tf_sust
    tc = {"attn_fwd": ("attn_fwd_simt_kernel" if fp32 else "attn_fwd_tc_kernel", fl, fl)}
    tc.update({k: BWD_TC[k](fl) for k in bwd_parts if k in BWD_TC})
    kernels = {}
    for k, (kname, alg, exe) in tc.items():
        a_tf = alg / (per[k] * 1e-3) / 1e12
        kernels[k] = {"kernel": f"{kname}<{w.head_dim}>", "ms": per[k], "algorithmic_tflop": alg / 1e12,
                      "achieved_tflops": a_tf, "frac": a_tf / peak_k,
                      "executed_tflops": exe / (per[k] * 1e-3) / 1e12,
                      "executed_frac": exe / (per[k] * 1e-3) / 1e12 / peak_k}
    # dQ from the stored dS tiles reads them once: bound by HBM
    hbm_kernels = {}
    if "bwd_dq_ds" in per:
        nb = dq_ds_bytes(w, es)
        gbs = nb / (per["bwd_dq_ds"] * 1e-3) / 1e9
        hbm_kernels["bwd_dq_ds"] = {"bound": "hbm", "kernel": f"dq_ds_kernel<{w.head_dim}>", "achieved": gbs,
                                    "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "bytes_per_launch": nb,
                                    "traffic": TRAFFIC.get(("bwd_dq_ds", w.name)),
                                    "note": "bytes: every stored dS tile, K and dQ once each"}
    bwd_modes = None
    if bwd_ms:
        by_mode = {r["bwd_mode"]: {k: per[k] for k in bwd_parts}}
        by_mode.update({m: {k: statistics.mean(v) for k, v in kp.items()} for m, kp in r["alt_per"].items()})
        bwd_modes = {}
        for m, kms in by_mode.items():
            main_k = max((k for k in kms if k in BWD_TC), key=lambda k: kms[k])
            kname, alg, exe = BWD_TC[main_k](fl)
            a_tf = alg / (kms[main_k] * 1e-3) / 1e12
            bwd_modes[m] = {"ms": sum(kms.values()), "kernel_ms": kms, "kernel": f"{kname}<{w.head_dim}>",
                            "kernel_achieved_tflops": a_tf, "kernel_frac": a_tf / tf_sust,
                            "kernel_executed_tflops": exe / (kms[main_k] * 1e-3) / 1e12, "note": BWD_NOTES[m]}
        bwd_modes["headline_uses"] = r["bwd_mode"]
    dominant = max(kernels, key=lambda k: kernels[k]["ms"])
    dk = kernels[dominant]
    # One exponential per (query, key) pair the forward computes, against the
    # measured ex2 rate per SM per cycle at the median SM clock of the run.
    exps = w.B * w.n_head * (w.S * (w.S + 1) / 2 if w.causal else float(w.S) * w.S)
    clk_hz = (r["clocks"].get("sm_mhz") or 0) * 1e6
    mufu = None
    if clk_hz > 0 and r["ex2_rate"] > 0 and not fp32:
        ach = exps / (attn_ms * 1e-3) / (r["sms"] * clk_hz)
        mufu = {"bound": "mufu", "kernel": f"attn_fwd_tc_kernel<{w.head_dim}>", "achieved": ach,
                "peak": r["ex2_rate"], "unit": "ex2/SM/cycle", "frac": ach / r["ex2_rate"], "exps_per_launch": exps,
                "peak_source": "measured on this GPU by ulysses_selftest_ex2_rate",
                "note": "exponentials per forward / kernel time / (SMs x median SM clock)"}
    fwd_tokens = job_throughput(tokens, (per["pack_qkv"] + attn_ms + per["unpack_out"]) * 1e-3, world)
    line = {
        "metric": METRIC, "value": job_throughput(tokens, ms * 1e-3, world), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded normal inputs of the workload's shape)",
        "config": line_config(w, "fwd+bwd" if r["backward"] else "fwd",
                              "inputs larger than L2 (Q/K/V/O each >= 128 MiB); no flush",
                              "replicas" if world > 1 else "single GPU, P virtual ranks"),
        "fwd_tokens_per_s": fwd_tokens,
        "attn_fwd_tflops": attn_tflops, "attn_fwd_ms": attn_ms,
        "attn_bwd_tflops": bwd_tflops, "attn_bwd_ms": bwd_ms,
        "attn_bwd_tflops_2p5x": bwd_tflops * 1.25 if bwd_tflops else None,
        "attn_bwd_flops_note": "backward algorithmic FLOPs = 2x forward (dV, dP, dQ, dK); the QK^T recompute is not "
                               "counted (attn_bwd_tflops_2p5x counts it: 2.5x forward)",
        "pack_gbs": pack_gbs, "unpack_gbs": unpack_gbs,
        "kernel_ms": per,
        "kernel_ms_median": {k: statistics.median(v) for k, v in r["per"].items()},
        "kernel_ms_min": {k: min(v) for k, v in r["per"].items()},
        "tensor_kernels": kernels,
        "bwd_modes": bwd_modes,
        "roofline": {"bound": "alu" if fp32 else "tensor", "achieved": dk["achieved_tflops"], "peak": peak_k,
                     "unit": "TFLOP/s", "frac": dk["frac"], "traffic": TRAFFIC.get((dominant, w.name)),
                     "peak_source": (f"derived fp32 FMA: {r['sms']} SMs x 128 lanes x 2 FLOP x {sm_max:.0f} MHz"
                                     if fp32 else f"{peak_src} bf16 sustained"), "kernel": dk["kernel"],
                     "peak_burst": None if fp32 else tf_burst,
                     "frac_burst": None if fp32 else dk["achieved_tflops"] / tf_burst,
                     "sm_mhz": r["clocks"].get("sm_mhz"), "bwd_mode": r["bwd_mode"],
                     # DRAM rate of the same launch (traffic from the ncu capture over this run's time)
                     "dram_gbs": (TRAFFIC[(dominant, w.name)] / (dk["ms"] * 1e-3) / 1e9
                                  if (dominant, w.name) in TRAFFIC else None),
                     "note": "dominant kernel by time; achieved counts its algorithmic products only; frac is "
                             "against the sustained (power-capped) cuBLAS figure, frac_burst against the burst "
                             "one; sm_mhz is the median SM clock sampled while the timed steps ran"
                             + ("; in the dS-store backward the dK/dV kernel also writes every tile pair's dS "
                                "(dram_gbs: its DRAM traffic over its time)" if dominant == "bwd_dkdv_ds" else "")},
        "secondary_rooflines": {**{k: {"bound": "alu" if fp32 else "tensor", "achieved": v["achieved_tflops"],
                                       "peak": peak_k,
                                       "unit": "TFLOP/s", "frac": v["frac"], "traffic": TRAFFIC.get((k, w.name))}
                                   for k, v in kernels.items() if k != dominant},
                                **hbm_kernels,
                                "pack_qkv": {"bound": "hbm", "achieved": pack_gbs, "peak": hbm, "unit": "GB/s",
                                             "frac": pack_gbs / hbm},
                                "unpack_out": {"bound": "hbm", "achieved": unpack_gbs, "peak": hbm, "unit": "GB/s",
                                               "frac": unpack_gbs / hbm},
                                **({"attn_fwd_mufu": mufu} if mufu else {})},
        "clocks": r["clocks"],
        "e2e": {"value": job_throughput(tokens, e2e_ms * 1e-3, world), "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "host_link": {**r.get("link", {}),
                      "note": "pinned host <-> device copy rate on this machine, one copy at a time (h2d_gbs, "
                              "d2h_gbs) and with an upload and a download running at once (*_both_ways, as the "
                              "end-to-end leg runs them); the end-to-end leg hides every step's copies behind the "
                              "compute but the first upload and the last download"},
        "gpu_launches": r["launches"],
        # the folded mode (both All-to-Alls as addressing) is timed beside the
        # headline path, not on it: it needs q and k rotated by their producer
        # (RoPE off), and its backward reads dO and Q in sequence layout with
        # strided tile rows, which costs more than the dO pack it saves
        "folded_mode": ({**r["folded"], "on_headline_path": False,
                         "note": "RoPE off (q, k rotated by their producer); timed beside the headline path"}
                        if r["folded"] else None),
        "device_status": r["status"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ob = OracleBench(w, backward=r["backward"])
        n_rows = ob.calibrate(4.0)
        t_full, _, _, wall = ob.step(n_rows)
        line["cpu_baseline"] = {"value": tokens / t_full, "unit": "tokens/s", "cores": ob.nthreads,
                                "kind": "oracle", "passes": ob.passes, "sample": ob.describe(n_rows),
                                "value_kind": "extrapolated_from_sample", "sample_wall_s": wall}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
