"""Steps of the path from pinned host memory to pinned host memory, with the
transfers of neighbouring steps overlapping the compute.

The C ABI's calls are asynchronous on the stream they are given, so a caller
whose inputs arrive from the host can keep the GPU busy the way the pages'
pipeline keeps its ranks busy: while step k computes, step k+1's inputs are
uploaded and step k's finished outputs downloaded.  `StreamedPath` does that
with two device buffer sets (each with its own workspace) and three streams,
handing over between them at the granularity of the C-ABI calls:

    upload stream    q, k, v of step k into set k % 2 once step k-2's pack has
                     read them; then dO once step k-2's backward prepare has;
    compute stream   pack (after q, k, v arrive), attention, unpack; then (after
                     dO arrives) the backward's prepare, dK/dV and dQ steps;
    download stream  O as soon as the unpack is done (it overlaps the backward),
                     dK and dV after the dK/dV step (they overlap dQ), dQ last.

So a run of K steps waits, beyond the compute, only for the first step's q, k,
v and the last step's dQ (the O download alone without a backward); dO of the
first step arrives while its forward runs.  Before a step overwrites one of
its outputs, the download of that output from two steps back has finished.

Orchestration only: every step is the same sequence of C-ABI calls as
`binding.Buffers.forward` followed by the three calls that make up
`ulysses_attn_bwd` (bwd_mode "two_kernel"), `ulysses_attn_bwd_ds` (bwd_mode
"ds_store": dK/dV storing dS, then dQ from the stored tiles, each set's
workspace holding its tiles) or `ulysses_attn_bwd_fused` (bwd_mode "fused");
nothing here computes.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Union

import torch

from . import binding as U

HostSet = Dict[str, torch.Tensor]


def _pick(x: Union[HostSet, Sequence[HostSet]], k: int) -> HostSet:
    return x if isinstance(x, dict) else x[k % len(x)]


class StreamedPath:
    IN = ("q_seq", "k_seq", "v_seq")
    OUT = ("o_seq",)
    IN_BWD = ("do_seq",)
    OUT_BWD = ("dq_seq", "dk_seq", "dv_seq")

    BWD_MODES = ("two_kernel", "ds_store", "fused")

    def __init__(self, prob: U.Problem, backward: bool = False, device="cuda", bwd_mode: str = "two_kernel"):
        if bwd_mode not in self.BWD_MODES:
            raise ValueError(f"bwd_mode must be one of {self.BWD_MODES}")
        self.prob, self.backward, self.bwd_mode = prob, backward, bwd_mode
        self.dev = torch.device(device)
        self.sets = [U.Buffers(prob, device=self.dev, backward=backward, fused=backward and bwd_mode == "fused",
                               ds=backward and bwd_mode == "ds_store") for _ in range(2)]
        for b in self.sets:
            U.ulysses_workspace_init(prob, b.ws)
        self.compute = torch.cuda.current_stream(self.dev)
        self.up = torch.cuda.Stream(self.dev)
        self.down = torch.cuda.Stream(self.dev)
        # per buffer set, the last step's hand-over events (None: not yet used)
        names = ("qkv_read", "do_read", "o_down", "dkv_down", "dq_down")
        self._ev: List[Dict[str, Optional[torch.cuda.Event]]] = [dict.fromkeys(names) for _ in range(2)]

    def in_names(self):
        return self.IN + (self.IN_BWD if self.backward else ())

    def out_names(self):
        return self.OUT + (self.OUT_BWD if self.backward else ())

    def _record(self, stream) -> torch.cuda.Event:
        e = torch.cuda.Event()
        e.record(stream)
        return e

    def _wait(self, stream, ev: Optional[torch.cuda.Event]) -> None:
        if ev is not None:
            stream.wait_event(ev)

    def run(self, host_in: Union[HostSet, Sequence[HostSet]], host_out: Union[HostSet, Sequence[HostSet]],
            steps: int) -> None:
        """Enqueue `steps` steps.  host_in maps q_seq, k_seq, v_seq (and do_seq)
        to pinned host tensors in sequence layout; host_out maps o_seq (and
        dq_seq, dk_seq, dv_seq) to pinned host tensors that receive the results.
        Either may be a list of such maps, step k using entry k % len.  Returns
        once enqueued; the compute stream is ordered after the last download, so
        synchronizing it (or an event recorded on it) waits for everything."""
        p = self.prob
        start = self._record(self.compute)
        self.up.wait_event(start)
        self.down.wait_event(start)
        for k in range(steps):
            b, ev = self.sets[k % 2], self._ev[k % 2]
            hin, hout = _pick(host_in, k), _pick(host_out, k)
            # upload q, k, v (and dO) once step k-2 has read this set's copies
            self._wait(self.up, ev["qkv_read"])
            with torch.cuda.stream(self.up):
                for n in self.IN:
                    getattr(b, n).copy_(hin[n], non_blocking=True)
            qkv_up = self._record(self.up)
            if self.backward:
                self._wait(self.up, ev["do_read"])
                with torch.cuda.stream(self.up):
                    b.do_seq.copy_(hin["do_seq"], non_blocking=True)
                do_up = self._record(self.up)
            # forward
            self.compute.wait_event(qkv_up)
            U.ulysses_pack_qkv(p, b.q_seq, b.k_seq, b.v_seq, b.q_head, b.k_head, b.v_head, b.ws, self.compute)
            ev["qkv_read"] = self._record(self.compute)
            U.ulysses_attn_fwd(p, b.q_head, b.k_head, b.v_head, b.o_head, b.lse, b.ws, self.compute)
            self._wait(self.compute, ev["o_down"])
            U.ulysses_unpack_out(p, b.o_head, b.o_seq, self.compute)
            o_ready = self._record(self.compute)
            self.down.wait_event(o_ready)
            with torch.cuda.stream(self.down):
                hout["o_seq"].copy_(b.o_seq, non_blocking=True)
            ev["o_down"] = self._record(self.down)
            if not self.backward:
                continue
            # backward: prepare, dK/dV, dQ; each result downloaded when it is done
            self.compute.wait_event(do_up)
            U.ulysses_attn_bwd_prepare(p, b.o_head, b.lse, b.do_seq, b.ws, self.compute)
            ev["do_read"] = self._record(self.compute)
            self._wait(self.compute, ev["dkv_down"])
            if self.bwd_mode == "ds_store":
                U.ulysses_attn_bwd_dkdv_ds(p, b.q_head, b.k_head, b.v_head, b.dk_seq, b.dv_seq, b.ws, self.compute)
            elif self.bwd_mode == "fused":
                U.ulysses_attn_bwd_dkdvq(p, b.q_head, b.k_head, b.v_head, b.dk_seq, b.dv_seq, b.ws, self.compute)
            else:
                U.ulysses_attn_bwd_dkdv(p, b.q_head, b.k_head, b.v_head, b.dk_seq, b.dv_seq, b.ws, self.compute)
            dkv_ready = self._record(self.compute)
            self._wait(self.compute, ev["dq_down"])
            if self.bwd_mode == "ds_store":
                U.ulysses_attn_bwd_dq_ds(p, b.k_head, b.dq_seq, b.ws, self.compute)
            elif self.bwd_mode == "fused":
                U.ulysses_attn_bwd_dq_finish(p, b.dq_seq, b.ws, self.compute)
            else:
                U.ulysses_attn_bwd_dq(p, b.q_head, b.k_head, b.v_head, b.dq_seq, b.ws, self.compute)
            dq_ready = self._record(self.compute)
            self.down.wait_event(dkv_ready)
            with torch.cuda.stream(self.down):
                hout["dk_seq"].copy_(b.dk_seq, non_blocking=True)
                hout["dv_seq"].copy_(b.dv_seq, non_blocking=True)
            ev["dkv_down"] = self._record(self.down)
            self.down.wait_event(dq_ready)
            with torch.cuda.stream(self.down):
                hout["dq_seq"].copy_(b.dq_seq, non_blocking=True)
            ev["dq_down"] = self._record(self.down)
        # the compute stream waits for every download (the download stream is in order)
        self.compute.wait_event(self._record(self.down))

    def status(self) -> int:
        """OR of both buffer sets' device status words (synchronizes)."""
        return U.ulysses_read_status(self.sets[0].ws) | U.ulysses_read_status(self.sets[1].ws)
