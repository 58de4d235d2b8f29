"""Steps of the path from pinned host memory to pinned host memory, with the
transfers of neighbouring steps overlapping the compute.

The C ABI's calls are asynchronous on the stream they are given, so a caller
whose inputs arrive from the host can keep the GPU busy the way the pages'
pipeline keeps its ranks busy: while step k computes, step k+1's inputs are
uploaded and step k-1's results downloaded.  `StreamedPath` does exactly that
with two device buffer sets (each with its own workspace) and three streams:

    upload stream    H2D of step k's inputs into set k % 2, after step k-2's
                     compute has finished with that set;
    compute stream   pack, attention, unpack (and the backward) on set k % 2,
                     after its upload and after step k-2's download from it;
    download stream  D2H of step k's outputs, after its compute.

Orchestration only: every step is the same sequence of C-ABI calls as
`binding.Buffers.forward` / `.backward`; nothing here computes.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import torch

from . import binding as U


class StreamedPath:
    IN = ("q_seq", "k_seq", "v_seq")
    OUT = ("o_seq",)
    IN_BWD = ("do_seq",)
    OUT_BWD = ("dq_seq", "dk_seq", "dv_seq")

    def __init__(self, prob: U.Problem, backward: bool = False, device="cuda"):
        self.prob, self.backward = prob, backward
        self.dev = torch.device(device)
        self.sets = [U.Buffers(prob, device=self.dev, backward=backward) for _ in range(2)]
        for b in self.sets:
            U.ulysses_workspace_init(prob, b.ws)
        self.compute = torch.cuda.current_stream(self.dev)
        self.up = torch.cuda.Stream(self.dev)
        self.down = torch.cuda.Stream(self.dev)
        self._computed: List[Optional[torch.cuda.Event]] = [None, None]
        self._downloaded: List[Optional[torch.cuda.Event]] = [None, None]

    def in_names(self):
        return self.IN + (self.IN_BWD if self.backward else ())

    def out_names(self):
        return self.OUT + (self.OUT_BWD if self.backward else ())

    def run(self, host_in: Dict[str, torch.Tensor], host_out: Dict[str, torch.Tensor], steps: int) -> None:
        """Enqueue `steps` steps.  host_in maps q_seq, k_seq, v_seq (and do_seq)
        to pinned host tensors in sequence layout; host_out maps o_seq (and dq_seq,
        dk_seq, dv_seq) to pinned host tensors that receive every step's results.
        Returns once enqueued; the compute stream is ordered after the last
        download, so synchronizing it (or an event recorded on it) waits for
        everything."""
        start = torch.cuda.Event()
        start.record(self.compute)
        self.up.wait_event(start)
        self.down.wait_event(start)
        for k in range(steps):
            s = k % 2
            b = self.sets[s]
            if self._computed[s] is not None:
                self.up.wait_event(self._computed[s])
            with torch.cuda.stream(self.up):
                for n in self.in_names():
                    getattr(b, n).copy_(host_in[n], non_blocking=True)
            uploaded = torch.cuda.Event()
            uploaded.record(self.up)
            self.compute.wait_event(uploaded)
            if self._downloaded[s] is not None:
                self.compute.wait_event(self._downloaded[s])
            b.forward(stream=self.compute)
            if self.backward:
                b.backward(stream=self.compute)
            computed = torch.cuda.Event()
            computed.record(self.compute)
            self._computed[s] = computed
            self.down.wait_event(computed)
            with torch.cuda.stream(self.down):
                for n in self.out_names():
                    host_out[n].copy_(getattr(b, n), non_blocking=True)
            downloaded = torch.cuda.Event()
            downloaded.record(self.down)
            self._downloaded[s] = downloaded
        for e in self._downloaded:
            if e is not None:
                self.compute.wait_event(e)

    def status(self) -> int:
        """OR of both buffer sets' device status words (synchronizes)."""
        return U.ulysses_read_status(self.sets[0].ws) | U.ulysses_read_status(self.sets[1].ws)
