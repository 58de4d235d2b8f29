"""The streamed host-to-host path (two device buffer sets, upload / compute /
download streams handing over per C-ABI call) gives exactly what the plain
device path gives, for every step, with different inputs at every step so
that a result read or written out of order cannot go unnoticed; with either
backward (two-kernel, or dS-store)."""
import pytest
import torch

from pathcheck import GpuRun
from test_gpu_forward import wl
from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300.streamed import StreamedPath

pytestmark = pytest.mark.gpu


def _outs(sp):
    return {n: torch.empty(getattr(sp.sets[0], n).shape, dtype=getattr(sp.sets[0], n).dtype, pin_memory=True)
            for n in sp.out_names()}


@pytest.mark.parametrize("backward,mode", [(False, "two_kernel"), (True, "two_kernel"), (True, "ds_store")])
def test_streamed_steps_match_the_device_path(backward, mode):
    w = wl(4, 1, 1024, 8, 4, 128).with_(backward=backward)
    sp = StreamedPath(U.Problem.from_workload(w), backward=backward, bwd_mode=mode)
    refs, hosts = [], []
    for seed in (7, 8, 9):
        ref = GpuRun(w.with_(seed=seed), backward=backward, ds=mode == "ds_store")
        ref.forward()
        if backward and mode == "ds_store":
            ref.backward_ds()
        elif backward:
            ref.backward()
        refs.append({n: getattr(ref.buf, n).cpu() for n in sp.out_names()})
        hosts.append({n: getattr(ref.buf, n).cpu().pin_memory() for n in sp.in_names()})
    # one input set for every step
    outs = _outs(sp)
    for i, steps in ((0, 1), (1, 3), (2, 2)):
        sp.run(hosts[i], outs, steps)
        torch.cuda.synchronize()
        assert sp.status() == 0
        for n in sp.out_names():
            assert torch.equal(outs[n], refs[i][n]), (i, n)
    # a different input set at every step (step k uses set k % 3), each
    # step's results into their own host buffers
    outs = [_outs(sp) for _ in range(3)]
    for steps in (3, 5, 4):
        for o in outs:
            for t in o.values():
                t.zero_()
        sp.run(hosts, outs, steps)
        torch.cuda.synchronize()
        assert sp.status() == 0
        for i in range(min(steps, 3)):
            for n in sp.out_names():
                assert torch.equal(outs[i][n], refs[i][n]), (steps, i, n)
