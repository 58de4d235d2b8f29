"""The streamed host-to-host path (two device buffer sets, upload / compute /
download streams) gives exactly what the plain device path gives."""
import pytest
import torch

from pathcheck import GpuRun
from test_gpu_forward import wl
from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300.streamed import StreamedPath

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("backward", [False, True])
def test_streamed_steps_match_the_device_path(backward):
    w = wl(4, 1, 1024, 8, 4, 128).with_(backward=backward)
    sp = StreamedPath(U.Problem.from_workload(w), backward=backward)
    outs = {n: torch.empty(getattr(sp.sets[0], n).shape, dtype=getattr(sp.sets[0], n).dtype, pin_memory=True)
            for n in sp.out_names()}
    for seed, steps in ((7, 1), (8, 3), (9, 2)):
        ref = GpuRun(w.with_(seed=seed), backward=backward)
        ref.forward()
        if backward:
            ref.backward()
        host = {n: getattr(ref.buf, n).cpu().pin_memory() for n in sp.in_names()}
        sp.run(host, outs, steps)
        torch.cuda.synchronize()
        assert sp.status() == 0
        for n in sp.out_names():
            assert torch.equal(outs[n], getattr(ref.buf, n).cpu()), (seed, n)
