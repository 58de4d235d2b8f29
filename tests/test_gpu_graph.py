"""The path is stream-ordered through the C ABI, so a whole step (pack,
attention forward, unpack, and the dS-store or two-kernel backward) can be
captured once into a CUDA graph and replayed: every replay gives, bit for bit,
what the same calls give when launched one by one, for new inputs copied into
the same buffers between replays."""
import pytest
import torch

from pathcheck import GpuRun
from test_gpu_forward import wl
from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300.synthetic import make_inputs

pytestmark = pytest.mark.gpu

OUTS = ("o_seq", "dq_seq", "dk_seq", "dv_seq")


@pytest.mark.parametrize("mode", ["ds_store", "two_kernel"])
def test_step_replays_from_a_cuda_graph(mode):
    w = wl(8, 1, 1024, 8, 2, 128).with_(backward=True)
    run = GpuRun(w, backward=True, ds=mode == "ds_store")
    b = run.buf
    backward = b.backward_ds if mode == "ds_store" else b.backward

    def step():
        b.forward()
        backward()

    step()                                  # warm-up outside the capture (first-use host setup)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    torch.cuda.synchronize()
    for seed in (11, 12):
        ins = make_inputs(w.with_(seed=seed), with_grad=True)
        for name, key in (("q_seq", "q"), ("k_seq", "k"), ("v_seq", "v"), ("do_seq", "do")):
            getattr(b, name).copy_(U.seq_layout(ins[key], w.P))
        step()                              # one by one
        torch.cuda.synchronize()
        want = {n: getattr(b, n).clone() for n in OUTS}
        for n in OUTS:
            getattr(b, n).fill_(float("nan"))
        graph.replay()                      # the captured step
        torch.cuda.synchronize()
        assert U.ulysses_read_status(b.ws) == 0
        for n in OUTS:
            assert torch.equal(getattr(b, n), want[n]), (seed, n)
