"""Failure detection on the GPU without a fault: a bounded pipeline wait is made
to run out (a barrier nothing completes), the status word reports it, kernels
launched on that workspace afterwards refuse to start, and once the workspace is
prepared again the path computes the same result as before."""
import pytest
import torch

from pathcheck import GpuRun
from test_gpu_forward import wl
from ulysses_sequence_attention_seq_gb300 import binding as U

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_is_reported():
    w = wl(2, 1, 256, 4, 4, 64)
    run = GpuRun(w)
    run.forward()
    good = run.buf.o_seq.clone()

    U.ulysses_selftest_wait_timeout(run.buf.ws, 20_000_000)   # 20 ms
    word = torch.zeros(1, dtype=torch.int32).pin_memory()
    U.ulysses_read_status_async(run.buf.ws, word)             # enqueued behind the self-test
    torch.cuda.synchronize()
    assert int(word.item()) & U.STATUS_FWD_TIMEOUT
    assert U.ulysses_read_status(run.buf.ws) & U.STATUS_FWD_TIMEOUT

    # with a timeout bit set the attention kernel does not start: O is left alone
    run.buf.o_head.fill_(0)
    run.buf.forward()
    torch.cuda.synchronize()
    assert U.ulysses_read_status(run.buf.ws) & U.STATUS_FWD_TIMEOUT
    assert not run.buf.o_head.any()

    # the context is still usable: prepare the workspace again and the path runs
    U.ulysses_workspace_init(run.prob, run.buf.ws)
    run.forward()
    assert torch.equal(run.buf.o_seq, good)


def test_every_backward_mode_refuses_to_start_after_a_timeout():
    """With a timeout bit in the status word the two-kernel, dS-store and fused
    backwards write no gradient; prepared again, each gives its earlier bits."""
    w = wl(2, 1, 256, 4, 4, 64).with_(backward=True)
    run = GpuRun(w, backward=True, ds=True, fused=True)
    run.forward()
    b = run.buf
    grads = ("dq_seq", "dk_seq", "dv_seq")
    modes = {"two-kernel": b.backward, "dS-store": b.backward_ds, "fused": b.backward_fused}
    good = {}
    for name, call in modes.items():
        call()
        torch.cuda.synchronize()
        assert U.ulysses_read_status(b.ws) == 0
        good[name] = [getattr(b, n).clone() for n in grads]

    U.ulysses_selftest_wait_timeout(b.ws, 20_000_000)        # 20 ms
    for name, call in modes.items():
        for n in grads:
            getattr(b, n).zero_()
        call()
        torch.cuda.synchronize()
        assert U.ulysses_read_status(b.ws) & U.STATUS_FWD_TIMEOUT
        assert not any(getattr(b, n).any() for n in grads), f"{name} backward wrote after a timeout"

    U.ulysses_workspace_init(run.prob, b.ws)
    for name, call in modes.items():
        call()
        torch.cuda.synchronize()
        assert U.ulysses_read_status(b.ws) == 0
        assert all(torch.equal(getattr(b, n), g) for n, g in zip(grads, good[name])), name
