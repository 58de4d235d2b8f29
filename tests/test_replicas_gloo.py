"""Multi-process replica logic of bench.py on CPU (gloo, world size 2).

The path has no exchange between GPUs (every virtual rank of one Ulysses group
lives in one HBM), so N GPUs run N independent replicas; the only collective
is the max-over-ranks reduction of the timed region.  This checks that logic
with two gloo ranks that report different times."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = 0.010 * (rank + 1)                     # rank 1 is the slow one
    tmax = bench.max_over_ranks(t, world)
    rate = bench.job_throughput(32768, tmax, world)
    out[rank] = (tmax, rate)
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_replicas_report_slowest_rank_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0][0] == pytest.approx(0.020) and out[1][0] == pytest.approx(0.020)
    assert out[0][1] == pytest.approx(2 * 32768 / 0.020)
    assert out[0] == out[1]
