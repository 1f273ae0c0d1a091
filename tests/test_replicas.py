"""Host-side logic of the multi-GPU bench path (replicas only), on CPU with
world-size-2 gloo process groups: the slowest rank's time is taken, and the
job value aggregates every replica's bytes over it."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.max_over_ranks(times[rank], world)
        out[rank] = (t, bench.whole_job_gbs(1.0e9, t, world))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    times = [1.25, 2.5]  # ms per step on each replica
    mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
    for rank in range(world):
        t, value = out[rank]
        assert t == pytest.approx(2.5)                 # the slowest replica
        assert value == pytest.approx(2 * 1.0 / 2.5e-3)  # 2 GB per step / 2.5 ms = 800 GB/s


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_gbs(2.0e9, 1.0, 1) == pytest.approx(2000.0)
