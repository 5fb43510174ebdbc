"""The multi-GPU bench path runs independent replicas, one per rank, with no
collective on the data path. Its only cross-rank steps are a barrier and a max
over the ranks' timed regions. This test runs that logic as two gloo ranks on
the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [10.0, 12.5][rank]  # each rank's own timed region
        bench.barrier(world)
        ms_max = bench.max_over_ranks(ms, world)
        value = bench.job_throughput(1000, 4, world, ms_max)
        q.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms_max, value in got:
        assert ms_max == 12.5
        # 2 ranks x 4 steps x 1000 samples in 12.5 ms
        assert value == pytest.approx(2 * 4 * 1000 / 12.5e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(10, 2, 1, 4.0) == pytest.approx(5000.0)
