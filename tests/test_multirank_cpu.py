"""The N > 1 path of the benchmark on the CPU: two gloo ranks, each with its
own replica of the workload (slices are independent, so there is no
data-path collective).  The reported time is the max over ranks and the
throughput counts every rank's slices."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    ms = bench.max_over_ranks(1.0 + rank * 0.5, "cpu")      # rank 1 is slower
    out[rank] = (ms, bench.weak_scaling_value(74, world, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        ms, val = out[r]
        assert ms == 1.5
        assert val == pytest.approx(74 * 2 / 1.5e-3)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(2.0, "cpu") == 2.0
    assert bench.weak_scaling_value(74, 1, 2.0) == pytest.approx(37000.0)
