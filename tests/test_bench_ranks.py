"""The benchmark's multi-rank host logic on CPU with two gloo ranks: the
job's step time is the slowest rank's, and the whole-job throughput sums the
ranks' work over that time (replicas: no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
    value = bench.whole_job_tflops(2.0 * 8192 * 4096 * 12288, ms, world)
    dist.barrier()
    out[rank] = (ms, value)
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, times = 2, [0.571, 0.604]
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
    for r in range(world):
        ms, value = out[r]
        assert ms == pytest.approx(0.604)
        assert value == pytest.approx(2 * 2.0 * 8192 * 4096 * 12288 / 0.604e-3 / 1e12)


def test_one_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(0.5, 1, torch.device("cpu")) == 0.5
    assert bench.whole_job_tflops(1e12, 1000.0, 1) == pytest.approx(1.0)
