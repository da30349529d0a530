"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

Every rank runs its own batch of (b, h) units with no collective on the data
path; the job's time is the slowest rank's and its throughput counts the
units of all ranks.  The GPU path itself runs one rank per GPU under
torchrun; here two CPU processes check the aggregation."""

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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per_rank_ms = [3.0, 5.0][rank]
        ms = bench.max_over_ranks(per_rank_ms, dist, "cpu")
        units = 1 * 16 * 65536
        out[rank] = (ms, bench.job_value(world, units, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_throughput():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert set(out.keys()) == {0, 1}
    for r in range(world):
        ms, value = out[r]
        assert ms == 5.0
        assert value == pytest.approx(2 * 16 * 65536 / 5e-3)


def test_single_rank_is_the_identity():
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.job_value(1, 1000, 2.0) == pytest.approx(5e5)
