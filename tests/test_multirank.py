"""The benchmark's multi-rank path on CPU (gloo, world size 2).

One process per GPU, each running its own replica of the decode round (no
collective on the data path); the job's time is the slowest rank's, found by
one max all-reduce, and the job's throughput counts every rank's bytes.  This
checks that host logic with two CPU ranks that report different times.
"""
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


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took (r + 1) seconds for 10 steps of 1e9 bytes each
        value, elapsed = bench.job_rate(float(rank + 1), 10 ** 9, 10, world)
        out[rank] = (value, elapsed)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_rate_takes_the_slowest_rank_and_sums_the_work():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        value, elapsed = out[rank]
        assert elapsed == 2.0  # the slower rank's time
        assert value == pytest.approx(10.0)  # 2 ranks x 10 GB in 2 s


def test_job_rate_single_rank_needs_no_collective():
    import bench
    value, elapsed = bench.job_rate(0.5, 10 ** 9, 4, 1)
    assert elapsed == 0.5 and value == pytest.approx(8.0)
