"""The N-replica host logic of the benchmark on CPU (gloo, world size 2): the
row reductions shard into independent replicas with no data-path collective,
so the only exchange is the timing reduction, the slowest rank's time, and the
job's throughput counts every replica's work over that time."""
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


def _worker(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(times[rank], "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_reaches_every_rank():
    world = 2
    times = [1.25, 3.5]
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), times, out), nprocs=world, join=True)
    assert out[0] == out[1] == max(times)


def test_job_throughput_counts_every_replica():
    one = bench.job_gbs(1, 100, 1e9, 50.0)
    two = bench.job_gbs(2, 100, 1e9, 50.0)
    assert two == pytest.approx(2 * one)
    assert bench.job_gbs(2, 100, 1e9, 100.0) == pytest.approx(one)   # a slower rank sets the job's time
