"""The benchmark's multi-rank bookkeeping on CPU with two gloo ranks.

With N GPUs the benchmark runs N replicas of the workload (the path has no exchange
step) and reports the whole job's throughput from the slowest rank's time; these
tests run that reduction across two real processes without a GPU.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], dist, "cpu")
        steps = int(bench.max_over_ranks(float(100 + rank), dist, "cpu"))
        out[rank] = (slowest, steps)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_step_count():
    world, port = 2, _free_port()
    times = [12.5, 17.25]
    manager = mp.get_context("spawn").Manager()    # no fork of a threaded test process
    out = manager.dict()
    mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
    assert out[0] == out[1] == (17.25, 101)


def test_whole_job_throughput_counts_every_rank_at_the_slowest_time():
    flops = 2 * 1024 ** 3
    one = bench.whole_job_tflops(flops, 100, 1, 1.0)
    assert one == pytest.approx(flops * 100 / 1e-3 / 1e12)
    assert bench.whole_job_tflops(flops, 100, 4, 1.0) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.0, None, "cpu") == 3.0
