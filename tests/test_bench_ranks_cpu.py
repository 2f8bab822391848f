"""The multi-rank bench logic on CPU: two gloo ranks (replicas) agree on the
slowest rank's time, and the whole-job throughput counts every replica."""
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


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank          # rank 1 is the slower replica
        out[rank] = bench.max_over_ranks(mine, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 15.0


def test_job_throughput_counts_all_replicas():
    one = bench.job_tflops(1, 4_000_000_000_000, 10, 20.0)
    assert one == pytest.approx(2000.0)
    assert bench.job_tflops(2, 4_000_000_000_000, 10, 20.0) == pytest.approx(2 * one)
