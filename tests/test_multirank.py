"""The bench's multi-process path on CPU (gloo, world size 2).

The attention path shards with no exchange (every rank runs its own replica:
sequences and KV heads are independent), so the only cross-rank step is the
timing: the whole job takes as long as its slowest rank, and its throughput
is every rank's units over that time.  Run as two gloo processes on
127.0.0.1.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        own_ms = 10.0 + 5.0 * rank            # rank 1 is the slower one
        ms = bench.max_over_ranks(torch, own_ms, world, torch.device("cpu"))
        rate = bench.whole_job_rate(1000.0, world, ms)
        results[rank] = (ms, rate)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = free_port()
        procs = [ctx.Process(target=worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(60)
            assert p.exitcode == 0
        assert results[0] == results[1] == (15.0, 2 * 1000.0 / 0.015)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(torch, 7.5, 1, torch.device("cpu")) == 7.5
    assert bench.whole_job_rate(3.0, 1, 1000.0) == pytest.approx(3.0)
