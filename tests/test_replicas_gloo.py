"""Replica mode of bench.py on the CPU: two gloo ranks (world_size 2).

The path is run as independent replicas (one per GPU, no collective on the
data path); only the timing is reduced across ranks: the slowest replica's
time, and the whole-job throughput = units of all ranks / that time."""

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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                          # rank 1 is the slower replica
        slowest = bench.max_over_ranks(mine, "cpu")
        value = bench.job_throughput(1e9, 4, world, slowest, 1e9)
        results[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_use_the_slowest_replica():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        results = manager.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        got = dict(results)
    assert got[0] == got[1]
    slowest, value = got[0]
    assert slowest == 15.0
    # 1e9 units per step, 4 steps, 2 replicas in 15 ms -> 533.3 units/ns scaled by 1e9
    assert value == pytest.approx(1e9 * 4 * 2 / 0.015 / 1e9)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(2e9, 10, 1, 1000.0, 1e9) == pytest.approx(20.0)

