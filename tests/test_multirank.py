"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank replicates the workload (weak scaling, no data-path collective); the only
cross-rank step is the max over ranks of the timed region, and rank 0 reports
the whole job's work over that time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total_ms = 10.0 + 5.0 * rank  # rank 1 is the slowest
        slowest = bench.max_over_ranks(total_ms, "cpu")
        value = bench.job_throughput(1e12, world, steps=4, total_ms=slowest)
        results[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    # both ranks agree on the slowest time; throughput counts both ranks' work
    assert got[0][0] == pytest.approx(15.0) and got[1][0] == pytest.approx(15.0)
    assert got[0][1] == pytest.approx(1e12 * 2 * 4 / 15e-3 / 1e12)


def test_single_process_reduction_is_identity():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_throughput(2e12, 1, 2, 1000.0) == pytest.approx(4.0)
