"""The multi-rank path of bench.py on CPU: two gloo ranks combine their timings
the way the GPU ranks do (max over ranks, whole-job bytes), and rank-dependent
seeds give each rank its own copy of the workload."""
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


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 10.0 + 5.0 * rank           # rank 1 is the slower one
        ms_per_step, gbs = bench.combine_ranks(ms_local, 100, 1e6, world, dist, device="cpu")
        results[rank] = (ms_per_step, gbs)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_all_bytes():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
    assert set(results.keys()) == {0, 1}
    for r in range(world):
        ms_per_step, gbs = results[r]
        assert ms_per_step == pytest.approx(15.0 / 100)
        assert gbs == pytest.approx(1e6 * world / (0.15e-3) / 1e9)


def test_single_rank_needs_no_process_group():
    ms_per_step, gbs = bench.combine_ranks(8.0, 4, 2e6, 1)
    assert ms_per_step == 2.0 and gbs == pytest.approx(2e6 / 2e-3 / 1e9)
