"""The multi-rank path of bench.py on CPU (two gloo ranks, no GPU).

Each rank runs an independent problem of the same size (weak scaling, no
collective on the data path); the job's time is the slowest rank's and its
throughput counts the units of every rank.  The ranks here report different
step times and must all see the maximum.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import bench

    assert bench._dist() == (ws, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        local_ms = 10.0 + 5.0 * rank                    # rank 1 is the slow one
        slowest = bench.max_over_ranks(local_ms, ws, "cpu")
        value = bench.weak_scaling_value(32768, ws, slowest)
        results[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_units():
    ws = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.start_processes(_rank_main, args=(ws, port, results), nprocs=ws, join=True, start_method="spawn")
    slowest = 10.0 + 5.0 * (ws - 1)
    for rank in range(ws):
        got_ms, got_value = results[rank]
        assert got_ms == slowest
        assert got_value == pytest.approx(32768 * ws / (slowest / 1e3))


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.weak_scaling_value(1000, 1, 2.0) == pytest.approx(5e5)
