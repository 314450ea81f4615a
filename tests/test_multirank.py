"""The N > 1 path of bench.py (one independent replica per rank, timing
reduced by MAX over ranks) on CPU with two gloo ranks."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, results):
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # rank r timed (r + 1) * 10 ms over 4 steps: the job's figure follows the slowest
        us = bench.per_step_us(10.0 * (rank + 1), 4, world, torch.device("cpu"))
        dist.barrier()
        results[rank] = us
    finally:
        dist.destroy_process_group()


def test_per_step_us_two_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    expect = 20.0 * 1e3 / (4 * world)
    assert got == {0: pytest.approx(expect), 1: pytest.approx(expect)}


def test_per_step_us_single_rank():
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    assert bench.per_step_us(12.5, 5, 1) == pytest.approx(12.5 * 1e3 / 5)
