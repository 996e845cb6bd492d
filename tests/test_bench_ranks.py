"""The multi-rank timing logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py runs one replica per GPU (the path needs no exchange); its only
cross-rank step is taking the slowest rank's time, and the whole-job value
counts every rank's bytes over that time.
"""
import os
import socket

import pytest

import bench

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 7.5][rank]
        out[rank] = bench.max_over_ranks(ms, world)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_every_rank_counts():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 7.5
    # 2 ranks x 1 GB in 7.5 ms -> 0.2667 TB/s for the job
    assert bench.job_tbps(world, 1e9, 7.5e-3) == pytest.approx(2e9 / 7.5e-3 / 1e12)


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(4.25, 1) == 4.25
    assert bench.job_tbps(1, 2e12, 1.0) == 2.0
