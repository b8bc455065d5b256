"""The N > 1 path of bench.py on CPU: two gloo ranks agree on the slowest
rank's time and on the whole-job rate (weak scaling, one scalar all-reduce,
no data-path collective)."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, l = bench.dist_env()
        ms = 10.0 + 5.0 * r                  # rank 1 is the slow one
        slow = bench.max_over_ranks(ms, w, torch.device("cpu"))
        rate = bench.whole_job_rate(1000, w, 4, slow)
        out[r] = (w, r, l, slow, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_rate():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        w, rr, l, slow, rate = out[r]
        assert (w, rr, l) == (2, r, r)
        assert slow == 15.0                   # max over ranks
        assert rate == pytest.approx(1000 * 2 * 4 / 0.015)


def test_single_rank_is_identity(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("LOCAL_RANK", raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
