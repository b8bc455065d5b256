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


def _replica_main(rank, world, port, out):
    """One weak-scaling replica: this rank's own batch (the bench's per-rank
    draw) through the fp64 oracle as the step, on CPU."""
    import numpy as np
    import oracle
    from chunked_kimi_delta_gb300.inputs import KdaConfig, oracle_kwargs
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = KdaConfig("replica", B=1, T=70, H=2, dk=16, dv=16, dtype="f32", initial_state=True)
        inp = bench.rank_inputs(cfg, "cpu", rank)
        p = oracle.Problem(inp["q"][0], inp["k"][0], inp["v"][0], inp["g"][0], inp["beta"][0],
                           cu_seqlens=[0, cfg.T], scale=cfg.dk ** -0.5, a_log=inp["a_log"],
                           dt_bias=inp["dt_bias"], **oracle_kwargs(cfg))
        o, fin = oracle.chunk_fwd(p, inp["initial_state"])
        sums = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sums, torch.tensor([float(inp["q"].double().sum())], dtype=torch.float64))
        slow = bench.max_over_ranks(1.0 + rank, world, torch.device("cpu"))
        out[rank] = (np.asarray(o).copy(), [float(x) for x in sums], slow)
    finally:
        dist.destroy_process_group()


def test_replicas_draw_their_own_batches_and_run_independently():
    """Each rank processes its own batch (seeded by its rank) with no
    data-path collective: the inputs differ across ranks, each rank's result
    equals a single-process run on that rank's batch, and the time is the
    slowest rank's."""
    import numpy as np
    import oracle
    from chunked_kimi_delta_gb300.inputs import KdaConfig, oracle_kwargs
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_replica_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    cfg = KdaConfig("replica", B=1, T=70, H=2, dk=16, dv=16, dtype="f32", initial_state=True)
    o0, sums0, slow0 = out[0]
    o1, sums1, slow1 = out[1]
    assert sums0 == sums1 and sums0[0] != sums0[1]      # every rank sees both; they differ
    assert slow0 == slow1 == 2.0
    for r, o in ((0, o0), (1, o1)):
        inp = bench.rank_inputs(cfg, "cpu", r)
        p = oracle.Problem(inp["q"][0], inp["k"][0], inp["v"][0], inp["g"][0], inp["beta"][0],
                           cu_seqlens=[0, cfg.T], scale=cfg.dk ** -0.5, a_log=inp["a_log"],
                           dt_bias=inp["dt_bias"], **oracle_kwargs(cfg))
        ref, _ = oracle.chunk_fwd(p, inp["initial_state"])
        np.testing.assert_array_equal(o, ref)
    assert not np.allclose(o0, o1)
