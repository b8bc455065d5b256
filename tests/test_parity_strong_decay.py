"""GPU parity under strong gate decay, against the fp64 oracle.

"Hyper-Parallel Chunk KDA current implementation design" section 8.2 records
a strong-decay accuracy failure of a chunked KDA backward, and its section 4
gives lower_bound = -5 for the safe_gate option: decays of several nats per
token are a regime the method meets.  The tensor-core path factors each
decay 2^{G_r - G_j} around a reference gate per 16-token sub-block ("KDA Chunk
Backward - TPU/Pallas Kernel Design", section 3.7); when a sub-block decays so
fast that the factors could leave the floating-point range, the prep computes
the at-risk parts (the diagonal blocks, the affected channels' factors) from
exact gate differences, and lists the chunk for the backward's exact pass.
These cases drive that path: a_log ~ U(1, 3), so e^{a_log} is 2.7 to 20 and
the per-token decay runs from about -2 to -60 nats, and hand-built gates with
a cliff inside a sub-block.  Each case first checks on the CPU that it really
contains such sub-blocks."""
import numpy as np
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import KdaConfig, make_cotangents
from kda_testutil import check, fwd_kwargs, gpu_fwd, make, oracle_problem, to_cuda

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634
# sub-blocks whose chunk-local gate moves by more than this (log2 units) take
# the exact paths
STRONG_LOG2 = 96.0
GRADS = ["dq", "dk", "dv", "dg", "dbeta"]


def _strong_and_weak(cfg, inp_c):
    """(#items with a strongly decaying 16-token sub-block, #items without),
    from the oracle's gate: the largest |cumulative gate| inside a sub-block,
    measured from the sub-block's start, per (chunk, head)."""
    p = oracle_problem(cfg, inp_c)
    g = oracle.preprocess(p)[3] * LOG2E  # [T, H, dk], log2 units
    cu = p.cu
    strong = weak = 0
    for n in range(len(cu) - 1):
        for c0 in range(int(cu[n]), int(cu[n + 1]), 64):
            c1 = min(c0 + 64, int(cu[n + 1]))
            worst = np.zeros(g.shape[1])
            for b0 in range(c0, c1, 16):
                blk = np.cumsum(g[b0:min(b0 + 16, c1)], axis=0)
                worst = np.maximum(worst, np.abs(blk).max(axis=(0, 2)))
            strong += int((worst > STRONG_LOG2).sum())
            weak += int((worst <= STRONG_LOG2).sum())
    return strong, weak


def _mixed_channels(inp):
    """dt_bias -8 on even channels (decay ~e^{a_log - 8} per token: weak) and
    +2 on odd ones (strong): the state and the summaries keep the weak
    channels' part while every chunk has strongly decaying sub-blocks."""
    dtb = inp["dt_bias"].clone()
    dtb[:, 0::2] = -8.0
    dtb[:, 1::2] = 2.0
    inp["dt_bias"] = dtb
    return inp


def _fwd_case(cuda_lib, cfg, inp_c, need_weak=False):
    strong, weak = _strong_and_weak(cfg, inp_c)
    assert strong > 0, "case has no strongly decaying sub-block"
    if need_weak:
        assert weak > 0, "case has no ordinary item"
    out, fin = gpu_fwd(cuda_lib, cfg, to_cuda(inp_c))
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(cfg, inp_c), inp_c["initial_state"])
    check(out.reshape(o_ref.shape), o_ref, cfg.dtype, "o")
    check(fin, f_ref, cfg.dtype, "final_state")


@pytest.mark.parametrize("T", [65, 130, 1000])
def test_fwd_strong_decay(cuda_lib, T):
    cfg = KdaConfig("strong", B=2, T=T, H=3, dk=128, dv=128, dtype="bf16", use_exp2=True,
                    initial_state=True, a_log_range=(1.0, 3.0), seed=40 + T)
    _fwd_case(cuda_lib, cfg, make(cfg))


def test_fwd_strong_and_ordinary_items_in_one_call(cuda_lib):
    """Heads with a_log ~ U(-4, 3): listed and ordinary items side by side."""
    cfg = KdaConfig("mixed", B=2, T=640, H=8, dk=128, dv=128, dtype="bf16", use_exp2=True,
                    initial_state=True, a_log_range=(-4.0, 3.0), seed=17)
    _fwd_case(cuda_lib, cfg, make(cfg), need_weak=True)


def test_fwd_strong_decay_channel_mix_varlen(cuda_lib):
    lens = (1, 64, 65, 200, 17, 300)
    cfg = KdaConfig("strong_varlen", dtype="bf16", H=2, dk=128, dv=128, seq_lens=lens,
                    initial_state=True, use_exp2=True, a_log_range=(1.0, 3.0), seed=23)
    _fwd_case(cuda_lib, cfg, _mixed_channels(make(cfg)))


def test_fwd_gate_cliff_inside_a_sub_block(cuda_lib):
    """Precomputed natural-log gate: -0.01 per token except a cliff of -150
    nats at token 2 of every 16-token sub-block on half the channels.  After
    the cliff the decay between two tokens of a sub-block is near zero while
    both lie 216 log2 units below the sub-block's start - the pattern a single
    reference per sub-block cannot represent."""
    cfg = KdaConfig("cliff", B=1, T=200, H=2, dk=128, dv=128, dtype="bf16", gate_in_kernel=False,
                    initial_state=True, seed=31)
    inp = make(cfg)
    g = torch.full_like(inp["g"], -0.01)
    cliff = (torch.arange(cfg.T) % 16) == 2
    g[:, cliff, :, 1::2] = -150.0
    inp["g"] = g
    _fwd_case(cuda_lib, cfg, inp, need_weak=False)


def _chunk_gate_pattern(inp, cfg, kind):
    """Precomputed natural-log gates whose chunk totals are large while the
    16-token sub-blocks stay ordinary, or the other way round:
      near_edge:    -2.05 nats per token on every channel: 189 log2 units per
                    64-token chunk, 47 per sub-block
      past_edge:    -2.2 nats per token: 203 per chunk, 51 per sub-block
      cliff_inside: -0.01 per token and -80 nats at token 5 of every chunk on
                    odd channels: 116 log2 units inside one sub-block (listed
                    for the exact passes) in a chunk that moves little else
      channel_mix:  even channels -2.05 per token, odd channels -2.4"""
    g = torch.full_like(inp["g"], -0.01)
    t = torch.arange(cfg.T)
    if kind == "near_edge":
        g[:] = -2.05
    elif kind == "past_edge":
        g[:] = -2.2
    elif kind == "cliff_inside":
        g[:, (t % 64) == 5, :, 1::2] = -80.0
    elif kind == "channel_mix":
        g[..., 0::2] = -2.05
        g[..., 1::2] = -2.4
    inp["g"] = g
    return inp


def _chunk_moves(cfg, inp_c):
    """Largest move of the gate (log2 units) over any whole chunk, and over
    any 16-token sub-block, from the oracle's gate."""
    p = oracle_problem(cfg, inp_c)
    g = oracle.preprocess(p)[3] * LOG2E
    chunk = sub = 0.0
    for n in range(len(p.cu) - 1):
        for c0 in range(int(p.cu[n]), int(p.cu[n + 1]), 64):
            c1 = min(c0 + 64, int(p.cu[n + 1]))
            chunk = max(chunk, float(np.abs(g[c0:c1].sum(axis=0)).max()))
            for b0 in range(c0, c1, 16):
                sub = max(sub, float(np.abs(g[b0:min(b0 + 16, c1)].sum(axis=0)).max()))
    return chunk, sub


@pytest.mark.parametrize("kind", ["near_edge", "past_edge", "cliff_inside", "channel_mix"])
def test_fwd_large_chunk_decay(cuda_lib, kind):
    cfg = KdaConfig("ref_bound", B=2, T=200, H=2, dk=128, dv=128, dtype="bf16", gate_in_kernel=False,
                    initial_state=True, seed=61)
    inp_c = _chunk_gate_pattern(make(cfg), cfg, kind)
    chunk, sub = _chunk_moves(cfg, inp_c)
    if kind == "cliff_inside":
        assert sub > STRONG_LOG2 and chunk < 120.0, (chunk, sub)
    else:  # large chunk totals from sub-blocks that stay ordinary
        assert chunk > 180.0 and sub <= STRONG_LOG2, (chunk, sub)
    out, fin = gpu_fwd(cuda_lib, cfg, to_cuda(inp_c))
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(cfg, inp_c), inp_c["initial_state"])
    check(out.reshape(o_ref.shape), o_ref, cfg.dtype, "o")
    check(fin, f_ref, cfg.dtype, "final_state")


@pytest.mark.parametrize("kind", ["near_edge", "cliff_inside"])
def test_bwd_large_chunk_decay(cuda_lib, kind):
    """Backward on the same gate patterns: the cliff case's chunks go through
    the backward's exact pass."""
    cfg = KdaConfig("ref_bound_bwd", B=1, T=150, H=2, dk=128, dv=128, dtype="bf16",
                    gate_in_kernel=False, initial_state=True, seed=62)
    inp_c = _chunk_gate_pattern(make(cfg), cfg, kind)
    cot = make_cotangents(cfg, inp_c)
    inp = to_cuda(inp_c)
    got = cuda_lib.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                 cot["d_out"].cuda(), d_final_state=cot["d_final_state"].cuda(),
                                 want_d_initial_state=True, **fwd_kwargs(cfg, inp))
    torch.cuda.synchronize()
    ref = oracle.chunk_bwd(oracle_problem(cfg, inp_c), inp_c["initial_state"], cot["d_out"],
                           cot["d_final_state"])
    for name in GRADS:
        check(got[name].reshape(ref[name].shape), ref[name], "bf16", name)
    check(got["d_initial_state"], ref["d_initial"], "bf16", "d_initial_state")


def test_summary_scan_strong_decay(cuda_lib):
    cfg = KdaConfig("strong_seg", B=1, T=333, H=2, dk=128, dv=128, dtype="bf16", use_exp2=True,
                    initial_state=True, a_log_range=(1.0, 3.0), seed=12)
    inp_c = _mixed_channels(make(cfg))
    assert _strong_and_weak(cfg, inp_c)[0] > 0
    inp = to_cuda(inp_c)
    bounds = (0, 64, 100, 200, 333)
    kw = fwd_kwargs(cfg, inp)
    for key in ("initial_state", "cu_seqlens"):
        kw.pop(key)
    sb = torch.tensor(bounds, dtype=torch.int32, device="cuda")
    M, St = cuda_lib.kda_segment_summary(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], sb, **kw)
    torch.cuda.synchronize()
    p = oracle_problem(cfg, inp_c)
    M_ref, St_ref = oracle.segment_summary(p, bounds)
    check(M, M_ref, "bf16", "M")
    check(St, St_ref, "bf16", "S_tilde")
    S_in, S_fin = cuda_lib.kda_state_prefix_scan(M, St, inp["initial_state"][0])
    Si_ref, _ = oracle.state_prefix_scan(M_ref, St_ref, inp_c["initial_state"][0])
    _, f_ref = oracle.chunk_fwd(p, inp_c["initial_state"])
    check(S_in, Si_ref, "bf16", "S_in")
    check(S_fin, f_ref[0], "bf16", "scanned final state")


@pytest.mark.parametrize("case", ["a_log U(1,3)", "channel mix, varlen"])
def test_bwd_strong_decay(cuda_lib, case):
    if case == "a_log U(1,3)":
        cfg = KdaConfig("strong_bwd", B=2, T=130, H=2, dk=128, dv=128, dtype="bf16", use_exp2=True,
                        initial_state=True, a_log_range=(1.0, 3.0), seed=5)
        inp_c = make(cfg)
    else:
        cfg = KdaConfig("strong_bwd_varlen", dtype="bf16", H=2, dk=128, dv=128,
                        seq_lens=(65, 1, 200, 64), initial_state=True, use_exp2=True,
                        a_log_range=(1.0, 3.0), seed=6)
        inp_c = _mixed_channels(make(cfg))
    assert _strong_and_weak(cfg, inp_c)[0] > 0
    cot = make_cotangents(cfg, inp_c)
    inp = to_cuda(inp_c)
    got = cuda_lib.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                 cot["d_out"].cuda(), d_final_state=cot["d_final_state"].cuda(),
                                 want_d_initial_state=True, **fwd_kwargs(cfg, inp))
    torch.cuda.synchronize()
    ref = oracle.chunk_bwd(oracle_problem(cfg, inp_c), inp_c["initial_state"], cot["d_out"],
                           cot["d_final_state"])
    for name in GRADS:
        check(got[name].reshape(ref[name].shape), ref[name], "bf16", name)
    check(got["d_initial_state"], ref["d_initial"], "bf16", "d_initial_state")
    check(got["da_log"], ref["da_log"], "bf16", "da_log")
    check(got["ddt_bias"], ref["ddt_bias"], "bf16", "ddt_bias")
