"""GPU parity of the segment affine summary, the ordered prefix scan and
segment-mode processing (summary -> scan -> finish) against the fp64 oracle
and against the unsplit forward."""
import numpy as np
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import CONFIGS, KdaConfig
from kda_testutil import (check, cpu, fwd_kwargs, gpu_fwd, make, oracle_problem, rel_l2, scale_of,
                          to_cuda)

pytestmark = pytest.mark.gpu


def _summary(kda, cfg, inp, bounds):
    kw = fwd_kwargs(cfg, inp)
    for key in ("initial_state", "cu_seqlens"):
        kw.pop(key)
    sb = torch.tensor(bounds, dtype=torch.int32, device="cuda")
    M, St = kda.kda_segment_summary(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], sb, **kw)
    torch.cuda.synchronize()
    return M, St


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("bounds", [(0, 64, 100, 200, 333), (0, 1, 333), (0, 333)])
def test_summary_scan_finish_small(cuda_lib, dtype, bounds):
    cfg = KdaConfig("seg", B=1, T=333, H=2, dk=128, dv=128, dtype=dtype, use_exp2=True,
                    initial_state=True, seed=11)
    inp_c = make(cfg)
    inp = to_cuda(inp_c)
    M, St = _summary(cuda_lib, cfg, inp, bounds)
    p = oracle_problem(cfg, inp_c)
    M_ref, St_ref = oracle.segment_summary(p, bounds)
    check(M, M_ref, dtype, "M")
    check(St, St_ref, dtype, "S_tilde")
    # scan of the GPU summaries, seeded with the initial state
    S0 = inp["initial_state"][0]
    S_in, S_fin = cuda_lib.kda_state_prefix_scan(M, St, S0)
    Si_ref, Sf_ref = oracle.state_prefix_scan(M_ref, St_ref, inp_c["initial_state"][0])
    o_ref, f_ref = oracle.chunk_fwd(p, inp_c["initial_state"])
    check(S_fin, f_ref[0], dtype, "scanned final state")
    check(S_in, Si_ref, dtype, "S_in")
    # finish: every segment as its own sequence, started from its S_in
    sb = torch.tensor(bounds, dtype=torch.int32, device="cuda")
    T = cfg.T
    flat = lambda x: x.reshape(T, *x.shape[2:])
    out, fin = cuda_lib.kda_chunk_fwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]),
                                      flat(inp["g"]), flat(inp["beta"]),
                                      **{**fwd_kwargs(cfg, inp), "cu_seqlens": sb,
                                         "initial_state": S_in.contiguous()})
    check(out, o_ref.reshape(T, cfg.H, cfg.dv), dtype, "segment-mode o")
    check(fin[-1], f_ref[0], dtype, "segment-mode final")


def test_scan_matches_oracle_exactly_in_fp32(cuda_lib):
    """Scan alone on random contractive summaries: 2 chains x 5 segments."""
    rng = np.random.default_rng(2)
    C, S, H, K, V = 2, 5, 3, 128, 64
    M = rng.standard_normal((C, S, H, K, K)) / (2.5 * np.sqrt(K))
    St = rng.standard_normal((C, S, H, K, V))
    S0 = rng.standard_normal((C, H, K, V))
    Mt, Stt, S0t = (torch.tensor(x, dtype=torch.float32, device="cuda") for x in (M, St, S0))
    S_in, S_fin = cuda_lib.kda_state_prefix_scan(Mt, Stt, S0t)
    Si_ref, Sf_ref = oracle.state_prefix_scan(Mt.cpu(), Stt.cpu(), S0t.cpu())
    check(S_in, Si_ref, "f32", "S_in")
    check(S_fin, Sf_ref, "f32", "S_final")
    # without S0 the chain starts from zero
    S_in0, _ = cuda_lib.kda_state_prefix_scan(Mt, Stt, None)
    assert torch.count_nonzero(S_in0[:, 0]) == 0


def test_batched_sequences_segments(cuda_lib):
    """BSND with B=2: segments on the flattened token axis, two chains."""
    cfg = KdaConfig("segB", B=2, T=200, H=2, dk=64, dv=128, dtype="bf16", use_exp2=True, seed=4)
    inp_c = make(cfg)
    inp = to_cuda(inp_c)
    bounds = (0, 70, 200, 330, 400)
    M, St = _summary(cuda_lib, cfg, inp, bounds)
    S_in, S_fin = cuda_lib.kda_state_prefix_scan(M.view(2, 2, *M.shape[1:]),
                                                 St.view(2, 2, *St.shape[1:]))
    out, fin = gpu_fwd(cuda_lib, cfg, inp)
    check(S_fin, fin.cpu().double().numpy(), "bf16", "scan final vs unsplit forward")
    p = oracle_problem(cfg, inp_c)
    _, f_ref = oracle.chunk_fwd(p)
    check(S_fin, f_ref, "bf16", "scan final vs oracle")


def _segment_mode(kda, cfg, inp):
    """summary -> scan -> finish over cfg.num_segments equal segments."""
    sb = inp["seg_bounds"]
    M, St = _summary(kda, cfg, inp, sb.tolist())
    S_in, S_fin = kda.kda_state_prefix_scan(M, St, None)
    T = cfg.T
    flat = lambda x: x.reshape(T, *x.shape[2:])
    kw = {**fwd_kwargs(cfg, inp), "cu_seqlens": sb, "initial_state": S_in.contiguous()}
    out, fin = kda.kda_chunk_fwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]), flat(inp["g"]),
                                 flat(inp["beta"]), **kw)
    torch.cuda.synchronize()
    return M, St, S_in, S_fin, out, fin


def test_slow_decay_segment_workload(cuda_lib):
    """T = 65536, H = 8, 16 segments, slow decay (M stays far from zero):
    summaries of two heads against the oracle; segment mode against the
    unsplit forward on everything."""
    cfg = CONFIGS["long_segment_slow"]
    inp_c = make(cfg)
    inp = to_cuda(inp_c)
    M, St, S_in, S_fin, out, fin = _segment_mode(cuda_lib, cfg, inp)
    o_u, f_u = gpu_fwd(cuda_lib, cfg, inp)
    assert rel_l2(out.float().cpu().numpy(), o_u.reshape(out.shape).float().cpu().numpy()) < 2e-2
    assert rel_l2(S_fin.cpu().numpy(), f_u[0].cpu().numpy()) < 2e-2
    assert float(M.abs().max()) > 0.5   # the transition is not trivially zero
    bounds = inp_c["seg_bounds"].tolist()
    for h in (0, 5):
        sub = dict(inp_c, a_log=inp_c["a_log"][h:h + 1], dt_bias=inp_c["dt_bias"][h:h + 1])
        sl = lambda x: x[:, :, h:h + 1].contiguous()
        p = oracle_problem(cfg, sub, q=sl(inp_c["q"]), k=sl(inp_c["k"]), v=sl(inp_c["v"]),
                           g=sl(inp_c["g"]), beta=sl(inp_c["beta"]), cu=[0, cfg.T])
        M_ref, St_ref = oracle.segment_summary(p, bounds)
        check(M[:, h], M_ref[:, 0], "bf16", f"M[:, {h}]")
        check(St[:, h], St_ref[:, 0], "bf16", f"S_tilde[:, {h}]")
        Si_ref, Sf_ref = oracle.state_prefix_scan(M_ref, St_ref)
        check(S_in[:, h], Si_ref[:, 0], "bf16", f"S_in[:, {h}]")


def test_long_segment_workload(cuda_lib):
    """T = 2^20, H = 8, 16 segments of 65536 ("KDA Context Parallelism (KCP)",
    "L'algorithme"): summary -> scan -> finish on the GPU, and for two heads
    the fp64 oracle's token recurrence over all 2^20 tokens, run segment by
    segment from its own carried state.  Every state entering a segment
    (S_in), every zero-start segment state (S~), the output of every segment
    and the final state are compared element-wise; the segment-mode result
    is also compared with the unsplit GPU forward.  (M itself is a product of
    65536 contractions with decay, zero to far below the tolerance here; it
    acts through S_in[j + 1] = M_j S_in[j] + S~_j, which is checked.)"""
    cfg = CONFIGS["long_segment_bf16"]
    inp = make(cfg, device="cuda")
    M, St, S_in, S_fin, out, fin = _segment_mode(cuda_lib, cfg, inp)
    o_u, f_u = gpu_fwd(cuda_lib, cfg, inp)
    assert rel_l2(out.float().cpu().numpy(), o_u.reshape(out.shape).float().cpu().numpy()) < 2e-2
    assert rel_l2(S_fin.cpu().numpy(), f_u[0].cpu().numpy()) < 2e-2
    heads = [3, 6]
    S, L, T = cfg.num_segments, cfg.T // cfg.num_segments, cfg.T
    out = out.reshape(T, cfg.H, cfg.dv)
    hs = torch.tensor(heads, device="cuda")
    a_log, dt_bias = inp["a_log"][hs].cpu(), inp["dt_bias"][hs].cpu()
    S_prev = np.zeros((1, len(heads), cfg.dk, cfg.dv))
    for j in range(S):
        seg = lambda x: x[0, j * L:(j + 1) * L].index_select(1, hs).cpu()
        # the segment twice: from the carried state (true states and o) and
        # from zero (S~), four independent units for the oracle's threads
        two = {n: torch.cat([seg(inp[n])] * 2) for n in ("q", "k", "v", "g", "beta")}
        sub = dict(a_log=a_log, dt_bias=dt_bias)
        p = oracle_problem(cfg, sub, cu=[0, L, 2 * L], **two)
        o_ref, f_ref = oracle.chunk_fwd(p, np.concatenate([S_prev, np.zeros_like(S_prev)]))
        if j:
            check(S_in[j][hs], S_prev[0], "bf16", f"S_in[{j}]")
        else:  # no initial state: the first segment starts from zero
            np.testing.assert_array_equal(S_in[0].cpu().numpy(), 0.0)
        check(St[j][hs], f_ref[1], "bf16", f"S_tilde[{j}]")
        check(out[j * L:(j + 1) * L].index_select(1, hs), o_ref[:L], "bf16", f"o of segment {j}")
        S_prev = f_ref[:1]
    check(S_fin[hs], S_prev[0], "bf16", "final state")
    check(fin[-1][hs], S_prev[0], "bf16", "final state of the finish")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_segment_finish_reuses_prepared_chunks(cuda_lib, dtype):
    """The finish may reuse the summary's prepared chunks (KDA_REUSE_PREP on
    the summary's workspace); results are identical to recomputing them."""
    cfg = KdaConfig("reuse", B=1, T=700, H=2, dk=128, dv=128, dtype=dtype, use_exp2=True, seed=13)
    inp = to_cuda(make(cfg))
    bounds = (0, 64, 300, 333, 700)
    sb = torch.tensor(bounds, dtype=torch.int32, device="cuda")
    kw = fwd_kwargs(cfg, inp)
    for key in ("initial_state", "cu_seqlens"):
        kw.pop(key)
    T = cfg.T
    flat = lambda x: x.reshape(T, *x.shape[2:])
    q, k, v, g, b = (flat(inp[n]) for n in ("q", "k", "v", "g", "beta"))
    a, M, St, ws = cuda_lib.prepare_segment_summary(q, k, v, g, b, sb, **kw)
    import ctypes
    lib = cuda_lib.load_library()
    assert lib.kda_segment_summary(ctypes.byref(a), sb.data_ptr(), len(bounds) - 1, M.data_ptr(),
                                   St.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    S_in, _ = cuda_lib.kda_state_prefix_scan(M, St, None)
    S_in = S_in.contiguous()
    o1, f1 = cuda_lib.kda_chunk_fwd(q, k, v, g, b, cu_seqlens=sb, initial_state=S_in, **kw)
    o2, f2 = cuda_lib.kda_chunk_fwd(q, k, v, g, b, cu_seqlens=sb, initial_state=S_in,
                                    workspace=ws, reuse_prep=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
