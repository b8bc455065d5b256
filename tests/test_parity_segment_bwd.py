"""GPU parity of the backward segment path: the backward segment summary E
(the local state gradient of each segment), the reverse-order state-gradient
scan, and segment-mode backward (forward summary -> scan -> backward summary
-> reverse scan -> per-segment kda_chunk_bwd), against the fp64 oracle and
against the unsplit backward."""
import numpy as np
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import CONFIGS, KdaConfig, make_cotangents
from kda_testutil import check, fwd_kwargs, make, oracle_problem, rel_l2, to_cuda

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg", "dbeta", "da_log", "ddt_bias")


def _flat(x, T):
    return x.reshape(T, *x.shape[2:]).contiguous()


def _segment_mode_bwd(kda, cfg, inp, cot, bounds):
    """Returns (E, dS_out, dS0, grads) of segment-mode backward on GPU for a
    one-sequence batch (B = 1)."""
    T = cfg.T
    kw = fwd_kwargs(cfg, inp)
    kw.pop("initial_state")
    kw.pop("cu_seqlens")
    sb = torch.tensor(bounds, dtype=torch.int32, device="cuda")
    q, k, v, g, be = (_flat(inp[n], T) for n in ("q", "k", "v", "g", "beta"))
    dO = _flat(cot["d_out"], T)
    M, St = kda.kda_segment_summary(q, k, v, g, be, sb, **kw)
    S0 = inp["initial_state"][0] if inp["initial_state"] is not None else None
    S_in, _ = kda.kda_state_prefix_scan(M, St, S0)
    E = kda.kda_segment_bwd_summary(q, k, v, g, be, dO, sb, **kw)
    dS_out, dS0 = kda.kda_state_grad_scan(M, E, cot["d_final_state"][0])
    grads = kda.kda_chunk_bwd(q, k, v, g, be, dO, d_final_state=dS_out.contiguous(),
                              initial_state=S_in.contiguous(), cu_seqlens=sb,
                              want_d_initial_state=True, **kw)
    torch.cuda.synchronize()
    return M, E, dS_out, dS0, grads


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
@pytest.mark.parametrize("bounds", [(0, 64, 100, 200, 333), (0, 1, 333), (0, 333)])
def test_segment_backward_small(cuda_lib, dtype, d, bounds):
    cfg = KdaConfig("segbwd", B=1, T=333, H=2, dk=d, dv=d, dtype=dtype, use_exp2=True,
                    initial_state=True, seed=11)
    inp_c = make(cfg)
    cot_c = make_cotangents(cfg, inp_c)
    M, E, dS_out, dS0, grads = _segment_mode_bwd(cuda_lib, cfg, to_cuda(inp_c), to_cuda(cot_c), bounds)
    p = oracle_problem(cfg, inp_c)
    do = cot_c["d_out"].reshape(cfg.T, cfg.H, cfg.dv)
    E_ref = oracle.segment_bwd_summary(p, bounds, do)
    check(E, E_ref, dtype, "E")
    M_ref, _ = oracle.segment_summary(p, bounds)
    dS_out_ref, dS0_ref = oracle.state_grad_scan(M_ref, E_ref, cot_c["d_final_state"][0])
    check(dS_out, dS_out_ref, dtype, "dS_out")
    whole = oracle.chunk_bwd(p, inp_c["initial_state"], do, cot_c["d_final_state"])
    check(dS0, whole["d_initial"][0], dtype, "scanned initial-state gradient")
    for name in GRADS:
        check(grads[name].reshape(whole[name].shape), whole[name], dtype, f"segment-mode {name}")
    # the first segment's entering-state gradient is the whole initial-state gradient
    check(grads["d_initial_state"][0], whole["d_initial"][0], dtype, "segment 0 d_initial")


def test_grad_scan_matches_oracle_in_fp32(cuda_lib):
    """Reverse scan alone on random contractive transitions: 2 chains x 5 segments."""
    rng = np.random.default_rng(4)
    C, S, H, K, V = 2, 5, 3, 128, 64
    M = rng.standard_normal((C, S, H, K, K)) * (0.9 / np.sqrt(K))
    E = rng.standard_normal((C, S, H, K, V))
    g = rng.standard_normal((C, H, K, V))
    t = lambda x: torch.tensor(x, dtype=torch.float32, device="cuda")
    dS_out, dS0 = cuda_lib.kda_state_grad_scan(t(M), t(E), t(g))
    torch.cuda.synchronize()
    ref_out, ref0 = oracle.state_grad_scan(t(M).cpu(), t(E).cpu(), t(g).cpu())
    check(dS_out, ref_out, "f32", "dS_out")
    check(dS0, ref0, "f32", "dS_initial")


def test_segment_backward_slow_decay_workload(cuda_lib):
    """T = 65536, H = 8, 16 segments, slow decay (M far from zero): the
    segment-mode backward equals the unsplit backward (itself checked against
    the oracle); the per-segment E equals the oracle's on two segments of one
    head."""
    cfg = CONFIGS["long_segment_slow"]
    inp_c = make(cfg)
    cot_c = make_cotangents(cfg, inp_c)
    inp, cot = to_cuda(inp_c), to_cuda(cot_c)
    bounds = [int(x) for x in inp_c["seg_bounds"]]
    M, E, dS_out, dS0, seg = _segment_mode_bwd(cuda_lib, cfg, inp, cot, bounds)
    kw = fwd_kwargs(cfg, inp)
    whole = cuda_lib.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                   cot["d_out"], d_final_state=cot["d_final_state"],
                                   want_d_initial_state=True, **kw)
    torch.cuda.synchronize()
    for name in GRADS:
        e = rel_l2(seg[name].reshape(whole[name].shape).float().cpu().numpy(),
                   whole[name].float().cpu().numpy())
        assert e <= 2e-2, f"segment-mode {name}: rel L2 {e:.3e}"
    e = rel_l2(dS0.cpu().numpy(), whole["d_initial_state"][0].cpu().numpy())
    assert e <= 2e-2, f"initial-state gradient: rel L2 {e:.3e}"
    # M is far from zero here, so the scan really composes
    assert float(M.abs().max()) > 0.5
    h = 3
    for s in (0, 15):
        a, b = bounds[s], bounds[s + 1]
        sub = dict(inp_c)
        for n in ("q", "k", "v", "g", "beta"):
            sub[n] = inp_c[n][:, a:b, h:h + 1].contiguous()
        sub["a_log"] = inp_c["a_log"][h:h + 1]
        sub["dt_bias"] = inp_c["dt_bias"][h:h + 1]
        c = cfg.replace(T=b - a, H=1)
        p = oracle_problem(c, sub)
        E_ref = oracle.segment_bwd_summary(p, [0, b - a],
                                           cot_c["d_out"][:, a:b, h:h + 1].reshape(b - a, 1, cfg.dv))
        check(E[s, h:h + 1], E_ref[0], "bf16", f"E segment {s}")
