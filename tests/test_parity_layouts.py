"""GPU tests of the head-major token layouts ("Hyper-Parallel Chunk KDA
current implementation design" section 4.2: BNSD [B, H, T, D] and NTD
[H, T_total, D] beside BSND / TND).  The library converts at the boundary,
so every result must equal the token-major result in the other layout, bit
for bit; one case is also checked against the oracle."""
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import KdaConfig, make_cotangents
from kda_testutil import check, fwd_kwargs, gpu_fwd, make, oracle_problem, rel_l2, to_cuda

pytestmark = pytest.mark.gpu


def to_hm(x, varlen):
    ax = 0 if varlen else 1
    return x.transpose(ax, ax + 1).contiguous()


def _hm_inputs(inp, varlen):
    out = dict(inp)
    for n in ("q", "k", "v", "g", "beta"):
        out[n] = to_hm(inp[n], varlen)
    return out


@pytest.mark.parametrize("dtype,dk,dv,Hk", [("bf16", 128, 128, 4), ("f32", 64, 128, 4),
                                            ("bf16", 128, 128, 2)])
def test_forward_head_major(cuda_lib, dtype, dk, dv, Hk):
    cfg = KdaConfig("hm", B=2, T=150, H=4, dk=dk, dv=dv, dtype=dtype, initial_state=True,
                    use_exp2=True, seed=dk + Hk)
    inp = to_cuda(make(cfg))
    for n in ("q", "k"):
        inp[n] = inp[n][:, :, :Hk].contiguous()
    o_t, f_t = gpu_fwd(cuda_lib, cfg, inp)
    h = _hm_inputs(inp, False)
    kw = fwd_kwargs(cfg, inp)
    o_h, f_h = cuda_lib.kda_chunk_fwd(h["q"], h["k"], h["v"], h["g"], h["beta"], head_major=True,
                                      **kw)
    torch.cuda.synchronize()
    assert o_h.shape == (2, 4, 150, dv)
    assert torch.equal(o_h, to_hm(o_t, False))
    assert torch.equal(f_h, f_t)


def test_forward_head_major_varlen_with_saves(cuda_lib):
    """NTD [H, T_total, D] with cu_seqlens; v_new_out head-major too, h_out
    and states unchanged; V-first states on top."""
    lens = (1, 64, 0, 65, 130)
    cfg = KdaConfig("hm_varlen", dtype="bf16", H=2, dk=128, dv=128, seq_lens=lens,
                    initial_state=True, seed=4)
    inp_c = make(cfg)
    inp = to_cuda(inp_c)
    T = sum(lens)
    nch = sum((n + 63) // 64 for n in lens)
    vn_t = torch.empty(T, 2, 128, device="cuda")
    h_t = torch.empty(nch, 2, 128, 128, device="cuda")
    o_t, f_t = gpu_fwd(cuda_lib, cfg, inp, v_new_out=vn_t, h_out=h_t)
    h = _hm_inputs(inp, True)
    kw = fwd_kwargs(cfg, inp)
    kw["initial_state"] = inp["initial_state"].transpose(-1, -2).contiguous()
    vn_h = torch.empty(2, T, 128, device="cuda")
    h_h = torch.empty(nch, 2, 128, 128, device="cuda")
    o_h, f_h = cuda_lib.kda_chunk_fwd(h["q"], h["k"], h["v"], h["g"], h["beta"], head_major=True,
                                      state_v_first=True, v_new_out=vn_h, h_out=h_h, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o_h, to_hm(o_t, True))
    assert torch.equal(vn_h, to_hm(vn_t, True))
    assert torch.equal(f_h, f_t.transpose(-1, -2))
    assert torch.equal(h_h, h_t.transpose(-1, -2))
    _, f_ref = oracle.chunk_fwd(oracle_problem(cfg, inp_c), inp_c["initial_state"])
    check(f_h.transpose(-1, -2), f_ref, "bf16", "final_state")


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_backward_head_major(cuda_lib, dtype, d):
    cfg = KdaConfig("hm_bwd", B=2, T=130, H=2, dk=d, dv=d, dtype=dtype, initial_state=True,
                    seed=8)
    inp_c = make(cfg)
    cot_c = make_cotangents(cfg, inp_c)
    inp, cot = to_cuda(inp_c), to_cuda(cot_c)
    kw = fwd_kwargs(cfg, inp)
    gt = cuda_lib.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cot["d_out"],
                                d_final_state=cot["d_final_state"], want_d_initial_state=True, **kw)
    h = _hm_inputs(inp, False)
    gh = cuda_lib.kda_chunk_bwd(h["q"], h["k"], h["v"], h["g"], h["beta"], to_hm(cot["d_out"], False),
                                d_final_state=cot["d_final_state"], want_d_initial_state=True,
                                head_major=True, **kw)
    torch.cuda.synchronize()
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(gh[name], to_hm(gt[name], False)), name
    for name in ("da_log", "ddt_bias", "d_initial_state"):
        assert torch.equal(gh[name], gt[name]), name


def test_summaries_head_major(cuda_lib):
    bounds = (0, 64, 100, 200, 333)
    cfg = KdaConfig("hm_seg", B=1, T=333, H=2, dk=128, dv=128, dtype="bf16", use_exp2=True, seed=11)
    inp = to_cuda(make(cfg))
    cot = to_cuda(make_cotangents(cfg, inp))
    kw = fwd_kwargs(cfg, inp)
    kw.pop("initial_state")
    kw.pop("cu_seqlens")
    sb = torch.tensor(bounds, dtype=torch.int32, device="cuda")
    M_t, S_t = cuda_lib.kda_segment_summary(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], sb,
                                            **kw)
    E_t = cuda_lib.kda_segment_bwd_summary(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                           cot["d_out"], sb, **kw)
    h = _hm_inputs(inp, False)
    M_h, S_h = cuda_lib.kda_segment_summary(h["q"], h["k"], h["v"], h["g"], h["beta"], sb,
                                            head_major=True, **kw)
    E_h = cuda_lib.kda_segment_bwd_summary(h["q"], h["k"], h["v"], h["g"], h["beta"],
                                           to_hm(cot["d_out"], False), sb, head_major=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(M_h, M_t) and torch.equal(S_h, S_t) and torch.equal(E_h, E_t)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_all_boundary_options_together(cuda_lib, dtype, d):
    """Packed sequences in NTD (head-major) layout, V-first states and two
    key heads for four value heads, forward and backward, against the plain
    token-major K-first run on q/k expanded to the value heads: the
    conversions are exact, so o, the states and every per-value-head gradient
    agree bit for bit; dq, dk agree with the group sums of the expanded run."""
    lens = (1, 64, 0, 65, 130)
    H, Hk = 4, 2
    cfg = KdaConfig("combo", dtype=dtype, H=H, dk=d, dv=d, seq_lens=lens, initial_state=True,
                    seed=23)
    inp = to_cuda(make(cfg))
    cot = to_cuda(make_cotangents(cfg, inp))
    T = sum(lens)
    small, wide = dict(inp), dict(inp)
    for n in ("q", "k"):
        x = inp[n][:, :Hk].contiguous()
        small[n] = x
        wide[n] = x.repeat_interleave(H // Hk, dim=1).contiguous()
    kw = fwd_kwargs(cfg, inp)
    o_w, f_w = cuda_lib.kda_chunk_fwd(wide["q"], wide["k"], wide["v"], wide["g"], wide["beta"], **kw)
    g_w = cuda_lib.kda_chunk_bwd(wide["q"], wide["k"], wide["v"], wide["g"], wide["beta"], cot["d_out"],
                                 d_final_state=cot["d_final_state"], want_d_initial_state=True, **kw)
    hm = {n: to_hm(small[n], True) for n in ("q", "k", "v", "g", "beta")}
    kv = dict(kw)
    kv["initial_state"] = inp["initial_state"].transpose(-1, -2).contiguous()
    o_c, f_c = cuda_lib.kda_chunk_fwd(hm["q"], hm["k"], hm["v"], hm["g"], hm["beta"], head_major=True,
                                      state_v_first=True, **kv)
    g_c = cuda_lib.kda_chunk_bwd(hm["q"], hm["k"], hm["v"], hm["g"], hm["beta"], to_hm(cot["d_out"], True),
                                 d_final_state=cot["d_final_state"].transpose(-1, -2).contiguous(),
                                 want_d_initial_state=True, head_major=True, state_v_first=True, **kv)
    torch.cuda.synchronize()
    assert torch.equal(o_c, to_hm(o_w, True))
    assert torch.equal(f_c, f_w.transpose(-1, -2))
    for name in ("dv", "dg", "dbeta"):
        assert torch.equal(g_c[name], to_hm(g_w[name], True)), name
    for name in ("da_log", "ddt_bias"):
        assert torch.equal(g_c[name], g_w[name]), name
    assert torch.equal(g_c["d_initial_state"], g_w["d_initial_state"].transpose(-1, -2))
    for name in ("dq", "dk"):
        # the library sums the value heads' fp32 gradients and rounds once;
        # the expanded run rounds each head's gradient to the input dtype
        want = g_w[name].float().reshape(T, Hk, H // Hk, d).sum(dim=2)
        got = g_c[name].float().transpose(0, 1)
        if dtype == "bf16":
            assert rel_l2(got.cpu().numpy(), want.cpu().numpy()) <= 1e-2, name
        else:
            torch.testing.assert_close(got, want, rtol=1e-5, atol=1e-5)
