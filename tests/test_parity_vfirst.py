"""GPU tests of V-first states ("Hyper-Parallel Chunk KDA current
implementation design" section 4.1, state_v_first: the caller's states are
[.., dv, dk]).  The library converts at the boundary, so every result must be
the K-first result transposed, bit for bit; one case per call is also checked
against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import KdaConfig, make_cotangents
from kda_testutil import check, fwd_kwargs, gpu_fwd, make, oracle_problem, to_cuda

pytestmark = pytest.mark.gpu

T_ = lambda x: x.transpose(-1, -2).contiguous()


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("f32", 64, 128), ("bf16", 128, 64)])
def test_forward_v_first_is_the_transpose(cuda_lib, dtype, dk, dv):
    cfg = KdaConfig("vf", B=2, T=200, H=3, dk=dk, dv=dv, dtype=dtype, initial_state=True,
                    use_exp2=True, seed=dk + dv)
    inp_c = make(cfg)
    inp = to_cuda(inp_c)
    nch = 2 * 4
    h_k = torch.empty(nch, 3, dk, dv, device="cuda")
    out_k, fin_k = gpu_fwd(cuda_lib, cfg, inp, h_out=h_k)
    h_v = torch.empty(nch, 3, dv, dk, device="cuda")
    kw = fwd_kwargs(cfg, inp)
    kw["initial_state"] = T_(inp["initial_state"])
    out_v, fin_v = cuda_lib.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                          state_v_first=True, h_out=h_v, **kw)
    torch.cuda.synchronize()
    assert fin_v.shape == (2, 3, dv, dk)
    assert torch.equal(out_v, out_k)
    assert torch.equal(fin_v, T_(fin_k))
    assert torch.equal(h_v, T_(h_k))
    _, f_ref = oracle.chunk_fwd(oracle_problem(cfg, inp_c), inp_c["initial_state"])
    check(T_(fin_v), f_ref, dtype, "final_state")


def test_forward_v_first_varlen_h_out_stays_in_bounds(cuda_lib):
    """Packed sequences: h_out holds exactly the chunks that exist; the
    conversion must not write past them."""
    lens = (1, 64, 0, 65, 130)
    cfg = KdaConfig("vf_varlen", dtype="bf16", H=2, dk=128, dv=128, seq_lens=lens,
                    initial_state=True, seed=4)
    inp = to_cuda(make(cfg))
    nch = sum((n + 63) // 64 for n in lens)
    h_k = torch.empty(nch, 2, 128, 128, device="cuda")
    _, fin_k = gpu_fwd(cuda_lib, cfg, inp, h_out=h_k)
    guard = torch.full((nch + 3, 2, 128, 128), 7.0, device="cuda")
    kw = fwd_kwargs(cfg, inp)
    kw["initial_state"] = T_(inp["initial_state"])
    _, fin_v = cuda_lib.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                      state_v_first=True, h_out=guard[:nch], **kw)
    torch.cuda.synchronize()
    assert torch.equal(fin_v, T_(fin_k))
    assert torch.equal(guard[:nch], T_(h_k))
    assert torch.all(guard[nch:] == 7.0)


def test_host_io_v_first(cuda_lib):
    cfg = KdaConfig("vf_host", B=2, T=1500, H=2, dk=128, dv=128, dtype="bf16", initial_state=True,
                    seed=6)
    inp = to_cuda(make(cfg))
    kw = fwd_kwargs(cfg, inp)
    kw.pop("cu_seqlens")
    kw["initial_state"] = T_(inp["initial_state"])
    o_ref, f_ref = cuda_lib.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                          state_v_first=True, **kw)
    h = {n: inp[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta")}
    out, fin = cuda_lib.kda_chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"],
                                           state_v_first=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out, o_ref.cpu()) and torch.equal(fin, f_ref)


@pytest.mark.parametrize("dtype,dk,dv", [("f32", 64, 128), ("bf16", 128, 128)])
def test_backward_v_first_is_the_transpose(cuda_lib, dtype, dk, dv):
    cfg = KdaConfig("vf_bwd", B=2, T=130, H=2, dk=dk, dv=dv, dtype=dtype, initial_state=True,
                    seed=8)
    inp_c = make(cfg)
    cot_c = make_cotangents(cfg, inp_c)
    inp, cot = to_cuda(inp_c), to_cuda(cot_c)
    kw = fwd_kwargs(cfg, inp)
    gk = cuda_lib.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cot["d_out"],
                                d_final_state=cot["d_final_state"], want_d_initial_state=True, **kw)
    kw["initial_state"] = T_(inp["initial_state"])
    gv = cuda_lib.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cot["d_out"],
                                d_final_state=T_(cot["d_final_state"]), want_d_initial_state=True,
                                state_v_first=True, **kw)
    torch.cuda.synchronize()
    for name in ("dq", "dk", "dv", "dg", "dbeta", "da_log", "ddt_bias"):
        assert torch.equal(gv[name], gk[name]), name
    assert torch.equal(gv["d_initial_state"], T_(gk["d_initial_state"]))
    ref = oracle.chunk_bwd(oracle_problem(cfg, inp_c), inp_c["initial_state"], cot_c["d_out"],
                           cot_c["d_final_state"])
    check(T_(gv["d_initial_state"]), ref["d_initial"], dtype, "d_initial_state")


@pytest.mark.parametrize("pool_dtype", [torch.float32, torch.bfloat16])
def test_decode_v_first_pool(cuda_lib, pool_dtype):
    N, T, H, dk, dv, rows = 3, 2, 2, 128, 64, 5
    cfg = KdaConfig("vf_dec", B=N, T=T, H=H, dk=dk, dv=dv, dtype="bf16", seed=12)
    inp_c = make(cfg)
    gen = torch.Generator().manual_seed(5)
    pool_k = (torch.randn(rows, H, dk, dv, generator=gen) * 0.1).to(pool_dtype).cuda()
    pool_v = T_(pool_k)
    idx = torch.tensor([4, -1, 1], dtype=torch.int32).cuda()
    dev = {n: inp_c[n].cuda() for n in ("q", "k", "v", "g", "beta", "a_log", "dt_bias")}
    kw = dict(scale=dk ** -0.5, a_log=dev["a_log"], dt_bias=dev["dt_bias"], beta_sigmoid=True,
              gate_in_kernel=True)
    o_k = cuda_lib.kda_recurrent_step(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], pool_k,
                                      idx, **kw)
    o_v = cuda_lib.kda_recurrent_step(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], pool_v,
                                      idx, state_v_first=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o_v, o_k)
    assert torch.equal(pool_v, T_(pool_k))
