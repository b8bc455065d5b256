"""Heads of 64 channels with bf16 inputs on the tensor-core kernels.

The library runs its 128-wide kernels on zero-padded copies of the narrow
tensors (a padded key channel: zero q and k, no decay; a padded value
channel: zero v) and cuts the outputs back.  Two kinds of check:
- the plumbing, bit for bit: the same problem padded here by hand and run at
  d = 128 goes through the same kernels on the same data, so every output
  (o, final state, h_out, v_new_out, M, S~, E, every gradient) must equal
  the narrow call's exactly, including the states of packed sequences, whose
  count the library reads on the device;
- the numerics, against the fp64 oracle: ordinary and strongly decaying
  gates, segment mode with the prepared chunks reused.
The ragged, packed-sequence, V-first and backward parity files cover further
narrow-head shapes against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import KdaConfig, make_cotangents
from kda_testutil import check, fwd_kwargs, make, oracle_problem, to_cuda

pytestmark = pytest.mark.gpu

NARROW = [(64, 64), (64, 128), (128, 64)]


def _widen(x, fill=0.0):
    """Last dimension padded to 128 with `fill`."""
    if x is None or x.shape[-1] == 128:
        return x
    pad = torch.full((*x.shape[:-1], 128 - x.shape[-1]), fill, dtype=x.dtype, device=x.device)
    return torch.cat([x, pad], dim=-1).contiguous()


def _widen_state(S):
    if S is None:
        return None
    out = torch.zeros(*S.shape[:-2], 128, 128, dtype=S.dtype, device=S.device)
    out[..., :S.shape[-2], :S.shape[-1]] = S
    return out


def _wide_inputs(cfg, inp):
    """The problem at d = 128: a padded channel has no decay (raw gate input
    -1e30 through the in-kernel softplus, else a zero log-decay)."""
    w = dict(inp)
    for n in ("q", "k", "v"):
        w[n] = _widen(inp[n])
    w["g"] = _widen(inp["g"], -1e30 if cfg.gate_in_kernel else 0.0)
    w["dt_bias"] = _widen(inp["dt_bias"])
    w["initial_state"] = _widen_state(inp["initial_state"])
    return w


def _nchunks(cfg):
    lens = cfg.seq_lens if cfg.seq_lens else (cfg.T,) * cfg.B
    return sum((n + 63) // 64 for n in lens)


@pytest.mark.parametrize("dk,dv", NARROW)
@pytest.mark.parametrize("gate", [True, False])
def test_fwd_equals_padded_wide_bitwise(cuda_lib, dk, dv, gate):
    cfg = KdaConfig("narrow", dtype="bf16", H=2, dk=dk, dv=dv, seq_lens=(1, 64, 0, 65, 200, 3),
                    initial_state=True, gate_in_kernel=gate, use_exp2=gate, seed=dk + dv + gate)
    inp = to_cuda(make(cfg))
    win = _wide_inputs(cfg, inp)
    nch, H, T = _nchunks(cfg), cfg.H, inp["q"].shape[0]
    h_n = torch.full((nch, H, dk, dv), float("nan"), device="cuda")
    h_w = torch.full((nch, H, 128, 128), float("nan"), device="cuda")
    vn_n = torch.empty(T, H, dv, device="cuda")
    vn_w = torch.empty(T, H, 128, device="cuda")
    o_n, f_n = cuda_lib.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                      h_out=h_n, v_new_out=vn_n, **fwd_kwargs(cfg, inp))
    # the same scale: the narrow problem's
    o_w, f_w = cuda_lib.kda_chunk_fwd(win["q"], win["k"], win["v"], win["g"], win["beta"],
                                      h_out=h_w, v_new_out=vn_w, **fwd_kwargs(cfg, win))
    torch.cuda.synchronize()
    assert torch.equal(o_n, o_w[..., :dv])
    assert torch.equal(f_n, f_w[..., :dk, :dv])
    assert torch.equal(h_n, h_w[..., :dk, :dv])  # every chunk written, none past the count
    assert torch.equal(vn_n, vn_w[..., :dv])
    # padded outputs stay zero: the padded state rows and columns never move
    assert torch.count_nonzero(f_w[..., dk:, :]) == 0 and torch.count_nonzero(f_w[..., :, dv:]) == 0
    assert torch.count_nonzero(o_w[..., dv:]) == 0


@pytest.mark.parametrize("dk,dv", NARROW)
def test_stages_are_the_tensor_core_ones(cuda_lib, dk, dv):
    cfg = KdaConfig("stages", B=1, T=130, H=2, dk=dk, dv=dv, dtype="bf16", initial_state=True)
    inp = to_cuda(make(cfg))
    fa, _, _, _ = cuda_lib.prepare_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                            **fwd_kwargs(cfg, inp))
    assert cuda_lib.kda_chunk_fwd_stages(fa) == ["tc_prep", "tc_chain"]


@pytest.mark.parametrize("dk,dv", NARROW)
def test_summary_and_segment_bwd_equal_padded_wide_bitwise(cuda_lib, dk, dv):
    cfg = KdaConfig("narrow_seg", B=1, T=333, H=2, dk=dk, dv=dv, dtype="bf16", use_exp2=True, seed=7)
    inp = to_cuda(make(cfg))
    cot = to_cuda(make_cotangents(cfg, make(cfg)))
    win = _wide_inputs(cfg, inp)
    sb = torch.tensor((0, 64, 100, 200, 333), dtype=torch.int32, device="cuda")
    flat = lambda x: x.reshape(cfg.T, *x.shape[2:]).contiguous()
    res = []
    for x, d_out in ((inp, cot["d_out"]), (win, _widen(cot["d_out"]))):
        kw = fwd_kwargs(cfg, x)
        kw.pop("initial_state")
        kw.pop("cu_seqlens")
        args = [flat(x[n]) for n in ("q", "k", "v", "g", "beta")]
        M, St = cuda_lib.kda_segment_summary(*args, sb, **kw)
        E = cuda_lib.kda_segment_bwd_summary(*args, flat(d_out), sb, **kw)
        res.append((M, St, E))
    torch.cuda.synchronize()
    (M_n, St_n, E_n), (M_w, St_w, E_w) = res
    assert torch.equal(M_n, M_w[..., :dk, :dk])
    assert torch.equal(St_n, St_w[..., :dk, :dv])
    assert torch.equal(E_n, E_w[..., :dk, :dv])
    # the padded key channels carry the identity in M (no decay, zero keys)
    eye = torch.eye(128 - dk, device="cuda").expand(M_w.shape[0], cfg.H, -1, -1)
    assert torch.equal(M_w[..., dk:, dk:], eye)


@pytest.mark.parametrize("dk,dv", NARROW)
def test_bwd_equals_padded_wide_bitwise(cuda_lib, dk, dv):
    cfg = KdaConfig("narrow_bwd", dtype="bf16", H=2, dk=dk, dv=dv, seq_lens=(65, 1, 130),
                    initial_state=True, seed=dk * 3 + dv)
    inp_c = make(cfg)
    inp = to_cuda(inp_c)
    cot = to_cuda(make_cotangents(cfg, inp_c))
    win = _wide_inputs(cfg, inp)
    res = []
    for x, d_out, d_fin in ((inp, cot["d_out"], cot["d_final_state"]),
                            (win, _widen(cot["d_out"]), _widen_state(cot["d_final_state"]))):
        res.append(cuda_lib.kda_chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], d_out,
                                          d_final_state=d_fin, want_d_initial_state=True,
                                          **fwd_kwargs(cfg, x)))
    torch.cuda.synchronize()
    n, w = res
    assert torch.equal(n["dq"], w["dq"][..., :dk])
    assert torch.equal(n["dk"], w["dk"][..., :dk])
    assert torch.equal(n["dv"], w["dv"][..., :dv])
    assert torch.equal(n["dg"], w["dg"][..., :dk])
    assert torch.equal(n["dbeta"], w["dbeta"])
    assert torch.equal(n["da_log"], w["da_log"])
    assert torch.equal(n["ddt_bias"], w["ddt_bias"][..., :dk])
    assert torch.equal(n["d_initial_state"], w["d_initial_state"][..., :dk, :dv])


@pytest.mark.parametrize("dk,dv", NARROW)
def test_fwd_strong_decay_narrow_heads(cuda_lib, dk, dv):
    """a_log ~ U(1, 3): the exact strong-decay paths with padded channels
    that do not decay at all."""
    cfg = KdaConfig("narrow_strong", B=1, T=200, H=2, dk=dk, dv=dv, dtype="bf16", use_exp2=True,
                    initial_state=True, a_log_range=(1.0, 3.0), seed=5)
    inp_c = make(cfg)
    out, fin = cuda_lib.kda_chunk_fwd(*(to_cuda(inp_c)[n] for n in ("q", "k", "v", "g", "beta")),
                                      **fwd_kwargs(cfg, to_cuda(inp_c)))
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(cfg, inp_c), inp_c["initial_state"])
    check(out.reshape(o_ref.shape), o_ref, "bf16", "o")
    check(fin, f_ref, "bf16", "final_state")


@pytest.mark.parametrize("dk,dv", NARROW)
def test_segment_mode_reusing_prepared_chunks(cuda_lib, dk, dv):
    """Summary -> scan -> finish with KDA_REUSE_PREP on the summary's
    workspace: equal to recomputing the chunks, and to the oracle."""
    import ctypes
    cfg = KdaConfig("narrow_reuse", B=1, T=700, H=2, dk=dk, dv=dv, dtype="bf16", use_exp2=True,
                    seed=13)
    inp_c = make(cfg)
    inp = to_cuda(inp_c)
    bounds = (0, 64, 300, 333, 700)
    sb = torch.tensor(bounds, dtype=torch.int32, device="cuda")
    kw = fwd_kwargs(cfg, inp)
    for key in ("initial_state", "cu_seqlens"):
        kw.pop(key)
    flat = lambda x: x.reshape(cfg.T, *x.shape[2:]).contiguous()
    q, k, v, g, b = (flat(inp[n]) for n in ("q", "k", "v", "g", "beta"))
    a, M, St, ws = cuda_lib.prepare_segment_summary(q, k, v, g, b, sb, **kw)
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
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(cfg, inp_c), None)
    check(o2, o_ref.reshape(cfg.T, cfg.H, dv), "bf16", "segment-mode o")
    check(f2[-1], f_ref[0], "bf16", "segment-mode final state")
