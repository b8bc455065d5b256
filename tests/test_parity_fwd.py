"""GPU parity of kda_chunk_fwd against the fp64 oracle (through the C ABI).

Small cases are compared element by element in full; the full-size
workloads are compared in full where the oracle finishes in seconds (the mid
bf16 batch) and on sampled (sequence, head) units otherwise."""
import numpy as np
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import CONFIGS, KdaConfig
from kda_testutil import (check, cpu, gpu_fwd, make, max_rel, oracle_problem, rel_l2, to_cuda)

pytestmark = pytest.mark.gpu


def _run_both(kda, cfg, inp_cpu, nthreads=0):
    inp = to_cuda(inp_cpu)
    out, fin = gpu_fwd(kda, cfg, inp)
    p = oracle_problem(cfg, inp_cpu)
    o_ref, f_ref = oracle.chunk_fwd(p, inp_cpu["initial_state"], nthreads=nthreads)
    return out, fin, o_ref, f_ref


def test_tiny_f32_workload(cuda_lib):
    cfg = CONFIGS["tiny_f32"]
    inp = make(cfg)
    out, fin, o_ref, f_ref = _run_both(cuda_lib, cfg, inp)
    check(out.reshape(o_ref.shape), o_ref, "f32", "o")
    check(fin, f_ref, "f32", "final_state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 63, 65, 130])
def test_ragged_small(cuda_lib, dtype, dk, dv, T):
    cfg = KdaConfig("ragged", B=2, T=T, H=3, dk=dk, dv=dv, dtype=dtype, initial_state=True,
                    use_exp2=(T % 2 == 1), seed=T + dk)
    inp = make(cfg)
    out, fin, o_ref, f_ref = _run_both(cuda_lib, cfg, inp)
    check(out.reshape(o_ref.shape), o_ref, dtype, "o")
    check(fin, f_ref, dtype, "final_state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_precomputed_gate_and_beta_without_l2norm(cuda_lib, dtype):
    cfg = KdaConfig("pre", B=1, T=200, H=2, dk=128, dv=128, dtype=dtype, gate_in_kernel=False,
                    beta_sigmoid=False, l2norm=False, seed=5)
    inp = make(cfg)
    # unnormalised keys make the delta rule expand: keep them small
    inp["k"] = (inp["k"].float() * 0.08).to(inp["k"].dtype)
    out, fin, o_ref, f_ref = _run_both(cuda_lib, cfg, inp)
    check(out.reshape(o_ref.shape), o_ref, dtype, "o")
    check(fin, f_ref, dtype, "final_state")


@pytest.mark.parametrize("dtype,dv", [("f32", 64), ("bf16", 64), ("bf16", 128)])
def test_varlen_small(cuda_lib, dtype, dv):
    lens = (1, 64, 0, 65, 200, 3)
    cfg = KdaConfig("varlen_small", dtype=dtype, H=2, dk=128, dv=dv, seq_lens=lens,
                    initial_state=True, seed=9)
    inp = make(cfg)
    out, fin, o_ref, f_ref = _run_both(cuda_lib, cfg, inp)
    check(out.reshape(o_ref.shape), o_ref, dtype, "o")
    check(fin, f_ref, dtype, "final_state")
    # an empty sequence hands its initial state through unchanged
    np.testing.assert_array_equal(fin[2].cpu().numpy(), inp["initial_state"][2].numpy())


def test_empty_batch_passes_initial_state_through(cuda_lib):
    cfg = KdaConfig("empty", B=2, T=0, H=2, dk=64, dv=64, dtype="bf16", initial_state=True)
    inp = to_cuda(make(cfg))
    out, fin = gpu_fwd(cuda_lib, cfg, inp)
    assert out.numel() == 0
    torch.testing.assert_close(fin, inp["initial_state"], rtol=0, atol=0)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_h_out_and_v_new_out(cuda_lib, dtype, d):
    """h_out[c] is the state entering chunk c; v_new rows are the corrected
    values beta_r (v_r - (Diag(alpha_r) S_{r-1})^T k_r).  Both are checked
    against oracle runs over every prefix (CUDA-core path for fp32 d=64,
    tensor-core path for bf16 d=128)."""
    cfg = KdaConfig("save", B=1, T=130, H=2, dk=d, dv=d, dtype=dtype, initial_state=True, seed=3)
    inp_cpu = make(cfg)
    inp = to_cuda(inp_cpu)
    T, H, K, V = 130, 2, d, d
    h_out = torch.empty(3, H, K, V, device="cuda")
    vn = torch.empty(1, T, H, V, device="cuda")
    gpu_fwd(cuda_lib, cfg, inp, h_out=h_out, v_new_out=vn)
    p = oracle_problem(cfg, inp_cpu)
    qh, kh, b, g = oracle.preprocess(p)
    S0 = inp_cpu["initial_state"].double().numpy()
    prefix = {}
    for t in range(T + 1):
        if t == 0:
            prefix[0] = S0[0]
        else:
            pt = oracle.Problem(p.q[:t], p.k[:t], p.v[:t], p.g[:t], p.beta[:t], cu_seqlens=[0, t],
                                scale=p.scale, a_log=p.a_log, dt_bias=p.dt_bias,
                                gate_in_kernel=True, beta_sigmoid=True)
            prefix[t] = oracle.chunk_fwd(pt, S0, want_out=False)[1][0]
    for c in range(3):
        check(h_out[c], prefix[64 * c], dtype, f"h_out[{c}]")
    ref = np.zeros((T, H, V))
    for t in range(T):
        for h in range(H):
            Sd = np.exp(g[t, h])[:, None] * prefix[t][h]
            ref[t, h] = b[t, h] * (p.v[t, h] - Sd.T @ kh[t, h])
    check(vn[0], ref, dtype, "v_new")


def test_deterministic(cuda_lib):
    cfg = KdaConfig("det", B=2, T=300, H=4, dk=128, dv=128, dtype="bf16", initial_state=True)
    inp = to_cuda(make(cfg))
    o1, f1 = gpu_fwd(cuda_lib, cfg, inp)
    o2, f2 = gpu_fwd(cuda_lib, cfg, inp)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_mid_bf16_workload(cuda_lib):
    """B=2, T=4096, H=16, d=128 bf16: every output against the oracle."""
    cfg = CONFIGS["mid_bf16"]
    inp = make(cfg)
    out, fin, o_ref, f_ref = _run_both(cuda_lib, cfg, inp)
    check(out.reshape(o_ref.shape), o_ref, "bf16", "o")
    check(fin, f_ref, "bf16", "final_state")


def test_kimi_bf16_workload_sampled(cuda_lib):
    """B=4, T=8192, H=32, d=128, gate and base-2 decay in kernel, initial
    state: the whole batch on the GPU, four full-length (sequence, head)
    units through the oracle."""
    cfg = CONFIGS["kimi_bf16"]
    inp_c = make(cfg)
    out, fin = gpu_fwd(cuda_lib, cfg, to_cuda(inp_c))
    out, fin = out.cpu(), fin.cpu()
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    for (b, h) in [(0, 0), (1, 7), (2, 31), (3, 18)]:
        sub = dict(inp_c)
        sub["a_log"] = inp_c["a_log"][h:h + 1]
        sub["dt_bias"] = inp_c["dt_bias"][h:h + 1]
        sl = lambda x: x[b:b + 1, :, h:h + 1].contiguous()
        p = oracle_problem(cfg, sub, q=sl(inp_c["q"]), k=sl(inp_c["k"]), v=sl(inp_c["v"]),
                           g=sl(inp_c["g"]), beta=inp_c["beta"][b:b + 1, :, h:h + 1].contiguous(),
                           cu=[0, cfg.T])
        S0 = inp_c["initial_state"][b:b + 1, h:h + 1]
        o_ref, f_ref = oracle.chunk_fwd(p, S0)
        check(out[b, :, h], o_ref[:, 0], "bf16", f"o[{b},:,{h}]")
        check(fin[b, h], f_ref[0, 0], "bf16", f"final[{b},{h}]")
