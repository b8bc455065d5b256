"""GPU parity of kda_chunk_bwd (through the C ABI) against the fp64 oracle's
reverse-mode gradients of the token recurrence.

Every gradient the call returns is compared: dq, dk, dv, dbeta, dg (of the
inputs as given), dA_log, ddt_bias and the initial-state gradient, with the
forward's acceptance tolerances (fp32 inputs: max relative error <= 1e-4;
bf16 inputs: relative L2 <= 2e-2)."""
import numpy as np
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import CONFIGS, KdaConfig, make_cotangents
from kda_testutil import check, fwd_kwargs, make, oracle_problem, to_cuda

pytestmark = pytest.mark.gpu

GRADS = [("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dg", "dg"), ("dbeta", "dbeta")]


def _gpu_bwd(kda, cfg, inp, cot, *, with_dout=True, with_dfin=True):
    kw = fwd_kwargs(cfg, inp)
    return kda.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                             cot["d_out"] if with_dout else None,
                             d_final_state=cot["d_final_state"] if with_dfin else None,
                             want_d_initial_state=True, **kw)


def _compare(got, ref, cfg, dtype):
    for name, rname in GRADS:
        check(got[name].reshape(ref[rname].shape), ref[rname], dtype, name)
    check(got["d_initial_state"], ref["d_initial"], dtype, "d_initial_state")
    if cfg.gate_in_kernel:
        check(got["da_log"], ref["da_log"], dtype, "da_log")
        check(got["ddt_bias"], ref["ddt_bias"], dtype, "ddt_bias")
    else:
        assert got["da_log"] is None and got["ddt_bias"] is None


def _run(kda, cfg, *, with_dout=True, with_dfin=True, inp_c=None):
    inp_c = make(cfg) if inp_c is None else inp_c
    cot_c = make_cotangents(cfg, inp_c)
    got = _gpu_bwd(kda, cfg, to_cuda(inp_c), to_cuda(cot_c), with_dout=with_dout,
                   with_dfin=with_dfin)
    torch.cuda.synchronize()
    ref = oracle.chunk_bwd(oracle_problem(cfg, inp_c), inp_c["initial_state"],
                           cot_c["d_out"] if with_dout else None,
                           cot_c["d_final_state"] if with_dfin else None)
    return got, ref


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 63, 65, 130])
def test_bwd_ragged_small(cuda_lib, dtype, dk, dv, T):
    cfg = KdaConfig("bwd", B=2, T=T, H=2, dk=dk, dv=dv, dtype=dtype, initial_state=True,
                    use_exp2=(T % 2 == 1), seed=T + dk + dv)
    got, ref = _run(cuda_lib, cfg)
    _compare(got, ref, cfg, dtype)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 64), ("bf16", 128)])
def test_bwd_precomputed_gate_and_beta_without_l2norm(cuda_lib, dtype, d):
    cfg = KdaConfig("bwd_pre", B=1, T=150, H=2, dk=d, dv=d, dtype=dtype, gate_in_kernel=False,
                    beta_sigmoid=False, l2norm=False, initial_state=True, seed=5)
    inp = make(cfg)
    inp["k"] = (inp["k"].float() * 0.1).to(inp["k"].dtype)  # keep the unnormalised rule contractive
    got, ref = _run(cuda_lib, cfg, inp_c=inp)
    _compare(got, ref, cfg, dtype)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
@pytest.mark.parametrize("which", ["d_out only", "d_final only"])
def test_bwd_one_cotangent(cuda_lib, which, dtype, d):
    cfg = KdaConfig("bwd_one", B=1, T=200, H=2, dk=d, dv=d, dtype=dtype, initial_state=True,
                    seed=3)
    got, ref = _run(cuda_lib, cfg, with_dout=(which == "d_out only"),
                    with_dfin=(which == "d_final only"))
    _compare(got, ref, cfg, dtype)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_bwd_varlen(cuda_lib, dtype, d):
    lens = (1, 64, 0, 65, 200, 3)
    cfg = KdaConfig("bwd_varlen", dtype=dtype, H=2, dk=d, dv=d, seq_lens=lens, initial_state=True,
                    seed=9)
    got, ref = _run(cuda_lib, cfg)
    _compare(got, ref, cfg, dtype)
    # an empty sequence hands its state gradient through unchanged
    cot = make_cotangents(cfg, make(cfg))
    np.testing.assert_array_equal(got["d_initial_state"][2].cpu().numpy(),
                                  cot["d_final_state"][2].numpy())


@pytest.mark.parametrize("dtype,d,H,Hk", [("f32", 64, 4, 2), ("bf16", 128, 4, 1)])
def test_bwd_grouped_key_heads(cuda_lib, dtype, d, H, Hk):
    """dq, dk of a key head = the oracle's gradients of the expanded heads,
    summed over the value heads that share it."""
    cfg = KdaConfig("bwd_gqa", B=2, T=100, H=H, dk=d, dv=d, dtype=dtype, initial_state=True,
                    seed=17)
    inp = make(cfg)
    grp = H // Hk
    small, wide = dict(inp), dict(inp)
    for n in ("q", "k"):
        x = inp[n][..., :Hk, :].contiguous()
        small[n] = x
        wide[n] = x.repeat_interleave(grp, dim=-2).contiguous()
    cot = make_cotangents(cfg, inp)
    got = _gpu_bwd(cuda_lib, cfg, to_cuda(small), to_cuda(cot))
    torch.cuda.synchronize()
    ref = oracle.chunk_bwd(oracle_problem(cfg, wide), inp["initial_state"], cot["d_out"],
                           cot["d_final_state"])
    T = 2 * 100
    for name in ("dq", "dk"):
        r = ref[name].reshape(T, Hk, grp, d).sum(axis=2)
        check(got[name].reshape(T, Hk, d), r, dtype, name)
    for name in ("dv", "dg", "dbeta"):
        check(got[name].reshape(ref[name].shape), ref[name], dtype, name)
    check(got["d_initial_state"], ref["d_initial"], dtype, "d_initial_state")
    check(got["da_log"], ref["da_log"], dtype, "da_log")


def test_bwd_empty_batch(cuda_lib):
    cfg = KdaConfig("bwd_empty", B=2, T=0, H=2, dk=64, dv=64, dtype="bf16", initial_state=True)
    inp = to_cuda(make(cfg))
    cot = to_cuda(make_cotangents(cfg, inp))
    got = _gpu_bwd(cuda_lib, cfg, inp, cot)
    torch.cuda.synchronize()
    assert torch.equal(got["d_initial_state"], cot["d_final_state"])
    assert torch.count_nonzero(got["da_log"]) == 0


def test_bwd_deterministic(cuda_lib):
    cfg = KdaConfig("bwd_det", B=2, T=300, H=3, dk=128, dv=128, dtype="bf16", initial_state=True,
                    seed=1)
    inp = to_cuda(make(cfg))
    cot = to_cuda(make_cotangents(cfg, inp))
    a = _gpu_bwd(cuda_lib, cfg, inp, cot)
    b = _gpu_bwd(cuda_lib, cfg, inp, cot)
    torch.cuda.synchronize()
    for name in a:
        if a[name] is not None:
            assert torch.equal(a[name], b[name]), name


def test_bwd_kimi_bf16_workload_sampled(cuda_lib):
    """Full-size backward (B=4, T=8192, H=32, d=128); the oracle recomputes
    heads 0 and 31 over all four sequences (heads are independent problems),
    which also fixes dA_log and ddt_bias of those heads."""
    cfg = CONFIGS["kimi_bf16"]
    inp_c = make(cfg)
    cot_c = make_cotangents(cfg, inp_c)
    got = _gpu_bwd(cuda_lib, cfg, to_cuda(inp_c), to_cuda(cot_c))
    torch.cuda.synchronize()
    for h in (0, 31):
        sl = lambda x: x[:, :, h:h + 1].contiguous()
        sub = dict(inp_c)
        for n in ("q", "k", "v", "g", "beta"):
            sub[n] = sl(inp_c[n])
        sub["a_log"] = inp_c["a_log"][h:h + 1]
        sub["dt_bias"] = inp_c["dt_bias"][h:h + 1]
        sub["initial_state"] = inp_c["initial_state"][:, h:h + 1].contiguous()
        ref = oracle.chunk_bwd(oracle_problem(cfg.replace(H=1), sub), sub["initial_state"],
                               sl(cot_c["d_out"]), cot_c["d_final_state"][:, h:h + 1])
        for name, rname in GRADS:
            g = got[name][:, :, h:h + 1]
            check(g.reshape(ref[rname].shape), ref[rname], "bf16", f"{name} (head {h})")
        check(got["d_initial_state"][:, h:h + 1], ref["d_initial"], "bf16", "d_initial")
        check(got["da_log"][h:h + 1], ref["da_log"], "bf16", "da_log")
        check(got["ddt_bias"][h:h + 1], ref["ddt_bias"], "bf16", "ddt_bias")
