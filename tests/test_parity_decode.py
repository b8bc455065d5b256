"""GPU parity of kda_recurrent_step (decode on pool states, in place) against
the fp64 oracle's token recurrence: outputs, the written pool rows, rows
that must stay untouched, and the invalid-index / flag conventions."""
import numpy as np
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import KdaConfig
from kda_testutil import check, make, oracle_problem, scale_of

pytestmark = pytest.mark.gpu


def _pool(rows, H, dk, dv, dtype, gap, seed):
    g = torch.Generator().manual_seed(seed)
    payload = H * dk * dv
    base = torch.randn(rows, payload + gap, generator=g) * 0.1
    base = base.to(dtype).cuda()
    return base, base[:, :payload].view(rows, H, dk, dv)


@pytest.mark.parametrize("dtype,pool_dtype", [("f32", torch.float32), ("bf16", torch.float32),
                                              ("bf16", torch.bfloat16)])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("T", [1, 5])
@pytest.mark.parametrize("layout", ["aligned", "unaligned"])
def test_decode_against_oracle(cuda_lib, dtype, pool_dtype, dk, dv, T, layout):
    N, H, rows = 6, 3, 9
    cfg = KdaConfig("decode", B=N, T=T, H=H, dk=dk, dv=dv, dtype=dtype, beta_sigmoid=True,
                    gate_in_kernel=True, seed=dk + dv + T)
    inp = make(cfg)
    # gap 40 keeps the rows 16-byte aligned (vector accesses); gap 3 does not
    # (element-wise accesses)
    base, pool = _pool(rows, H, dk, dv, pool_dtype, gap=40 if layout == "aligned" else 3, seed=T)
    before = base.clone()
    idx = torch.tensor([4, -1, 0, 9, 7, 2], dtype=torch.int32)     # -1 and 9 (= rows) invalid
    flags = torch.tensor([True, True, False, True, True, True])       # row 0: start from zero
    S0 = torch.zeros(N, H, dk, dv, dtype=torch.float64)
    for i in range(N):
        r = int(idx[i])
        if 0 <= r < rows and flags[i]:
            S0[i] = pool[r].double().cpu()
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "g", "beta", "a_log", "dt_bias")}
    out = cuda_lib.kda_recurrent_step(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], pool,
                                      idx.cuda(), flags.cuda(), scale=scale_of(cfg),
                                      a_log=dev["a_log"], dt_bias=dev["dt_bias"], l2norm_qk=True,
                                      beta_sigmoid=True, gate_in_kernel=True)
    torch.cuda.synchronize()
    p = oracle_problem(cfg, inp)
    o_ref, f_ref = oracle.chunk_fwd(p, S0)
    tol = "f32" if dtype == "f32" else "bf16"
    check(out.reshape(o_ref.shape), o_ref, tol, "o")
    written = set()
    for i in range(N):
        r = int(idx[i])
        if 0 <= r < rows:
            check(pool[r], f_ref[i], "f32" if (dtype == "f32" and pool_dtype == torch.float32) else "bf16",
                  f"pool row {r}")
            written.add(r)
    payload = H * dk * dv
    for r in range(rows):
        if r not in written:
            assert torch.equal(base[r], before[r]), f"row {r} changed"
        assert torch.equal(base[r, payload:], before[r, payload:]), f"gap of row {r} changed"


def test_decode_int64_indices_and_no_flags(cuda_lib):
    """int64 indices, no flags: every valid row starts from its pool state."""
    N, H, dk, dv, rows = 3, 2, 128, 128, 5
    cfg = KdaConfig("decode64", B=N, T=2, H=H, dk=dk, dv=dv, dtype="bf16", beta_sigmoid=True,
                    gate_in_kernel=True, seed=3)
    inp = make(cfg)
    _, pool = _pool(rows, H, dk, dv, torch.float32, gap=0, seed=1)
    idx = torch.tensor([3, 1, 4], dtype=torch.int64)
    S0 = torch.stack([pool[int(r)].double().cpu() for r in idx])
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "g", "beta", "a_log", "dt_bias")}
    out = cuda_lib.kda_recurrent_step(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], pool,
                                      idx.cuda(), scale=scale_of(cfg), a_log=dev["a_log"],
                                      dt_bias=dev["dt_bias"], beta_sigmoid=True, gate_in_kernel=True)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(cfg, inp), S0)
    check(out.reshape(o_ref.shape), o_ref, "bf16", "o")
    for i in range(N):
        check(pool[int(idx[i])], f_ref[i], "bf16", f"row {int(idx[i])}")


def test_decode_matches_chunked_forward(cuda_lib):
    """T = 130 tokens through the decode step equal the chunked forward from
    the same initial states (both against the same recurrence)."""
    N, H, dk, dv, T = 2, 2, 128, 128, 130
    cfg = KdaConfig("decode_long", B=N, T=T, H=H, dk=dk, dv=dv, dtype="bf16", beta_sigmoid=True,
                    gate_in_kernel=True, initial_state=True, seed=8)
    inp = make(cfg)
    dev = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in inp.items()}
    pool = dev["initial_state"].clone()
    idx = torch.arange(N, dtype=torch.int32, device="cuda")
    out = cuda_lib.kda_recurrent_step(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], pool, idx,
                                      scale=scale_of(cfg), a_log=dev["a_log"], dt_bias=dev["dt_bias"],
                                      beta_sigmoid=True, gate_in_kernel=True)
    o_c, f_c = cuda_lib.kda_chunk_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                      scale=scale_of(cfg), a_log=dev["a_log"], dt_bias=dev["dt_bias"],
                                      initial_state=dev["initial_state"], beta_sigmoid=True,
                                      gate_in_kernel=True, use_exp2=True)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(cfg, inp), inp["initial_state"])
    check(out.reshape(o_ref.shape), o_ref, "bf16", "decode o")
    check(pool, f_ref, "bf16", "decode state")
    check(o_c.reshape(o_ref.shape), o_ref, "bf16", "chunked o")


def test_decode_layouts_agree_bit_for_bit(cuda_lib):
    """Vector and element-wise state accesses compute the same thing:
    identical outputs and states on a 64-sequence, 32-head pool step."""
    N, H, dk, dv, rows = 64, 32, 128, 128, 512
    cfg = KdaConfig("decode_forms", B=N, T=1, H=H, dk=dk, dv=dv, dtype="bf16", beta_sigmoid=True,
                    gate_in_kernel=True, seed=12)
    inp = make(cfg, device="cuda")
    _, pool = _pool(rows, H, dk, dv, torch.float32, gap=0, seed=2)
    base2 = torch.zeros(rows, H * dk * dv + 3, device="cuda")
    pool2 = base2[:, :H * dk * dv].view(rows, H, dk, dv)
    pool2.copy_(pool)
    idx = torch.randperm(rows, generator=torch.Generator().manual_seed(0))[:N].to(torch.int32).cuda()
    kw = dict(scale=scale_of(cfg), a_log=inp["a_log"], dt_bias=inp["dt_bias"], beta_sigmoid=True,
              gate_in_kernel=True)
    o1 = cuda_lib.kda_recurrent_step(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], pool, idx, **kw)
    o2 = cuda_lib.kda_recurrent_step(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], pool2, idx, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(pool, pool2)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128)])
def test_decode_many_states_against_oracle(cuda_lib, dk, dv):
    """More states than the GPU holds CTAs at once (384 states, aligned fp32
    pool): invalid rows, a false flag and untouched rows as in the small
    cases; three tokens per sequence."""
    N, H, T, rows = 48, 8, 3, 64
    cfg = KdaConfig("decode_many", B=N, T=T, H=H, dk=dk, dv=dv, dtype="bf16", beta_sigmoid=True,
                    gate_in_kernel=True, seed=dk + 5)
    inp = make(cfg)
    base, pool = _pool(rows, H, dk, dv, torch.float32, gap=0, seed=9)
    before = base.clone()
    perm = torch.randperm(rows, generator=torch.Generator().manual_seed(4))[:N].to(torch.int32)
    idx = perm.clone()
    idx[5] = -1
    idx[17] = rows  # past the pool: invalid
    flags = torch.ones(N, dtype=torch.bool)
    flags[9] = False
    S0 = torch.zeros(N, H, dk, dv, dtype=torch.float64)
    for i in range(N):
        r = int(idx[i])
        if 0 <= r < rows and flags[i]:
            S0[i] = pool[r].double().cpu()
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "g", "beta", "a_log", "dt_bias")}
    out = cuda_lib.kda_recurrent_step(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], pool,
                                      idx.cuda(), flags.cuda(), scale=scale_of(cfg),
                                      a_log=dev["a_log"], dt_bias=dev["dt_bias"], l2norm_qk=True,
                                      beta_sigmoid=True, gate_in_kernel=True)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(cfg, inp), S0)
    check(out.reshape(o_ref.shape), o_ref, "bf16", "o")
    written = set()
    for i in range(N):
        r = int(idx[i])
        if 0 <= r < rows:
            check(pool[r], f_ref[i], "bf16", f"pool row {r}")
            written.add(r)
    for r in range(rows):
        if r not in written:
            assert torch.equal(base[r], before[r]), f"row {r} changed"
