"""GPU parity with grouped key heads: q and k carry Hk heads shared by the H
value heads ("Hyper-Parallel Chunk KDA current implementation design",
section 4.2: value heads may outnumber query/key heads, which are expanded
to the value heads).  Value head h reads key head h // (H // Hk).

Each case checks the library against the fp64 oracle run on q/k expanded to
H heads, and against the library itself on the expanded q/k (bit for bit:
the grouping changes addressing only)."""
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import KdaConfig
from kda_testutil import check, fwd_kwargs, gpu_fwd, make, oracle_problem, scale_of, to_cuda

pytestmark = pytest.mark.gpu


def _group(inp, Hk):
    """Inputs with q, k cut to their first Hk heads, and the same expanded back
    to H heads (value head h <- key head h // (H // Hk))."""
    H = inp["v"].shape[-2]
    grp = H // Hk
    small = dict(inp)
    wide = dict(inp)
    for n in ("q", "k"):
        x = inp[n][..., :Hk, :].contiguous()
        small[n] = x
        wide[n] = x.repeat_interleave(grp, dim=-2).contiguous()
    return small, wide


@pytest.mark.parametrize("dtype,dk,dv,H,Hk,T", [
    ("bf16", 128, 128, 4, 1, 130),   # tensor-core path, one key head
    ("bf16", 128, 128, 6, 2, 200),   # tensor-core path, groups of 3
    ("bf16", 128, 128, 4, 4, 65),    # Hk = H: plain heads
    ("f32", 64, 64, 6, 3, 65),       # CUDA-core path
    ("bf16", 64, 128, 4, 2, 100),    # CUDA-core path, d_k != d_v
])
def test_gqa_forward(cuda_lib, dtype, dk, dv, H, Hk, T):
    cfg = KdaConfig("gqa", B=2, T=T, H=H, dk=dk, dv=dv, dtype=dtype, initial_state=True,
                    use_exp2=True, seed=H * 10 + Hk)
    small_c, wide_c = _group(make(cfg), Hk)
    small, wide = to_cuda(small_c), to_cuda(wide_c)
    out, fin = gpu_fwd(cuda_lib, cfg, small)
    assert out.shape == (2, T, H, dv) and fin.shape == (2, H, dk, dv)
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(cfg, wide_c), wide_c["initial_state"])
    check(out.reshape(o_ref.shape), o_ref, dtype, "o")
    check(fin, f_ref, dtype, "final_state")
    o_w, f_w = gpu_fwd(cuda_lib, cfg, wide)
    assert torch.equal(out, o_w) and torch.equal(fin, f_w)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_gqa_varlen(cuda_lib, dtype, d):
    lens = (1, 64, 0, 65, 200, 3)
    cfg = KdaConfig("gqa_varlen", dtype=dtype, H=4, dk=d, dv=d, seq_lens=lens, initial_state=True,
                    seed=21)
    small_c, wide_c = _group(make(cfg), 2)
    out, fin = gpu_fwd(cuda_lib, cfg, to_cuda(small_c))
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(cfg, wide_c), wide_c["initial_state"])
    check(out.reshape(o_ref.shape), o_ref, dtype, "o")
    check(fin, f_ref, dtype, "final_state")


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_gqa_segment_summary(cuda_lib, dtype, d):
    bounds = (0, 64, 100, 200, 333)
    cfg = KdaConfig("gqa_seg", B=1, T=333, H=4, dk=d, dv=d, dtype=dtype, use_exp2=True, seed=13)
    small_c, wide_c = _group(make(cfg), 1)
    small = to_cuda(small_c)
    kw = fwd_kwargs(cfg, small)
    kw.pop("initial_state")
    kw.pop("cu_seqlens")
    sb = torch.tensor(bounds, dtype=torch.int32, device="cuda")
    M, St = cuda_lib.kda_segment_summary(small["q"], small["k"], small["v"], small["g"],
                                         small["beta"], sb, **kw)
    torch.cuda.synchronize()
    assert M.shape == (4, 4, d, d)
    M_ref, St_ref = oracle.segment_summary(oracle_problem(cfg, wide_c), bounds)
    check(M, M_ref, dtype, "M")
    check(St, St_ref, dtype, "S_tilde")


def test_gqa_host_io_equals_device_forward(cuda_lib):
    cfg = KdaConfig("gqa_host", B=2, T=1500, H=4, dk=128, dv=128, dtype="bf16",
                    initial_state=True, seed=4)
    small_c, _ = _group(make(cfg), 2)
    small = to_cuda(small_c)
    o_ref, f_ref = gpu_fwd(cuda_lib, cfg, small)
    h = {n: small_c[n].pin_memory() for n in ("q", "k", "v", "g", "beta")}
    args = fwd_kwargs(cfg, small)
    args.pop("cu_seqlens")
    out, fin = cuda_lib.kda_chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], **args)
    torch.cuda.synchronize()
    assert torch.equal(out, o_ref.cpu()) and torch.equal(fin, f_ref)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_gqa_decode(cuda_lib, dtype, d):
    N, T, H, Hk, rows = 3, 3, 6, 2, 5
    cfg = KdaConfig("gqa_dec", B=N, T=T, H=H, dk=d, dv=d, dtype=dtype, seed=31)
    small_c, wide_c = _group(make(cfg), Hk)
    gen = torch.Generator().manual_seed(2)
    pool = (torch.randn(rows, H, d, d, generator=gen) * 0.1).cuda()
    idx = torch.tensor([4, 0, 2], dtype=torch.int32)
    S0 = torch.stack([pool[int(r)].double().cpu() for r in idx])
    dev = {n: small_c[n].cuda() for n in ("q", "k", "v", "g", "beta", "a_log", "dt_bias")}
    out = cuda_lib.kda_recurrent_step(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], pool,
                                      idx.cuda(), scale=scale_of(cfg), a_log=dev["a_log"],
                                      dt_bias=dev["dt_bias"], beta_sigmoid=True,
                                      gate_in_kernel=True)
    torch.cuda.synchronize()
    assert out.shape == (N, T, H, d)
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(cfg, wide_c), S0)
    check(out.reshape(o_ref.shape), o_ref, dtype, "o")
    for i in range(N):
        check(pool[int(idx[i])], f_ref[i], dtype, f"pool row {int(idx[i])}")
