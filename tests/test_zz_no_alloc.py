"""kda_chunk_fwd_static_scratch: the forward for callers that cannot allocate
device memory (a plugin whose host owns all device memory, or a path where
cudaMalloc is not allowed).  It runs the same kernels as kda_chunk_fwd with
its scratch in the library's fixed array, so its results must equal the
workspace forward's bit for bit, call after call (the array keeps the last
call's contents), for every layout and state orientation that changes the
scratch plan.  It must refuse problems whose scratch exceeds the array -
checked at the edge: the largest problem that fits runs, the next size up is
refused - and KDA_REUSE_PREP, which would read a previous call's leftovers.

This file is collected last on purpose: the other GPU tests run first."""
import ctypes

import pytest
import torch

import chunked_kimi_delta_gb300 as kda
from chunked_kimi_delta_gb300.inputs import KdaConfig
from kda_testutil import fwd_kwargs, make, to_cuda

pytestmark = pytest.mark.gpu

KDA_OK, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE = 0, 2, 4


def _head_major(inp):
    """[B, T, H, D] / [B, T, H] tensors as [B, H, T, D] / [B, H, T]."""
    out = dict(inp)
    for n in ("q", "k", "v", "g"):
        out[n] = inp[n].transpose(1, 2).contiguous()
    out["beta"] = inp["beta"].transpose(1, 2).contiguous()
    return out


def _v_first(inp):
    out = dict(inp)
    if inp["initial_state"] is not None:
        out["initial_state"] = inp["initial_state"].transpose(-1, -2).contiguous()
    return out


def _both(cuda_lib, cfg, inp, **layout):
    kw = {**fwd_kwargs(cfg, inp), **layout}
    q, k, v, g, b = inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"]
    ref_out, ref_fin = cuda_lib.kda_chunk_fwd(q, k, v, g, b, **kw)
    torch.cuda.synchronize()
    for call in range(2):  # the shared array keeps the previous call's contents
        out, fin = cuda_lib.kda_chunk_fwd_static_scratch(q, k, v, g, b, **kw)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), f"out differs on call {call}"
        assert torch.equal(fin, ref_fin), f"final state differs on call {call}"
        assert kda.kda_static_scratch_status() == KDA_OK


@pytest.mark.parametrize("v_first", [False, True], ids=["k_first", "v_first"])
@pytest.mark.parametrize("head_major", [False, True], ids=["token_major", "head_major"])
@pytest.mark.parametrize("cfg", [
    KdaConfig("noalloc_bf16", B=1, T=1000, H=8, dk=128, dv=128, dtype="bf16", use_exp2=True,
              initial_state=True, seed=21),
    KdaConfig("noalloc_f32", B=2, T=130, H=2, dk=64, dv=64, dtype="f32", initial_state=True,
              seed=22),
], ids=["bf16_d128", "f32_d64"])
def test_static_scratch_matches_workspace_forward(cuda_lib, cfg, head_major, v_first):
    inp = to_cuda(make(cfg))
    if v_first:
        inp = _v_first(inp)
    if head_major:
        inp = _head_major(inp)
    _both(cuda_lib, cfg, inp, head_major=head_major, state_v_first=v_first)


def _ws_bytes(T, H):
    """kda_chunk_fwd_workspace_size of a B=1, bf16 d=128 forward of T tokens
    (sizes only: host tensors serve for the query)."""
    q = torch.empty(1, T, H, 128, dtype=torch.bfloat16)
    g = torch.empty(1, T, H, 128)
    b = torch.empty(1, T, H)
    a = kda.make_fwd_args(q, q, q, g, b, out=q)
    return kda.load_library().kda_chunk_fwd_workspace_size(ctypes.byref(a))


def test_static_scratch_size_limit_at_the_edge(cuda_lib):
    """The largest T (B=1, H=8, bf16 d=128) whose scratch fits the array runs
    and matches the workspace forward; one more token is refused."""
    H, lo, hi = 8, 64, 1 << 16
    assert _ws_bytes(lo, H) <= kda.KDA_STATIC_SCRATCH_BYTES < _ws_bytes(hi, H)
    while hi - lo > 1:  # largest T that fits
        mid = (lo + hi) // 2
        if _ws_bytes(mid, H) <= kda.KDA_STATIC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    cfg = KdaConfig("noalloc_edge", B=1, T=lo, H=H, dk=128, dv=128, dtype="bf16", use_exp2=True,
                    initial_state=True, seed=23)
    _both(cuda_lib, cfg, to_cuda(make(cfg)))
    big = KdaConfig("noalloc_over", B=1, T=lo + 1, H=H, dk=128, dv=128, dtype="bf16", seed=24)
    inp = to_cuda(make(big))
    a = kda.make_fwd_args(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                          **{**fwd_kwargs(big, inp), "out": torch.empty_like(inp["v"])})
    lib = kda.load_library()
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(a)) > kda.KDA_STATIC_SCRATCH_BYTES
    assert lib.kda_chunk_fwd_static_scratch(ctypes.byref(a), None) == KDA_ERR_WORKSPACE


def test_static_scratch_refuses_reuse_of_leftovers(cuda_lib):
    cfg = KdaConfig("noalloc_reuse", B=1, T=256, H=2, dk=128, dv=128, dtype="bf16", seed=25)
    inp = to_cuda(make(cfg))
    a = kda.make_fwd_args(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                          extra_flags=kda.KDA_REUSE_PREP,
                          **{**fwd_kwargs(cfg, inp), "out": torch.empty_like(inp["v"])})
    assert kda.load_library().kda_chunk_fwd_static_scratch(ctypes.byref(a), None) == KDA_ERR_UNSUPPORTED
