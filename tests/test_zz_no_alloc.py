"""kda_chunk_fwd_static_scratch: the forward for callers that cannot allocate
device memory (a plugin whose host owns all device memory, or a path where
cudaMalloc is not allowed).  It must give the results of kda_chunk_fwd with a
caller workspace, call after call, and refuse problems whose scratch exceeds
the library's fixed array.

This file is collected last on purpose: the other GPU tests run first."""
import ctypes

import numpy as np
import pytest
import torch

import chunked_kimi_delta_gb300 as kda
from chunked_kimi_delta_gb300.inputs import KdaConfig
from kda_testutil import TOL_BF16_RELL2, TOL_F32_MAXREL, fwd_kwargs, make, max_rel, rel_l2, to_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [
    KdaConfig("noalloc_bf16", B=1, T=1000, H=8, dk=128, dv=128, dtype="bf16", use_exp2=True,
              initial_state=True, seed=21),
    KdaConfig("noalloc_f32", B=2, T=130, H=2, dk=64, dv=64, dtype="f32", initial_state=True,
              seed=22),
], ids=["bf16_d128", "f32_d64"])
def test_static_scratch_matches_workspace_forward(cuda_lib, cfg):
    inp = to_cuda(make(cfg))
    kw = fwd_kwargs(cfg, inp)
    q, k, v, g, b = inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"]
    ref_out, ref_fin = cuda_lib.kda_chunk_fwd(q, k, v, g, b, **kw)
    torch.cuda.synchronize()
    ref_out, ref_fin = ref_out.float().cpu().numpy(), ref_fin.cpu().numpy()
    for _ in range(2):  # the shared array keeps the previous call's contents
        out, fin = cuda_lib.kda_chunk_fwd_static_scratch(q, k, v, g, b, **kw)
        torch.cuda.synchronize()
        out, fin = out.float().cpu().numpy(), fin.cpu().numpy()
        if cfg.dtype == "f32":
            assert max_rel(out, ref_out) <= TOL_F32_MAXREL
            assert max_rel(fin, ref_fin) <= TOL_F32_MAXREL
        else:
            assert rel_l2(out, ref_out) <= TOL_BF16_RELL2
            assert rel_l2(fin, ref_fin) <= TOL_BF16_RELL2


def test_static_scratch_refuses_oversized_problem(cuda_lib):
    cfg = KdaConfig("noalloc_big", B=1, T=8192, H=8, dk=128, dv=128, dtype="bf16", seed=23)
    inp = to_cuda(make(cfg))
    a = kda.make_fwd_args(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                          **{**fwd_kwargs(cfg, inp), "out": torch.empty_like(inp["v"])})
    lib = kda.load_library()
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(a)) > kda.KDA_STATIC_SCRATCH_BYTES
    assert lib.kda_chunk_fwd_static_scratch(ctypes.byref(a), None) == 4  # KDA_ERR_WORKSPACE
