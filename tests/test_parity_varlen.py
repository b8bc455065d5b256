"""The varlen packed prefill workload on the GPU: 64 sequences with lengths
~ U{64..8192} (TND), initial states gathered by int32 index from a
[512, H, 128, 128] fp32 pool (about 10% gather zero through index -1 or a
false flag), the chunked forward, final states scattered back.

Gather and scatter are checked bit-exact on the whole pool; the forward is
checked against the oracle on sampled (sequence, head) units, including the
shortest and the longest sequence."""
import numpy as np
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import CONFIGS
from kda_testutil import check, gpu_fwd, make, oracle_problem, to_cuda

pytestmark = pytest.mark.gpu


def test_varlen_prefill_workload(cuda_lib):
    cfg = CONFIGS["varlen_bf16"]
    inp_c = make(cfg)
    inp = to_cuda(inp_c)
    pool, idx, flags = inp["pool"], inp["idx"], inp["flags"]
    S0 = cuda_lib.kda_state_gather(pool, idx, flags)
    S0_ref = oracle.state_gather(inp_c["pool"].numpy().reshape(-1), pool.shape[0],
                                 pool.stride(0), pool[0].numel(), inp_c["idx"].numpy(),
                                 inp_c["flags"].numpy())
    np.testing.assert_array_equal(S0.cpu().numpy().reshape(S0_ref.shape), S0_ref)
    inp["initial_state"] = S0
    out, fin = gpu_fwd(cuda_lib, cfg, inp)
    pool_before = pool.cpu().numpy().reshape(-1).copy()
    cuda_lib.kda_state_scatter(pool, idx, fin)
    pool_ref = oracle.state_scatter(pool_before, pool.shape[0], pool.stride(0), pool[0].numel(),
                                    inp_c["idx"].numpy(), fin.cpu().numpy().reshape(len(idx), -1))
    np.testing.assert_array_equal(pool.cpu().numpy().reshape(-1), pool_ref)

    lens = inp_c["seq_lens"].numpy()
    cu = np.concatenate([[0], np.cumsum(lens)])
    picks = [(int(np.argmin(lens)), 0), (int(np.argmax(lens)), 31), (5, 17)]
    bad = np.where((inp_c["idx"].numpy() < 0) | ~inp_c["flags"].numpy())[0]
    if len(bad):
        picks.append((int(bad[0]), 3))   # a sequence that started from zero
    out_c, fin_c = out.cpu(), fin.cpu()
    for (n, h) in picks:
        a, b = cu[n], cu[n + 1]
        sub = dict(inp_c, a_log=inp_c["a_log"][h:h + 1], dt_bias=inp_c["dt_bias"][h:h + 1],
                   cu_seqlens=None)
        sl = lambda x: x[a:b, h:h + 1].contiguous()
        p = oracle_problem(cfg, sub, q=sl(inp_c["q"]), k=sl(inp_c["k"]), v=sl(inp_c["v"]),
                           g=sl(inp_c["g"]), beta=sl(inp_c["beta"]), cu=[0, b - a])
        o_ref, f_ref = oracle.chunk_fwd(p, S0_ref[n].reshape(1, cfg.H, cfg.dk, cfg.dv)[:, h:h + 1])
        check(out_c[a:b, h], o_ref[:, 0], "bf16", f"o seq {n} head {h}")
        check(fin_c[n, h], f_ref[0, 0], "bf16", f"final seq {n} head {h}")
