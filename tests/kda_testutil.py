"""Helpers shared by the GPU parity tests: run the CUDA library and the fp64
oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import KdaConfig, make_inputs, oracle_kwargs

# Tolerances fixed by the acceptance criteria: fp32 inputs max relative error
# (max|x - y| / max|y|) <= 1e-4; bf16 inputs with fp32 state relative L2
# (||x - y|| / ||y||) <= 2e-2, on o and final_state (and M, S~, S_in).
TOL_F32_MAXREL = 1e-4
TOL_BF16_RELL2 = 2e-2


def max_rel(x, y) -> float:
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    den = np.max(np.abs(y))
    return float(np.max(np.abs(x - y)) / den) if den > 0 else float(np.max(np.abs(x)))


def rel_l2(x, y) -> float:
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    den = np.linalg.norm(y)
    return float(np.linalg.norm(x - y) / den) if den > 0 else float(np.linalg.norm(x))


def check(x, y, dtype: str, what: str):
    """Asserts the acceptance tolerance for the workload dtype."""
    x = x.detach().float().cpu().numpy() if hasattr(x, "detach") else x
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    if dtype == "f32":
        e = max_rel(x, y)
        assert e <= TOL_F32_MAXREL, f"{what}: max rel err {e:.3e} > {TOL_F32_MAXREL}"
    else:
        e = rel_l2(x, y)
        assert e <= TOL_BF16_RELL2, f"{what}: rel L2 {e:.3e} > {TOL_BF16_RELL2}"
    return e


def scale_of(cfg: KdaConfig) -> float:
    return float(np.float32(cfg.dk ** -0.5))


def fwd_kwargs(cfg: KdaConfig, inp: dict) -> dict:
    return dict(scale=scale_of(cfg), eps=1e-6, a_log=inp["a_log"], dt_bias=inp["dt_bias"],
                initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"],
                l2norm_qk=cfg.l2norm, beta_sigmoid=cfg.beta_sigmoid,
                gate_in_kernel=cfg.gate_in_kernel, use_exp2=cfg.use_exp2)


def to_cuda(inp: dict) -> dict:
    return {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "seq_lens" else v)
            for k, v in inp.items()}


def gpu_fwd(kda, cfg: KdaConfig, inp: dict, **kw):
    args = fwd_kwargs(cfg, inp)
    args.update(kw)
    out, fin = kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], **args)
    torch.cuda.synchronize()
    return out, fin


def oracle_problem(cfg: KdaConfig, inp: dict, q=None, k=None, v=None, g=None, beta=None, cu=None):
    """fp64 oracle problem from (CPU copies of) the inputs, flattened to [T, H, D]."""
    q = inp["q"] if q is None else q
    k = inp["k"] if k is None else k
    v = inp["v"] if v is None else v
    g = inp["g"] if g is None else g
    beta = inp["beta"] if beta is None else beta
    H = q.shape[-2]
    T = q.numel() // (H * q.shape[-1])
    if cu is None:
        if inp.get("cu_seqlens") is not None:
            cu = inp["cu_seqlens"].cpu().numpy()
        else:
            Tb = q.shape[1] if q.dim() == 4 else T
            cu = np.arange(0, T + 1, max(Tb, 1)) if T else np.array([0, 0])
    return oracle.Problem(q.reshape(T, H, -1), k.reshape(T, H, -1), v.reshape(T, H, -1),
                          g.reshape(T, H, -1), beta.reshape(T, H), cu_seqlens=cu,
                          scale=scale_of(cfg), eps=float(np.float32(1e-6)), a_log=inp["a_log"],
                          dt_bias=inp["dt_bias"], **oracle_kwargs(cfg))


def cpu(inp: dict) -> dict:
    return {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def make(cfg: KdaConfig, device="cpu", seed=None) -> dict:
    return make_inputs(cfg, device=device, seed=seed)
