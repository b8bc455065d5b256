"""Seeded synthetic inputs for the KDA forward, summary, scan and state copy.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  The same tensors feed the CUDA library and the fp64
oracle, so both see identical bytes.

Distributions (per the workload descriptions): q, k, v ~ N(0,1), rounded to
bf16 where the workload is bf16 (q and k are L2-normalised by the method);
beta logits b ~ N(0,1) (the method applies the sigmoid); raw gate input
x ~ N(0,1), a_log ~ U(-4, 0) per head (another range for the strong-decay
cases), dt_bias ~ N(0, 0.1) per (head,
channel) (the method applies g = -exp(a_log) softplus(x + dt_bias));
initial states ~ N(0, 0.1).  Draw order from one generator: sequence lengths
(varlen only), q, k, v, x, b, a_log, dt_bias, initial state, then pool rows,
indices and flags.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class KdaConfig:
    name: str
    B: int = 1
    T: int = 256
    H: int = 2
    dk: int = 64
    dv: int = 64
    dtype: str = "f32"               # q/k/v/out dtype: "f32" or "bf16"
    gate_in_kernel: bool = True      # pass raw x + a_log/dt_bias
    beta_sigmoid: bool = True        # pass beta logits
    use_exp2: bool = False           # base-2 internal decay
    l2norm: bool = True
    initial_state: bool = False
    seq_lens: Optional[tuple] = None  # varlen (TND) when set; B must be 1
    varlen_count: int = 0            # draw this many lengths ~ U{len_lo..len_hi}
    len_lo: int = 64
    len_hi: int = 8192
    num_segments: int = 0            # segment mode: equal segments per sequence
    pool_rows: int = 0               # state pool size for gather/scatter
    a_log_const: Optional[float] = None   # slow-decay variant
    a_log_range: tuple = (-4.0, 0.0)      # a_log ~ U(lo, hi) per head otherwise
    beta_logit_mean: float = 0.0
    seed: int = 0

    def replace(self, **kw) -> "KdaConfig":
        return dataclasses.replace(self, **kw)


# The five workloads, plus the slow-decay segment variant.
CONFIGS = {
    # B=1, T=256, H=2, d=64, fp32, initial state given.
    "tiny_f32": KdaConfig("tiny_f32", B=1, T=256, H=2, dk=64, dv=64, dtype="f32",
                          initial_state=True),
    # B=2, T=4096, H=16, d=128, bf16 q/k/v, fp32 gate/beta/state, no initial state.
    "mid_bf16": KdaConfig("mid_bf16", B=2, T=4096, H=16, dk=128, dv=128, dtype="bf16"),
    # Kimi-Linear-shaped training batch: B=4, T=8192, H=32, d=128, base-2 gate in kernel.
    "kimi_bf16": KdaConfig("kimi_bf16", B=4, T=8192, H=32, dk=128, dv=128, dtype="bf16",
                           use_exp2=True, initial_state=True),
    # Varlen packed prefill: 64 sequences, lengths ~ U{64..8192}, pool [512,H,128,128].
    "varlen_bf16": KdaConfig("varlen_bf16", B=1, T=0, H=32, dk=128, dv=128, dtype="bf16",
                             use_exp2=True, varlen_count=64, pool_rows=512),
    # Long sequence, segment mode: T = 2^20, H=8, 16 equal segments.
    "long_segment_bf16": KdaConfig("long_segment_bf16", B=1, T=1 << 20, H=8, dk=128, dv=128,
                                   dtype="bf16", use_exp2=True, num_segments=16),
    # Slow decay keeps the cumulative transition M far from zero.
    "long_segment_slow": KdaConfig("long_segment_slow", B=1, T=1 << 16, H=8, dk=128, dv=128,
                                   dtype="bf16", use_exp2=True, num_segments=16,
                                   a_log_const=-12.0, beta_logit_mean=-7.0),
}


_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def make_inputs(cfg: KdaConfig, device="cpu", seed: Optional[int] = None) -> dict:
    """Draw one problem.  Returns a dict of tensors on ``device``:

    q, k [B,T,H,dk] or [T_total,H,dk] (varlen), v likewise with dv, all in
    cfg.dtype; g fp32 [.., H, dk] (raw gate input x, or a natural-log decay when
    ``gate_in_kernel`` is off); beta fp32 [.., H] (logits, or beta itself when
    ``beta_sigmoid`` is off); a_log fp32 [H]; dt_bias fp32 [H, dk];
    initial_state fp32 [N,H,dk,dv] or None; cu_seqlens int32 [N+1] or None;
    seg_bounds int32 [S+1] (per sequence) when segment mode; pool fp32
    [pool_rows,H,dk,dv], idx int32 [N], flags bool [N] when a pool is used.
    """
    seed = cfg.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    f32 = torch.float32

    def randn(*shape, std=1.0, mean=0.0):
        return torch.randn(*shape, generator=gen, device=device, dtype=f32) * std + mean

    def rand(*shape):
        return torch.rand(*shape, generator=gen, device=device, dtype=f32)

    H, dk, dv = cfg.H, cfg.dk, cfg.dv
    cu = None
    lens = None
    if cfg.seq_lens is not None or cfg.varlen_count:
        if cfg.seq_lens is not None:
            lens = torch.tensor(cfg.seq_lens, dtype=torch.int64)
        else:
            lens = torch.randint(cfg.len_lo, cfg.len_hi + 1, (cfg.varlen_count,), generator=gen,
                                 device=device).to("cpu")
        cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(lens, 0)
        lead = (int(cu[-1]),)
        N = len(lens)
    else:
        lead = (cfg.B, cfg.T)
        N = cfg.B
    dt = torch_dtype(cfg.dtype)
    q = randn(*lead, H, dk).to(dt)
    k = randn(*lead, H, dk).to(dt)
    v = randn(*lead, H, dv).to(dt)
    if cfg.gate_in_kernel:
        g = randn(*lead, H, dk)
    else:
        # a natural-log decay drawn directly: g = -0.5 |N(0,1)| per element
        g = -0.5 * randn(*lead, H, dk).abs()
    if cfg.beta_sigmoid:
        beta = randn(*lead, H, mean=cfg.beta_logit_mean)
    else:
        beta = rand(*lead, H)
    if cfg.a_log_const is not None:
        a_log = torch.full((H,), cfg.a_log_const, dtype=f32, device=device)
        _ = rand(H)  # keep the draw order
    else:
        lo, hi = cfg.a_log_range
        a_log = rand(H) * (hi - lo) + lo
    dt_bias = randn(H, dk, std=0.1)
    S0 = randn(N, H, dk, dv, std=0.1) if cfg.initial_state else None
    out = dict(q=q, k=k, v=v, g=g, beta=beta, a_log=a_log, dt_bias=dt_bias,
               initial_state=S0, cu_seqlens=None if cu is None else cu.to(torch.int32).to(device),
               seg_bounds=None, pool=None, idx=None, flags=None, seq_lens=lens)
    if cfg.num_segments:
        T = cfg.T
        S = cfg.num_segments
        out["seg_bounds"] = torch.tensor([(T * j) // S for j in range(S + 1)], dtype=torch.int32,
                                         device=device)
    if cfg.pool_rows:
        pool = randn(cfg.pool_rows, H, dk, dv, std=0.1)
        perm = torch.randperm(cfg.pool_rows, generator=gen, device=device)[:N]
        u = rand(N)
        idx = torch.where(u < 0.05, torch.full_like(perm, -1), perm).to(torch.int32)
        flags = ~((u >= 0.05) & (u < 0.10))
        out.update(pool=pool, idx=idx, flags=flags)
    return out


def oracle_kwargs(cfg: KdaConfig) -> dict:
    """The method flags of ``cfg`` as keyword booleans (no arithmetic)."""
    return dict(l2norm=cfg.l2norm, beta_sigmoid=cfg.beta_sigmoid,
                gate_in_kernel=cfg.gate_in_kernel, use_exp2=cfg.use_exp2)


def make_cotangents(cfg: KdaConfig, inputs: dict, device="cpu", seed: Optional[int] = None) -> dict:
    """Seeded cotangents of a backward: d_out ~ N(0,1) with v's shape in
    cfg.dtype, d_final_state ~ N(0, 0.1) fp32 [N, H, dk, dv]."""
    seed = (cfg.seed if seed is None else seed) + 7919
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    v = inputs["v"]
    N = (inputs["cu_seqlens"].numel() - 1) if inputs.get("cu_seqlens") is not None else cfg.B
    d_out = torch.randn(*v.shape, generator=gen, device=device, dtype=torch.float32)
    d_fin = torch.randn(N, cfg.H, cfg.dk, cfg.dv, generator=gen, device=device,
                        dtype=torch.float32) * 0.1
    return dict(d_out=d_out.to(torch_dtype(cfg.dtype)), d_final_state=d_fin)
