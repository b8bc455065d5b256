#!/usr/bin/env python3
"""Benchmark of the chunked KDA forward on GB300.

One step = one pass of the hot path over one batch of the Kimi-Linear-shaped
bf16 workload (B=4, T=8192, H=32, d_k=d_v=128; gate activation, base-2 decay,
beta sigmoid and Q/K L2 norm in kernel):
  gather the 4 initial states from a [512, 32, 128, 128] fp32 state pool,
  kda_chunk_fwd (preprocess, intra-chunk, inter-chunk chain, output),
  scatter the 4 final states back to the pool.
The segment path (summary -> prefix scan -> segment finish) is timed on the
long-sequence workload (T = 2^20, H = 8, 16 segments) and reported beside it.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle instead, on a bounded sample of the same workload.
Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "chunk-KDA fwd tokens/s and TFLOP/s on 1 GB300 (% of bf16 tensor peak)"
WORKLOAD = "kimi_bf16"
# Algorithmic work per token-head at d_k = d_v = d, BT = 64 (lower triangles
# counted once): 6 d_k d_v + BT (3 d_k + 2 d_v) flop; bytes: q, k, v, o in bf16
# (2 d each), the raw gate in fp32 (4 d_k), beta in fp32 (4).
def alg_flops_per_token_head(dk, dv, bt=64):
    return 6 * dk * dv + bt * (3 * dk + 2 * dv)


def alg_bytes_per_token_head(dk, dv):
    return 2 * dk * 2 + 2 * dv * 2 + 4 * dk + 4


def intra_alg_bytes_per_token_head(dk, dv):   # inputs the intra-chunk stage must read
    return 2 * dk * 2 + 2 * dv + 4 * dk + 4


def dist_env():
    """(world, rank, local_rank) from the torchrun environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank gets the max (one scalar all-reduce)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_inputs(cfg, device, rank: int) -> dict:
    """The inputs of one rank: the workload drawn with the rank as its seed,
    so that the ranks process independent batches (weak scaling, no
    data-path collective)."""
    from chunked_kimi_delta_gb300.inputs import make_inputs
    return make_inputs(cfg, device=device, seed=rank)


def whole_job_rate(units_per_rank_step: float, world: int, steps: int, ms: float) -> float:
    """Units of all ranks per second over the slowest rank's time (weak scaling)."""
    return units_per_rank_step * world * steps / (ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
        load = [x for x in sm if smax and x > 0.3 * smax] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- reference arm

def cpu_oracle_sample(cfg, inp_cpu, units, ntokens, nthreads=0):
    """Times the fp64 oracle on `units` (b, h) pairs over the first `ntokens`
    tokens.  Returns (seconds, token_heads, threads)."""
    import numpy as np
    import oracle
    from chunked_kimi_delta_gb300.inputs import oracle_kwargs
    b = units[0][0]
    heads = [h for (_, h) in units]
    q = inp_cpu["q"][b:b + 1, :ntokens][:, :, heads]
    k = inp_cpu["k"][b:b + 1, :ntokens][:, :, heads]
    v = inp_cpu["v"][b:b + 1, :ntokens][:, :, heads]
    g = inp_cpu["g"][b:b + 1, :ntokens][:, :, heads]
    be = inp_cpu["beta"][b:b + 1, :ntokens][:, :, heads]
    H = len(heads)
    p = oracle.Problem(q.reshape(ntokens, H, -1), k.reshape(ntokens, H, -1),
                       v.reshape(ntokens, H, -1), g.reshape(ntokens, H, -1),
                       be.reshape(ntokens, H), cu_seqlens=[0, ntokens],
                       scale=float(np.float32(cfg.dk ** -0.5)), a_log=inp_cpu["a_log"][heads],
                       dt_bias=inp_cpu["dt_bias"][heads], **oracle_kwargs(cfg))
    S0 = inp_cpu["initial_state"][b:b + 1][:, heads] if inp_cpu["initial_state"] is not None else None
    threads = oracle.max_threads(nthreads)
    t = time.perf_counter()
    oracle.chunk_fwd(p, S0, nthreads=nthreads)
    return time.perf_counter() - t, ntokens * H, threads


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() in ("Model name", "Model"):
                name = ln.split(":", 1)[1].strip()
                if name and not name.isdigit():
                    return name
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def run_reference(args, rank):
    """The oracle timed on the host cores on the same sample as the GPU line's
    cpu_baseline: one step = one whole sequence of the workload (all H heads
    x T tokens, OpenMP over the heads)."""
    if rank != 0:
        return
    from chunked_kimi_delta_gb300.inputs import CONFIGS, make_inputs
    cfg = CONFIGS[args.workload]
    one = cfg.replace(B=1)   # one sequence of the workload's shape and distributions
    inp = make_inputs(one, device="cpu")
    units = [(0, h) for h in range(cfg.H)]
    for _ in range(args.warmup):
        cpu_oracle_sample(one, inp, units[:2], 256)
    secs, th, threads = 0.0, 0, 1
    for _ in range(args.steps):
        s, n, threads = cpu_oracle_sample(one, inp, units, cfg.T)
        secs += s
        th += n
    tok_s = th / secs / cfg.H   # tokens/s of the full H-head workload
    tflops = th * alg_flops_per_token_head(cfg.dk, cfg.dv) / secs / 1e12
    sample = (f"fp64 oracle, one whole sequence per step: all {cfg.H} heads x {cfg.T} tokens "
              f"(token-heads/s divided by H={cfg.H}); the GPU line's cpu_baseline times the same "
              f"unit on the batch's own sequences")
    line = {"impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_desc(cfg), "tflops": tflops,
            "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model(), "nproc": os.cpu_count()},
            "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def step_stats(ms_list):
    """median / min / p90 / mean of per-step times (ms)."""
    xs = sorted(ms_list)
    p90 = xs[min(len(xs) - 1, int(round(0.9 * (len(xs) - 1))))]
    return {"median": statistics.median(xs), "min": xs[0], "p90": p90,
            "mean": sum(xs) / len(xs), "n": len(xs)}


def config_desc(cfg):
    return {"workload": (f"{cfg.name}: B={cfg.B} T={cfg.T} H={cfg.H} d_k={cfg.dk} d_v={cfg.dv} "
                         f"bf16 q/k/v/o, fp32 gate/beta/state, gate+exp2+sigmoid+L2 in kernel, "
                         f"initial states gathered from a 512-row fp32 pool, final states "
                         f"scattered back"),
            "B": cfg.B, "T": cfg.T, "H": cfg.H, "dk": cfg.dk, "dv": cfg.dv, "chunk": 64,
            "l2_policy": (f"inputs ({cfg.B * cfg.T * cfg.H * intra_alg_bytes_per_token_head(cfg.dk, cfg.dv) / 1e9:.2f}"
                          f" GB) larger than L2 (129 MB); no flush")}


# ---------------------------------------------------------------- our arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-segment", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the lines of the mid and varlen workloads")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="fixed-length bf16 d=128 workload of the main line (default: the "
                         "Kimi-shaped batch; a smaller one serves profiling)")
    ap.add_argument("--bwd-config", default=None,
                    help="named workload of the bwd line (default: the forward's workload)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank)

    import torch
    import torch.distributed as dist
    import chunked_kimi_delta_gb300 as kda
    from chunked_kimi_delta_gb300.inputs import CONFIGS, make_inputs

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    lib = kda.load_library()
    dev = torch.device("cuda", local)
    hbm_peak, tc_peak, tc_sus, peak_src = load_peaks()

    cfg = CONFIGS[args.workload]
    if cfg.seq_lens or cfg.varlen_count or cfg.dtype != "bf16" or cfg.dk != 128 or cfg.num_segments:
        raise SystemExit("--workload takes a fixed-length bf16 d=128 workload")
    inp = rank_inputs(cfg, dev, rank)
    H, K, V = cfg.H, cfg.dk, cfg.dv
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + rank)
    pool = torch.randn(512, H, K, V, generator=gen, device=dev) * 0.1
    idx = torch.randperm(512, generator=gen, device=dev)[:cfg.B].to(torch.int32)
    S0 = torch.empty(cfg.B, H, K, V, device=dev)
    scale = float(K ** -0.5)
    fa, out, fin, ws = kda.prepare_chunk_fwd(
        inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=scale, a_log=inp["a_log"],
        dt_bias=inp["dt_bias"], initial_state=S0, l2norm_qk=True, beta_sigmoid=True,
        gate_in_kernel=True, use_exp2=True)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    stages = kda.kda_chunk_fwd_stages(fa)
    # one event set per timed step, read after the timed region
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
               for _ in range(args.steps)]
    for es in ev_sets:
        for e in es:
            e.record(stream)

    def step(events=None):
        kda.kda_state_gather(pool, idx, packed=S0, stream=stream)
        if events is not None:
            kda.kda_chunk_fwd_profiled(fa, events, stream=stream)
        else:
            st = lib.kda_chunk_fwd(ctypes.byref(fa), sp)
            if st:
                raise kda.KdaError(st, "kda_chunk_fwd")
        kda.kda_state_scatter(pool, idx, fin, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = kda.kda_get_device_status(ws)
    if status:
        raise kda.KdaError(status, "device status after warm-up")

    # timed region: whole steps, CUDA events on the launching stream; the
    # per-stage events of each forward give each kernel's duration
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    t0.record(stream)
    for i in range(args.steps):
        step_ev[i].record(stream)
        step(ev_sets[i])
    step_ev[args.steps].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_per_step = ms / args.steps
    tokens = cfg.B * cfg.T
    token_heads = tokens * H
    value = whole_job_rate(tokens, world, args.steps, ms)
    tflops = token_heads * world * args.steps * alg_flops_per_token_head(K, V) / (ms / 1e3) / 1e12
    stage_avg = [sum(es[j].elapsed_time(es[j + 1]) for es in ev_sets) / args.steps
                 for j in range(len(stages))]
    status = kda.kda_get_device_status(ws)
    if status:
        raise kda.KdaError(status, "device status after timed region")

    # dominant kernel: its algorithmic bytes per launch / its average duration
    dom = max(range(len(stages)), key=lambda i: stage_avg[i])
    dom_name = stages[dom]
    state_bytes = 2 * 4 * K * V * cfg.B * H          # initial + final state
    if dom_name.startswith("intra") or dom_name == "tc_prep":
        dom_bytes = intra_alg_bytes_per_token_head(K, V) * token_heads
    elif dom_name.startswith("inter") or dom_name == "tc_chain":
        dom_bytes = 2 * V * token_heads + state_bytes  # the output o and the states
    else:
        dom_bytes = alg_bytes_per_token_head(K, V) * token_heads + state_bytes
    achieved = dom_bytes / (stage_avg[dom] / 1e3) / 1e9
    fwd_ms = sum(stage_avg)
    fwd_bytes = alg_bytes_per_token_head(K, V) * token_heads + state_bytes
    traffic = load_traffic(dom_name)

    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": config_desc(cfg),
        "tflops": tflops, "tensor_peak_frac": tflops / tc_peak,
        "hbm_frac_fwd": fwd_bytes / (fwd_ms / 1e3) / 1e9 / hbm_peak,
        "peaks": {"hbm_gbs": hbm_peak, "bf16_tflops": tc_peak, "source": peak_src},
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "alg_bytes_per_launch": dom_bytes, "avg_launch_ms": stage_avg[dom],
                     "peak_source": peak_src},
        "stages_ms": dict(zip(stages, stage_avg)),
        "step_ms": step_stats([step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps)]),
        "gpu_launches": args.steps * (len(stages) + 2),
        "clocks": clk,
    }
    if rank == 0 and not args.no_segment:
        result["segment_mode"] = bench_segment(kda, dev, stream)
    if rank == 0 and not args.no_decode:
        result["decode"] = bench_decode(kda, dev, stream, hbm_peak)
    if rank == 0 and not args.no_bwd:
        if args.bwd_config and args.bwd_config != cfg.name:
            from chunked_kimi_delta_gb300.inputs import CONFIGS, make_inputs
            bcfg = CONFIGS[args.bwd_config]
            if bcfg.seq_lens or bcfg.varlen_count or bcfg.dtype != "bf16":
                raise SystemExit("--bwd-config takes a fixed-length bf16 workload")
            binp = make_inputs(bcfg, device=dev)
            result["bwd"] = bench_bwd(kda, lib, bcfg, binp, binp.get("initial_state"), dev, stream, hbm_peak)
            del binp
        else:
            result["bwd"] = bench_bwd(kda, lib, cfg, inp, S0, dev, stream, hbm_peak)
    if rank == 0 and not args.no_bwd and not args.no_segment:
        result["segment_mode_bwd"] = bench_segment_bwd(kda, dev, stream)
    if rank == 0 and not args.no_configs:
        result["config_lines"] = {name: bench_workload(kda, lib, CONFIGS[name], dev, stream, hbm_peak, tc_peak)
                                  for name in ("mid_bf16", "varlen_bf16")}
        # the same batch under strong gate decay (a_log ~ U(1, 3): about -2 to -60 nats per
        # token), where the chunks whose 16-token sub-blocks decay past the factored range are
        # recomputed exactly; reported with the share of such (chunk, head) items
        strong = cfg.replace(name=cfg.name + "_strong_decay", a_log_range=(1.0, 3.0))
        line = bench_workload(kda, lib, strong, dev, stream, hbm_peak, tc_peak)
        line["strong_item_share"] = strong_item_share(strong, dev)
        result["strong_decay"] = line
    if not args.no_e2e:
        result["e2e"] = bench_e2e(kda, lib, cfg, inp, pool, idx, fa, out, fin, S0, stream, world)
    if rank == 0 and not args.no_cpu_baseline:
        inp_cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        # whole sequences of the batch (all heads, all tokens), cycling through
        # the batch rows until about 10 s of CPU work (at most 16 sequences)
        secs, th, nseq, threads = 0.0, 0, 0, 1
        while secs < 10.0 and nseq < 16:
            b = nseq % cfg.B
            s_, n_, threads = cpu_oracle_sample(cfg, inp_cpu, [(b, h) for h in range(H)], cfg.T)
            secs, th, nseq = secs + s_, th + n_, nseq + 1
        # single-threaded: 4 heads of one sequence, whole length (~1 s)
        s1, n1, _ = cpu_oracle_sample(cfg, inp_cpu, [(0, h) for h in range(4)], cfg.T, nthreads=1)
        result["cpu_baseline"] = {
            "value": th / secs / H, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle on {nseq} whole sequences of the batch (rows 0..{cfg.B - 1} in "
                      f"turn), all {H} heads x {cfg.T} tokens each ({th} token-heads, {secs:.1f} s); "
                      f"tokens/s = token-heads/s / H",
            "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "single_thread": {"value": n1 / s1 / H, "unit": "tokens/s", "cores": 1,
                              "sample": f"4 heads x {cfg.T} tokens of sequence 0 ({s1:.1f} s), "
                                        f"token-heads/s / H"}}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def load_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when there is no capture or the kernel source changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            ent = json.load(f)[kernel]
        with open(os.path.join(ROOT, ent["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != ent["source_sha256"]:
                return None
        return ent["bytes"]
    except Exception:
        return None


def bench_workload(kda, lib, cfg, dev, stream, hbm_peak, tc_peak, steps=50, warmup=5):
    """One forward workload other than the headline: mid_bf16 (B=2, T=4096,
    H=16, no initial state) or varlen_bf16 (64 packed sequences with states
    gathered from and scattered back to a 512-row pool, ~10% invalid rows).
    A 256 MiB buffer is written between steps (L2 flush); each step is timed
    with CUDA events, kernel durations from events between the stages."""
    import torch
    from chunked_kimi_delta_gb300.inputs import make_inputs
    inp = make_inputs(cfg, device=dev)
    H, K, V = cfg.H, cfg.dk, cfg.dv
    kw = dict(scale=float(K ** -0.5), a_log=inp["a_log"], dt_bias=inp["dt_bias"], l2norm_qk=cfg.l2norm,
              beta_sigmoid=cfg.beta_sigmoid, gate_in_kernel=cfg.gate_in_kernel, use_exp2=cfg.use_exp2)
    cu = inp["cu_seqlens"]
    pool = inp.get("pool")
    N = (cu.numel() - 1) if cu is not None else cfg.B
    S0 = torch.empty(N, H, K, V, device=dev) if pool is not None else inp["initial_state"]
    fa, out, fin, ws = kda.prepare_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                             cu_seqlens=cu, initial_state=S0, **kw)
    stages = kda.kda_chunk_fwd_stages(fa)
    sp = stream.cuda_stream

    def step(events=None):
        if pool is not None:
            kda.kda_state_gather(pool, inp["idx"], flags=inp["flags"], packed=S0, stream=stream)
        if events is not None:
            kda.kda_chunk_fwd_profiled(fa, events, stream=stream)
        else:
            st = lib.kda_chunk_fwd(ctypes.byref(fa), sp)
            if st:
                raise kda.KdaError(st, "kda_chunk_fwd")
        if pool is not None:
            kda.kda_state_scatter(pool, inp["idx"], fin, stream=stream)

    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(steps)]
    se = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for es in ev:  # the library records them by handle: create them first
        for e in es:
            e.record(stream)
    for i in range(steps):
        flush.zero_()
        se[i][0].record(stream)
        step(ev[i])
        se[i][1].record(stream)
    torch.cuda.synchronize()
    status = kda.kda_get_device_status(ws)
    if status:
        raise kda.KdaError(status, "device status")
    st = step_stats([a.elapsed_time(b) for a, b in se])
    stage_avg = [sum(e[j].elapsed_time(e[j + 1]) for e in ev) / steps for j in range(len(stages))]
    tokens = int(inp["q"].numel() // (inp["q"].shape[-2] * K))
    th = tokens * H
    n_init = N if S0 is not None else 0               # states read by the forward
    state_bytes = 4 * K * V * H * (n_init + N)        # + final states written
    dom = max(range(len(stages)), key=lambda i: stage_avg[i])
    name = stages[dom]
    if name.startswith("intra") or name == "tc_prep":
        dom_bytes = intra_alg_bytes_per_token_head(K, V) * th
    elif name.startswith("inter") or name == "tc_chain":
        dom_bytes = 2 * V * th + state_bytes
    else:
        dom_bytes = alg_bytes_per_token_head(K, V) * th
    fwd_bytes = alg_bytes_per_token_head(K, V) * th + state_bytes
    ms = st["median"]
    desc = (f"{cfg.name}: B={cfg.B} T={cfg.T} H={H} d={K} bf16" if cu is None else
            f"{cfg.name}: {N} packed sequences, {tokens} tokens (lengths U{{{cfg.len_lo}..{cfg.len_hi}}}), "
            f"H={H} d={K} bf16, states gathered from / scattered to a {cfg.pool_rows}-row fp32 pool")
    res = {"workload": desc, "tokens": tokens, "tokens_per_s": tokens / (ms / 1e3), "step_ms": st,
           "tflops": th * alg_flops_per_token_head(K, V) / (ms / 1e3) / 1e12,
           "hbm_frac_step": fwd_bytes / (ms / 1e3) / 1e9 / hbm_peak,
           "stages_ms": dict(zip(stages, stage_avg)),
           "l2_policy": "256 MiB buffer written between steps (flush)",
           "roofline": {"bound": "hbm", "kernel": name, "achieved": dom_bytes / (stage_avg[dom] / 1e3) / 1e9,
                        "peak": hbm_peak, "unit": "GB/s",
                        "frac": dom_bytes / (stage_avg[dom] / 1e3) / 1e9 / hbm_peak,
                        "alg_bytes_per_launch": dom_bytes, "avg_launch_ms": stage_avg[dom]}}
    res["tensor_peak_frac"] = res["tflops"] / tc_peak
    del inp, fa, out, fin, ws, flush
    torch.cuda.empty_cache()
    return res


def strong_item_share(cfg, dev) -> float:
    """Share of (chunk, head) items with a 16-token sub-block whose decay
    exceeds 96 log2 units in some channel (the items the library recomputes
    exactly), from the workload's own gate: g = -exp(a_log) softplus(x +
    dt_bias), summed over each sub-block."""
    import torch
    from chunked_kimi_delta_gb300.inputs import make_inputs
    inp = make_inputs(cfg, device=dev)
    g = -torch.exp(inp["a_log"])[:, None] * torch.nn.functional.softplus(inp["g"] + inp["dt_bias"])
    B, T, H, K = g.shape
    sub = g.reshape(B, T // 16, 16, H, K).sum(2) * 1.4426950408889634   # [B, T/16, H, K]
    strong_sub = (-sub > 96.0).any(-1)                                    # [B, T/16, H]
    item = strong_sub.reshape(B, T // 64, 4, H).any(2)                    # [B, T/64, H]
    share = float(item.float().mean())
    del inp, g, sub
    return share


def bench_decode(kda, dev, stream, hbm_peak, steps=50, warmup=5):
    """Recurrent decode on pool states: 64 sequences x 32 heads x d=128, one
    new token each, states read from and written back to a 512-row fp32 pool
    in place.  The state traffic bounds it: 2 x 64 KB per (sequence, head)."""
    import torch
    N, T, H, K, V, rows = 64, 1, 32, 128, 128, 512
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    bf = torch.bfloat16
    q = torch.randn(N, T, H, K, generator=gen, device=dev).to(bf)
    k = torch.randn(N, T, H, K, generator=gen, device=dev).to(bf)
    v = torch.randn(N, T, H, V, generator=gen, device=dev).to(bf)
    g = torch.randn(N, T, H, K, generator=gen, device=dev)
    beta = torch.randn(N, T, H, generator=gen, device=dev)
    a_log = torch.randn(H, generator=gen, device=dev) * 0.5 - 1.0
    dt_bias = torch.randn(H, K, generator=gen, device=dev) * 0.1
    pool = torch.randn(rows, H, K, V, generator=gen, device=dev) * 0.1
    idx = torch.randperm(rows, generator=gen, device=dev)[:N].to(torch.int32)
    out = torch.empty(N, T, H, V, dtype=bf, device=dev)
    kw = dict(scale=float(K ** -0.5), a_log=a_log, dt_bias=dt_bias, l2norm_qk=True,
              beta_sigmoid=True, gate_in_kernel=True, out=out, stream=stream)
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)   # > L2 between steps
    for _ in range(warmup):
        kda.kda_recurrent_step(q, k, v, g, beta, pool, idx, **kw)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        kda.kda_recurrent_step(q, k, v, g, beta, pool, idx, **kw)
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    state_bytes = 2 * N * H * K * V * 4
    io_bytes = N * T * H * (2 * K * 2 + V * 2 + K * 4 + 4 + V * 2)
    gbs = (state_bytes + io_bytes) / (ms / 1e3) / 1e9
    return {"workload": f"decode: {N} sequences x {H} heads, d={K}, {T} token each, bf16 q/k/v/o, "
                        f"fp32 states in a {rows}-row pool (read and written in place)",
            "tokens_per_s": N * T / (ms / 1e3), "ms_per_step": ms, "steps": steps,
            "l2_policy": "256 MiB buffer written between steps (flush)",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "alg_bytes_per_launch": state_bytes + io_bytes}}


def bwd_alg_bytes_per_token_head(dk, dv):
    """Reads q, k, v, d_out (bf16), gate, beta (fp32); writes dq, dk, dv (bf16),
    dg, dbeta (fp32)."""
    return (2 * dk * 2 + dv * 2 + dv * 2 + 4 * dk + 4) + (2 * dk * 2 + dv * 2 + 4 * dk + 4)


def bench_bwd(kda, lib, cfg, inp, S0, dev, stream, hbm_peak, steps=5, warmup=3):
    """Backward of a workload (by default the forward's: B=4, T=8192, H=32,
    d=128, bf16): all gradients (q, k, v, gate input, beta logits, a_log,
    dt_bias, initial state) of <d_out, o> + <d_final, final_state>."""
    import torch
    from chunked_kimi_delta_gb300.inputs import make_cotangents
    cot = make_cotangents(cfg, inp, device=dev)
    K, V, H = cfg.dk, cfg.dv, cfg.H
    b, grads, ws = kda.prepare_chunk_bwd(
        inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cot["d_out"],
        d_final_state=cot["d_final_state"], initial_state=S0, scale=float(K ** -0.5),
        a_log=inp["a_log"], dt_bias=inp["dt_bias"], l2norm_qk=True, beta_sigmoid=True,
        gate_in_kernel=True, use_exp2=True)
    sp = stream.cuda_stream

    def one():
        st = lib.kda_chunk_bwd(ctypes.byref(b), sp)
        if st:
            raise kda.KdaError(st, "kda_chunk_bwd")

    for _ in range(warmup):
        one()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, e in evs:
        a.record(stream)
        one()
        e.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(e) for a, e in evs)
    th = cfg.B * cfg.T * H
    nbytes = bwd_alg_bytes_per_token_head(K, V) * th + 3 * 4 * K * V * cfg.B * H
    in_bytes = sum(t.numel() * t.element_size() for t in (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                                          cot["d_out"]))
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": f"{cfg.name} backward: B={cfg.B} T={cfg.T} H={H} d={K}, bf16 q/k/v/d_out and "
                        f"dq/dk/dv, fp32 gate/beta gradients, dA_log, ddt_bias, initial-state gradient",
            "tokens_per_s": cfg.B * cfg.T / (ms / 1e3), "ms_per_step": ms, "steps": steps,
            "launches_per_step": 6,
            "l2_policy": f"inputs ({in_bytes / 1e9:.2f} GB) " + ("larger than L2 (129 MB); no flush"
                                                                 if in_bytes > 129e6 else "fit in L2: no flush"),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "alg_bytes_per_launch": nbytes,
                         "scope": "whole backward call"}}


def bench_segment_bwd(kda, dev, stream, steps=1, warmup=1):
    """Segment-mode backward on the long-sequence workload (T = 2^20, H = 8,
    16 segments): forward summary -> scan -> backward summary -> reverse
    scan -> per-segment backward, all gradients."""
    import torch
    from chunked_kimi_delta_gb300.inputs import CONFIGS, make_cotangents, make_inputs
    cfg = CONFIGS["long_segment_bf16"]
    inp = make_inputs(cfg, device=dev)
    cot = make_cotangents(cfg, inp, device=dev)
    T, H, K, V = cfg.T, cfg.H, cfg.dk, cfg.dv
    S = cfg.num_segments
    sb = inp["seg_bounds"]
    kw = dict(scale=float(K ** -0.5), a_log=inp["a_log"], dt_bias=inp["dt_bias"], l2norm_qk=True,
              beta_sigmoid=True, gate_in_kernel=True, use_exp2=True)
    flat = lambda x: x.reshape(T, *x.shape[2:])
    q, k, v, g, be = (flat(inp[n]) for n in ("q", "k", "v", "g", "beta"))
    dO = flat(cot["d_out"])
    M = torch.empty(S, H, K, K, device=dev)
    St = torch.empty(S, H, K, V, device=dev)
    S_in = torch.empty(S, H, K, V, device=dev)
    E = torch.empty(S, H, K, V, device=dev)
    dS_out = torch.empty(S, H, K, V, device=dev)
    dS0 = torch.empty(H, K, V, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    bargs = {}

    def one(rec):
        if rec:
            ev[0].record(stream)
        kda.kda_segment_summary(q, k, v, g, be, sb, M=M, S_tilde=St, stream=stream, **kw)
        kda.kda_state_prefix_scan(M, St, None, S_in=S_in, stream=stream)
        if rec:
            ev[1].record(stream)
        kda.kda_segment_bwd_summary(q, k, v, g, be, dO, sb, E=E, stream=stream, **kw)
        if rec:
            ev[2].record(stream)
        kda.kda_state_grad_scan(M, E, cot["d_final_state"][0], dS_out=dS_out, dS_initial=dS0,
                                stream=stream)
        if rec:
            ev[3].record(stream)
        if "b" not in bargs:
            bargs["b"] = kda.prepare_chunk_bwd(q, k, v, g, be, dO, d_final_state=dS_out,
                                               initial_state=S_in, cu_seqlens=sb, **kw)
        st = kda.load_library().kda_chunk_bwd(ctypes.byref(bargs["b"][0]), stream.cuda_stream)
        if st:
            raise kda.KdaError(st, "segment backward finish")
        if rec:
            ev[4].record(stream)

    for _ in range(warmup):
        one(False)
    torch.cuda.synchronize()
    parts = [0.0] * 4
    for _ in range(steps):
        one(True)
        ev[4].synchronize()
        for i in range(4):
            parts[i] += ev[i].elapsed_time(ev[i + 1])
    parts = [x / steps for x in parts]
    total = sum(parts)
    return {"workload": f"long_segment_bf16 backward: B=1 T={T} H={H} d={K} bf16, {S} segments, "
                        f"all gradients",
            "tokens_per_s": T / (total / 1e3), "ms_per_pass": total,
            "fwd_summary_scan_ms": parts[0], "bwd_summary_ms": parts[1], "grad_scan_ms": parts[2],
            "finish_ms": parts[3]}


def bench_segment(kda, dev, stream, steps=3, warmup=2):
    """Segment mode on the long-sequence workload: summary -> scan -> finish."""
    import torch
    from chunked_kimi_delta_gb300.inputs import CONFIGS, make_inputs
    cfg = CONFIGS["long_segment_bf16"]
    inp = make_inputs(cfg, device=dev)
    T, H, K, V = cfg.T, cfg.H, cfg.dk, cfg.dv
    S = cfg.num_segments
    sb = inp["seg_bounds"]
    kw = dict(scale=float(K ** -0.5), a_log=inp["a_log"], dt_bias=inp["dt_bias"], l2norm_qk=True,
              beta_sigmoid=True, gate_in_kernel=True, use_exp2=True)
    M = torch.empty(S, H, K, K, device=dev)
    St = torch.empty(S, H, K, V, device=dev)
    S_in = torch.empty(S, H, K, V, device=dev)
    S_fin = torch.empty(H, K, V, device=dev)
    flat = lambda x: x.reshape(T, *x.shape[2:])
    q, k, v, g, be = (flat(inp[n]) for n in ("q", "k", "v", "g", "beta"))
    # the finish reuses the chunks the summary prepared (same workspace)
    sa, _, _, ws_sum = kda.prepare_segment_summary(q, k, v, g, be, sb, M=M, S_tilde=St, **kw)
    fa, out, fin, ws = kda.prepare_chunk_fwd(q, k, v, g, be, cu_seqlens=sb, initial_state=S_in,
                                             workspace=ws_sum, extra_flags=kda.KDA_REUSE_PREP, **kw)
    lib = kda.load_library()
    sp = stream.cuda_stream
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def one(rec):
        if rec:
            ev[0].record(stream)
        st = lib.kda_segment_summary(ctypes.byref(sa), sb.data_ptr(), S, M.data_ptr(), St.data_ptr(), sp)
        if st:
            raise kda.KdaError(st, "kda_segment_summary")
        if rec:
            ev[1].record(stream)
        kda.kda_state_prefix_scan(M, St, None, S_in=S_in, S_final=S_fin, stream=stream)
        if rec:
            ev[2].record(stream)
        st = lib.kda_chunk_fwd(ctypes.byref(fa), sp)
        if st:
            raise kda.KdaError(st, "segment finish")
        if rec:
            ev[3].record(stream)

    for _ in range(warmup):
        one(False)
    torch.cuda.synchronize()
    parts = [0.0, 0.0, 0.0]
    for _ in range(steps):
        one(True)
        ev[3].synchronize()
        for i in range(3):
            parts[i] += ev[i].elapsed_time(ev[i + 1])
    parts = [x / steps for x in parts]
    total = sum(parts)
    return {"workload": f"long_segment_bf16: B=1 T={T} H={H} d={K} bf16, {S} segments",
            "tokens_per_s": T / (total / 1e3), "ms_per_pass": total,
            "summary_ms": parts[0], "scan_ms": parts[1], "finish_ms": parts[2],
            "tflops_alg": T * H * alg_flops_per_token_head(K, V) / (total / 1e3) / 1e12}


def bench_e2e(kda, lib, cfg, inp, pool, idx, fa, out, fin, S0, stream, world, steps=3):
    """Same step through the public API with the step's inputs and output in
    page-locked host memory: kda_chunk_fwd_host streams q, k, v, gate, beta
    to the GPU and o back, overlapping the copies with the kernels."""
    import torch
    names = ["q", "k", "v", "g", "beta"]
    host = {n: torch.empty(inp[n].shape, dtype=inp[n].dtype, pin_memory=True) for n in names}
    for n in names:
        host[n].copy_(inp[n])
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    K = cfg.dk
    ha, o_host, hfin, hws = kda.prepare_chunk_fwd_host(
        host["q"], host["k"], host["v"], host["g"], host["beta"], device=inp["q"].device,
        final_state=fin, scale=float(K ** -0.5), a_log=inp["a_log"], dt_bias=inp["dt_bias"],
        initial_state=S0, l2norm_qk=True, beta_sigmoid=True, gate_in_kernel=True, use_exp2=True)
    d2h = o_host.numel() * o_host.element_size()
    sp = stream.cuda_stream

    def step():
        kda.kda_state_gather(pool, idx, packed=S0, stream=stream)
        st = lib.kda_chunk_fwd_host(ctypes.byref(ha), sp)
        if st:
            raise kda.KdaError(st, "kda_chunk_fwd_host")
        kda.kda_state_scatter(pool, idx, fin, stream=stream)

    step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    # the host link of this machine, measured with plain copies of the same sizes
    # (one page-locked source / destination of each direction)
    dev_buf = torch.empty(h2d, dtype=torch.uint8, device=inp["q"].device)
    hbuf = torch.empty(h2d, dtype=torch.uint8, pin_memory=True)
    link = {}
    for name, dst, src, nbytes in (("h2d", dev_buf, hbuf, h2d), ("d2h", hbuf[:d2h], dev_buf[:d2h], d2h)):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        link[name + "_gbs"] = nbytes / (a.elapsed_time(b) / 1e3) / 1e9
    link_ms = 1e3 * (h2d / (link["h2d_gbs"] * 1e9) + d2h / (link["d2h_gbs"] * 1e9))
    del dev_buf, hbuf
    return {"value": cfg.B * cfg.T * world / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "host_link": {**link, "serial_copy_ms": link_ms,
                          "note": "plain copies of the step's bytes on this box, one direction at a time"},
            "api": "kda_chunk_fwd_host (host q/k/v/gate/beta/o, page-locked)"}


if __name__ == "__main__":
    main()
