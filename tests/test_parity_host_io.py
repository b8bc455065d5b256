"""GPU tests of kda_chunk_fwd_host: host-resident inputs streamed through the
GPU in blocks.  Blocks end on chunk boundaries and the fp32 state is handed
over as is, so the results equal kda_chunk_fwd's bit for bit; one small case
is also compared with the fp64 oracle."""
import pytest
import torch

import oracle
from chunked_kimi_delta_gb300.inputs import KdaConfig
from kda_testutil import check, fwd_kwargs, gpu_fwd, make, oracle_problem, to_cuda

pytestmark = pytest.mark.gpu


def _host(inp):
    return {n: inp[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta")}


def _host_fwd(kda, cfg, inp, **kw):
    h = _host(inp)
    args = fwd_kwargs(cfg, inp)
    args.update(kw)
    args.pop("cu_seqlens")
    out, fin = kda.kda_chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], **args)
    torch.cuda.synchronize()
    return out, fin


@pytest.mark.parametrize("dtype,d,T", [("bf16", 128, 2500), ("bf16", 128, 1024), ("bf16", 128, 100),
                                       ("f32", 64, 1100), ("bf16", 64, 2049)])
def test_host_io_equals_device_forward(cuda_lib, dtype, d, T):
    cfg = KdaConfig("host", B=2, T=T, H=3, dk=d, dv=d, dtype=dtype, initial_state=True,
                    use_exp2=True, seed=T)
    inp = to_cuda(make(cfg))
    o_ref, f_ref = gpu_fwd(cuda_lib, cfg, inp)
    out, fin = _host_fwd(cuda_lib, cfg, inp)
    assert not out.is_cuda and out.is_pinned()
    assert torch.equal(out, o_ref.cpu())
    assert torch.equal(fin, f_ref)


def test_host_io_without_final_state_and_initial_state(cuda_lib):
    """The state crosses blocks through the workspace when final_state is not
    requested; a missing initial state starts from zero."""
    cfg = KdaConfig("host0", B=3, T=2200, H=2, dk=128, dv=128, dtype="bf16", seed=7)
    inp = to_cuda(make(cfg))
    o_ref, _ = gpu_fwd(cuda_lib, cfg, inp)
    out, fin = _host_fwd(cuda_lib, cfg, inp, output_final_state=False)
    assert fin is None
    assert torch.equal(out, o_ref.cpu())


def test_host_io_against_oracle(cuda_lib):
    cfg = KdaConfig("host_oracle", B=1, T=1300, H=2, dk=128, dv=128, dtype="bf16",
                    initial_state=True, seed=21)
    inp_c = make(cfg)
    out, fin = _host_fwd(cuda_lib, cfg, to_cuda(inp_c))
    p = oracle_problem(cfg, inp_c)
    o_ref, f_ref = oracle.chunk_fwd(p, inp_c["initial_state"])
    check(out.reshape(o_ref.shape), o_ref, "bf16", "o")
    check(fin, f_ref, "bf16", "final_state")


def test_host_io_stream_order(cuda_lib):
    """Two calls in a row on the same stream: the second reuses the first's
    outputs only after it, and both match the device forward."""
    cfg = KdaConfig("host_ord", B=2, T=1500, H=2, dk=128, dv=128, dtype="bf16",
                    initial_state=True, seed=5)
    inp = to_cuda(make(cfg))
    o1, f1 = gpu_fwd(cuda_lib, cfg, inp)
    o2, f2 = gpu_fwd(cuda_lib, cfg, inp, initial_state=f1)
    h = _host(inp)
    args = fwd_kwargs(cfg, inp)
    args.pop("cu_seqlens")
    a1, g1 = cuda_lib.kda_chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], **args)
    args["initial_state"] = g1
    a2, g2 = cuda_lib.kda_chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], **args)
    torch.cuda.synchronize()
    assert torch.equal(a1, o1.cpu()) and torch.equal(a2, o2.cpu()) and torch.equal(g2, f2)
