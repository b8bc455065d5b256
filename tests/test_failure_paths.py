"""Failure detection without faulting or hanging the GPU.

Device side: every wait of the tensor-core kernels is bounded; when one
gives up, the kernel records KDA_ERR_DEVICE_TIMEOUT in the workspace's error
word, lets the copies it started land, frees its tensor memory and returns.
The test-only flag KDA_TEST_WAIT_TIMEOUT makes the chain kernel wait once on a
barrier that nothing completes (1 ms limit), so that path runs for real; the
status must then be reported, cleared by the read, and the next call on the
same workspace must be correct.  Host side: a call that fails a check must
launch nothing ("vllm-ascend KDA prefill state copy": prepare fails closed) -
its outputs keep their previous contents."""
import ctypes

import pytest
import torch

import chunked_kimi_delta_gb300 as kda
import oracle
from chunked_kimi_delta_gb300.inputs import KdaConfig
from kda_testutil import check, fwd_kwargs, make, oracle_problem, to_cuda

pytestmark = pytest.mark.gpu

CFG = KdaConfig("fail", B=1, T=300, H=2, dk=128, dv=128, dtype="bf16", use_exp2=True,
                initial_state=True, seed=33)


def _args(inp):
    return (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])


def test_device_wait_timeout_is_reported_and_the_next_call_is_correct(cuda_lib):
    inp_c = make(CFG)
    inp = to_cuda(inp_c)
    kw = fwd_kwargs(CFG, inp)
    a = kda.make_fwd_args(*_args(inp), **{**kw, "out": torch.empty_like(inp["v"])})
    ws = torch.empty(kda.load_library().kda_chunk_fwd_workspace_size(ctypes.byref(a)),
                     dtype=torch.uint8, device="cuda")
    cuda_lib.kda_chunk_fwd(*_args(inp), workspace=ws, extra_flags=kda.KDA_TEST_WAIT_TIMEOUT, **kw)
    assert kda.kda_get_device_status(ws) == kda.KDA_ERR_DEVICE_TIMEOUT
    assert kda.kda_get_device_status(ws) == kda.KDA_OK  # the read cleared it
    out, fin = cuda_lib.kda_chunk_fwd(*_args(inp), workspace=ws, **kw)
    assert kda.kda_get_device_status(ws) == kda.KDA_OK
    o_ref, f_ref = oracle.chunk_fwd(oracle_problem(CFG, inp_c), inp_c["initial_state"])
    check(out.reshape(o_ref.shape), o_ref, "bf16", "o after a timeout")
    check(fin, f_ref, "bf16", "final_state after a timeout")


def test_static_scratch_timeout_is_reported(cuda_lib):
    """The allocation-free forward's callers read the status of its array."""
    inp = to_cuda(make(CFG))
    kw = fwd_kwargs(CFG, inp)
    ref_out, ref_fin = cuda_lib.kda_chunk_fwd(*_args(inp), **kw)
    cuda_lib.kda_chunk_fwd_static_scratch(*_args(inp), extra_flags=kda.KDA_TEST_WAIT_TIMEOUT, **kw)
    assert kda.kda_static_scratch_status() == kda.KDA_ERR_DEVICE_TIMEOUT
    out, fin = cuda_lib.kda_chunk_fwd_static_scratch(*_args(inp), **kw)
    assert kda.kda_static_scratch_status() == kda.KDA_OK
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)


def test_failed_checks_launch_nothing(cuda_lib):
    """A workspace one byte short, and a misaligned q, are refused by the
    library before any launch: the output and final state keep their canary
    contents."""
    inp = to_cuda(make(CFG))
    kw = fwd_kwargs(CFG, inp)
    out = torch.full_like(inp["v"], 7.0)
    fin = torch.full((1, CFG.H, CFG.dk, CFG.dv), 7.0, device="cuda")
    lib = kda.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    a = kda.make_fwd_args(*_args(inp), **{**kw, "out": out, "final_state": fin})
    need = lib.kda_chunk_fwd_workspace_size(ctypes.byref(a))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), need - 1
    assert lib.kda_chunk_fwd(ctypes.byref(a), stream) == kda.KDA_ERR_WORKSPACE
    flat = torch.empty(inp["q"].numel() + 1, dtype=inp["q"].dtype, device="cuda")
    q_mis = flat[1:].view(inp["q"].shape)  # 2 bytes off a 16-byte boundary
    q_mis.copy_(inp["q"])
    b = kda.make_fwd_args(q_mis, *_args(inp)[1:], **{**kw, "out": out, "final_state": fin})
    b.workspace, b.workspace_bytes = ws.data_ptr(), need
    assert lib.kda_chunk_fwd(ctypes.byref(b), stream) == kda.KDA_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((fin == 7.0).all())
