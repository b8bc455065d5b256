"""Chunked Kimi Delta Attention (KDA) forward for GB300 (sm_103a).

A thin ctypes binding over the C ABI of ``include/kda.h`` (``libkda.so``,
built in-tree by :mod:`chunked_kimi_delta_gb300.build`).  The Python
functions carry the C names and only marshal arguments: every step of the
computation runs in the library's CUDA kernels.  PyTorch supplies device
memory and the current stream.  There is no fallback: when the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libkda.so")

# include/kda.h constants
KDA_OK = 0
KDA_F32, KDA_BF16 = 0, 1
KDA_I32, KDA_I64 = 0, 1
KDA_L2NORM_QK = 1 << 0
KDA_BETA_SIGMOID = 1 << 1
KDA_GATE_IN_KERNEL = 1 << 2
KDA_USE_EXP2 = 1 << 3
KDA_REUSE_PREP = 1 << 4
KDA_SAFE_GATE = 1 << 8
KDA_ALLOW_NEG_EIGVAL = 1 << 9
KDA_STATE_V_FIRST = 1 << 10
KDA_LAYOUT_HEAD_MAJOR = 1 << 11
KDA_TEST_WAIT_TIMEOUT = 1 << 30   # test only: see include/kda.h
KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_ALIGNMENT = 1, 2, 3
KDA_ERR_WORKSPACE, KDA_ERR_CUDA, KDA_ERR_DEVICE_TIMEOUT = 4, 5, 6
CHUNK = 64


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class kda_fwd_args(ctypes.Structure):
    """Mirror of ``kda_fwd_args`` in include/kda.h."""
    _fields_ = [
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
        ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("chunk", ctypes.c_int32),
        ("qkv_dtype", ctypes.c_int),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("a_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("beta", ctypes.c_void_p),
        ("scale", ctypes.c_float), ("eps", ctypes.c_float),
        ("initial_state", ctypes.c_void_p), ("cu_seqlens", ctypes.c_void_p),
        ("num_seqs", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("out", ctypes.c_void_p), ("final_state", ctypes.c_void_p),
        ("h_out", ctypes.c_void_p), ("v_new_out", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("Hk", ctypes.c_int32),
    ]


class kda_decode_args(ctypes.Structure):
    """Mirror of ``kda_decode_args`` in include/kda.h."""
    _fields_ = [
        ("N", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
        ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("qkv_dtype", ctypes.c_int),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("a_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("scale", ctypes.c_float), ("eps", ctypes.c_float),
        ("flags", ctypes.c_uint32), ("out", ctypes.c_void_p), ("cache", ctypes.c_void_p),
        ("cache_dtype", ctypes.c_int), ("num_rows", ctypes.c_int64),
        ("row_stride_elems", ctypes.c_int64), ("idx", ctypes.c_void_p), ("idx_dtype", ctypes.c_int),
        ("init_flags", ctypes.c_void_p), ("Hk", ctypes.c_int32),
    ]


class kda_bwd_args(ctypes.Structure):
    """Mirror of ``kda_bwd_args`` in include/kda.h."""
    _fields_ = [
        ("fwd", kda_fwd_args),
        ("d_out", ctypes.c_void_p), ("d_final_state", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("dg", ctypes.c_void_p), ("dbeta", ctypes.c_void_p),
        ("da_log", ctypes.c_void_p), ("ddt_bias", ctypes.c_void_p),
        ("d_initial_state", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libkda.so (raises when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libkda.so not built ({path}); run "
                          "`python -m chunked_kimi_delta_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(path)
    vp, i32, i64, P = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(kda_fwd_args)
    sigs = {
        "kda_chunk_fwd_workspace_size": ([P], ctypes.c_size_t),
        "kda_chunk_fwd": ([P, vp], ctypes.c_int),
        "kda_segment_summary_workspace_size": ([P, i32], ctypes.c_size_t),
        "kda_segment_summary": ([P, vp, i32, vp, vp, vp], ctypes.c_int),
        "kda_state_prefix_scan": ([vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp], ctypes.c_int),
        "kda_state_gather": ([vp, ctypes.c_int, i64, i64, i64, vp, ctypes.c_int, vp, i64, vp, vp],
                             ctypes.c_int),
        "kda_state_scatter": ([vp, ctypes.c_int, i64, i64, i64, vp, ctypes.c_int, vp, ctypes.c_int,
                               i64, vp], ctypes.c_int),
        "kda_get_device_status": ([vp, vp], ctypes.c_int),
        "kda_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "kda_chunk_fwd_static_scratch": ([P, vp], ctypes.c_int),
        "kda_static_scratch_status": ([vp], ctypes.c_int),
        "kda_chunk_fwd_host_workspace_size": ([P], ctypes.c_size_t),
        "kda_chunk_fwd_host": ([P, vp], ctypes.c_int),
        "kda_recurrent_step": ([ctypes.POINTER(kda_decode_args), vp], ctypes.c_int),
        "kda_chunk_fwd_stages": ([P, ctypes.POINTER(ctypes.c_char_p), i32], i32),
        "kda_chunk_fwd_profiled": ([P, vp, ctypes.POINTER(vp), i32], ctypes.c_int),
        "kda_chunk_bwd_workspace_size": ([ctypes.POINTER(kda_bwd_args)], ctypes.c_size_t),
        "kda_chunk_bwd": ([ctypes.POINTER(kda_bwd_args), vp], ctypes.c_int),
        "kda_segment_bwd_summary_workspace_size": ([P, i32], ctypes.c_size_t),
        "kda_segment_bwd_summary": ([P, vp, vp, i32, vp, vp], ctypes.c_int),
        "kda_state_grad_scan": ([vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp], ctypes.c_int),
    }
    for name, (argt, rest) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = argt
        f.restype = rest
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().kda_status_string(status).decode()


def _check(status: int, what: str):
    if status != KDA_OK:
        raise KdaError(status, what)


# ---------------------------------------------------------------- marshalling

def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return KDA_F32
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _check_devices(devices, current: int):
    """``devices``: the torch devices of a call's tensors (None entries
    skipped).  They must all be the current CUDA device ``current``: the
    library launches on the current device and stream, and a pointer to
    another GPU's memory (or to host memory) would fault the device."""
    dev = None
    for d in devices:
        if d is None:
            continue
        if d.type != "cuda":
            raise ValueError("this call takes CUDA tensors (host tensors: kda_chunk_fwd_host)")
        if dev is None:
            dev = d
        elif d != dev:
            raise ValueError("all tensors of a call must be on one CUDA device")
    if dev is not None and dev.index != current:
        raise ValueError(f"the tensors are on {dev} but cuda:{current} is the current device: "
                         f"call under torch.cuda.device({dev.index})")


def _on_device(*ts):
    """The calls that launch kernels dereference every pointer on the
    current GPU: their tensors must be CUDA tensors of the current device."""
    devs = [None if t is None else t.device for t in ts]
    if any(d is not None and d.type != "cuda" for d in devs):
        raise ValueError("this call takes CUDA tensors (host tensors: kda_chunk_fwd_host)")
    if any(d is not None for d in devs):
        _check_devices(devs, _torch().cuda.current_device())


def _heads(x, head_major=False):
    """Head count of a [.., heads, D] (token-major) or [.., heads, T, D]
    (head-major) tensor."""
    return x.shape[-3] if head_major else x.shape[-2]


def _check_shapes(q, k, v, g, beta, out, head_major=False):
    """Token-major: q, k [.., Hk, dk]; v, out [.., H, dv]; g [.., H, dk];
    beta [.., H].  Head-major: q, k [.., Hk, T, dk]; v, out [.., H, T, dv];
    g [.., H, T, dk]; beta [.., H, T].  Same leading dims, Hk dividing H
    (the kernels trust these)."""
    if head_major:
        lead, H, T = tuple(v.shape[:-3]), v.shape[-3], v.shape[-2]
        qlead, Hk = tuple(q.shape[:-3]) + (q.shape[-2],), q.shape[-3]
        lead_t = lead + (T,)
        g_shape, b_shape = lead + (H, T, q.shape[-1]), lead + (H, T)
    else:
        lead, H = tuple(v.shape[:-2]), v.shape[-2]
        qlead, Hk, lead_t = tuple(q.shape[:-2]), q.shape[-2], lead
        g_shape, b_shape = lead + (H, q.shape[-1]), lead + (H,)
    if k.shape != q.shape or qlead != lead_t:
        raise ValueError("q and k must have v's leading dims and token count")
    if Hk < 1 or H % Hk != 0:
        raise ValueError("the key heads of q/k must divide the value heads of v")
    if tuple(g.shape) != g_shape:
        raise ValueError("g must have v's layout with dk channels")
    if tuple(beta.shape) != b_shape:
        raise ValueError("beta must be v's layout without the channel axis")
    if out is not None and out.shape != v.shape:
        raise ValueError("out must have v's shape")


def _state_shape(N, q, v, v_first=False, head_major=False):
    """Shape of N recurrent states: [N, H, dk, dv], or [N, H, dv, dk] V-first."""
    H, K, V = _heads(v, head_major), q.shape[-1], v.shape[-1]
    return (N, H, V, K) if v_first else (N, H, K, V)


# keyword arguments of make_fwd_args that are tensors
_FWD_TENSOR_KW = ("a_log", "dt_bias", "initial_state", "cu_seqlens", "out", "final_state", "h_out",
                  "v_new_out")


def make_fwd_args(q, k, v, g, beta, *, scale=None, eps=1e-6, a_log=None, dt_bias=None,
                  initial_state=None, cu_seqlens=None, l2norm_qk=True, beta_sigmoid=False,
                  gate_in_kernel=False, use_exp2=False, state_v_first=False, head_major=False,
                  extra_flags=0, out=None, final_state=None, h_out=None,
                  v_new_out=None) -> kda_fwd_args:
    """Fills a ``kda_fwd_args`` from tensors (BSND [B,T,H,D], or TND [T,H,D]
    with ``cu_seqlens``).  q and k may carry fewer heads than v (grouped key
    heads, Hk dividing H): value head h reads key head h // (H // Hk).
    Marshalling only: the calls that launch check where the tensors live."""
    _contig(q, k, v, g, beta, a_log, dt_bias, initial_state, cu_seqlens, out, final_state,
            h_out, v_new_out)
    a = kda_fwd_args()
    tax = 1 if head_major else 0  # token axis of a 3-D tensor
    if q.dim() == 3:    # TND [T, H, D] / NTD [H, T, D]: one token axis
        a.B, a.T = 1, q.shape[tax]
    elif q.dim() == 4:  # BSND [B, T, H, D] / BNSD [B, H, T, D]
        a.B, a.T = q.shape[0], q.shape[1 + tax]
    else:
        raise ValueError("q/k/v are [B, T, H, D] or [T_total, H, D] (head-major: [B, H, T, D], "
                         "[H, T_total, D])")
    if cu_seqlens is not None:
        if q.dim() != 3:
            raise ValueError("with cu_seqlens, q/k/v have one token axis")
        a.num_seqs = cu_seqlens.numel() - 1
        a.cu_seqlens = _ptr(cu_seqlens)
    _check_shapes(q, k, v, g, beta, out, head_major)
    a.H, a.Hk = _heads(v, head_major), _heads(q, head_major)
    a.dk, a.dv, a.chunk = q.shape[-1], v.shape[-1], CHUNK
    a.qkv_dtype = _dtype_code(q)
    a.q, a.k, a.v, a.g, a.beta = _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta)
    a.a_log, a.dt_bias = _ptr(a_log), _ptr(dt_bias)
    a.scale = float(q.shape[-1] ** -0.5 if scale is None else scale)
    a.eps = float(eps)
    a.initial_state = _ptr(initial_state)
    a.flags = ((KDA_L2NORM_QK if l2norm_qk else 0) | (KDA_BETA_SIGMOID if beta_sigmoid else 0)
               | (KDA_GATE_IN_KERNEL if gate_in_kernel else 0) | (KDA_USE_EXP2 if use_exp2 else 0)
               | (KDA_STATE_V_FIRST if state_v_first else 0)
               | (KDA_LAYOUT_HEAD_MAJOR if head_major else 0) | extra_flags)
    a.out, a.final_state = _ptr(out), _ptr(final_state)
    a.h_out, a.v_new_out = _ptr(h_out), _ptr(v_new_out)
    return a


def _workspace(nbytes: int, device, workspace=None):
    torch = _torch()
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def kda_chunk_fwd(q, k, v, g, beta, *, scale=None, eps=1e-6, a_log=None, dt_bias=None,
                  initial_state=None, cu_seqlens=None, l2norm_qk=True, beta_sigmoid=False,
                  gate_in_kernel=False, use_exp2=False, output_final_state=True, out=None,
                  final_state=None, h_out=None, v_new_out=None, workspace=None, stream=None,
                  reuse_prep=False, state_v_first=False, head_major=False, extra_flags=0):
    """Chunked KDA forward.  Returns ``(out, final_state)`` (final_state is
    None unless requested).  ``reuse_prep`` (with ``workspace``) sets
    KDA_REUSE_PREP: the workspace already holds this problem's intra-chunk
    results, e.g. from a kda_segment_summary whose seg_bounds are this call's
    cu_seqlens.  See ``kda_chunk_fwd`` in include/kda.h."""
    if reuse_prep:
        if workspace is None:
            raise ValueError("reuse_prep needs the workspace that holds the prepared chunks")
        extra_flags |= KDA_REUSE_PREP
    torch = _torch()
    lib = load_library()
    if cu_seqlens is not None:
        N = cu_seqlens.numel() - 1
    else:
        N = 1 if q.dim() == 3 else q.shape[0]
    if out is None:
        out = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    if output_final_state and final_state is None:
        final_state = torch.empty(_state_shape(N, q, v, state_v_first, head_major),
                                  dtype=torch.float32, device=q.device)
    a = make_fwd_args(q, k, v, g, beta, scale=scale, eps=eps, a_log=a_log, dt_bias=dt_bias,
                      initial_state=initial_state, cu_seqlens=cu_seqlens, l2norm_qk=l2norm_qk,
                      beta_sigmoid=beta_sigmoid, gate_in_kernel=gate_in_kernel, use_exp2=use_exp2,
                      state_v_first=state_v_first, head_major=head_major, extra_flags=extra_flags, out=out, final_state=final_state, h_out=h_out,
                      v_new_out=v_new_out)
    _on_device(q, k, v, g, beta, a_log, dt_bias, initial_state, cu_seqlens, out, final_state, h_out,
               v_new_out, workspace)
    ws = _workspace(lib.kda_chunk_fwd_workspace_size(ctypes.byref(a)), q.device, workspace)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    _check(lib.kda_chunk_fwd(ctypes.byref(a), _stream(stream)), "kda_chunk_fwd")
    return out, final_state


# include/kda.h KDA_STATIC_SCRATCH_BYTES
KDA_STATIC_SCRATCH_BYTES = 32 * 1024 * 1024
# include/kda.h KDA_HOST_BLOCK_TOKENS
KDA_HOST_BLOCK_TOKENS = 1024


def prepare_chunk_fwd_host(q, k, v, g, beta, *, device=None, output_final_state=True,
                           workspace=None, **kw):
    """Builds the ``kda_fwd_args`` of a host-IO forward once: q, k, v, g, beta
    and the returned ``out`` are host (CPU) tensors, ``out`` page-locked;
    final_state and the workspace live on ``device`` (default: the current
    CUDA device).  Returns (args, out, final_state, ws)."""
    torch = _torch()
    lib = load_library()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    for t in (q, k, v, g, beta):
        if t.is_cuda:
            raise ValueError("kda_chunk_fwd_host takes q, k, v, g, beta in host memory")
    out = kw.pop("out", None)
    if out is None:
        out = torch.empty(v.shape, dtype=q.dtype, pin_memory=True)
    fin = kw.pop("final_state", None)
    if output_final_state and fin is None:
        fin = torch.empty(_state_shape(q.shape[0], q, v, kw.get("state_v_first", False)),
                          dtype=torch.float32, device=device)
    a = make_fwd_args(q, k, v, g, beta, out=out, final_state=fin, **kw)
    ws = _workspace(lib.kda_chunk_fwd_host_workspace_size(ctypes.byref(a)), device, workspace)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    return a, out, fin, ws


def kda_chunk_fwd_host(q, k, v, g, beta, *, stream=None, **kw):
    """Forward on host-resident q, k, v, g, beta [B, T, H, D] (page-locked for
    overlap): the library streams them through the GPU in blocks of
    KDA_HOST_BLOCK_TOKENS tokens and writes o back to a host tensor.
    Returns ``(out, final_state)`` (out on the host, final_state on the GPU);
    both are complete when ``stream`` (default: current) passes the call.
    See ``kda_chunk_fwd_host`` in include/kda.h."""
    lib = load_library()
    a, out, fin, ws = prepare_chunk_fwd_host(q, k, v, g, beta, **kw)
    _check(lib.kda_chunk_fwd_host(ctypes.byref(a), _stream(stream)), "kda_chunk_fwd_host")
    return out, fin


def kda_chunk_fwd_static_scratch(q, k, v, g, beta, *, scale=None, eps=1e-6, a_log=None,
                                 dt_bias=None, initial_state=None, cu_seqlens=None,
                                 l2norm_qk=True, beta_sigmoid=False, gate_in_kernel=False,
                                 use_exp2=False, output_final_state=True, out=None,
                                 final_state=None, state_v_first=False, head_major=False,
                                 extra_flags=0, stream=None):
    """The forward for callers that cannot allocate device memory: same
    arguments and results as :func:`kda_chunk_fwd`, but no workspace; the
    library's fixed scratch array is used instead (problems whose workspace
    exceeds ``KDA_STATIC_SCRATCH_BYTES`` raise KdaError(KDA_ERR_WORKSPACE);
    KDA_REUSE_PREP raises KdaError(KDA_ERR_UNSUPPORTED)).  Output tensors are
    allocated here only when not supplied.  Calls sharing a GPU must not
    overlap in time; :func:`kda_static_scratch_status` reads the error word of
    the last call."""
    torch = _torch()
    lib = load_library()
    if cu_seqlens is not None:
        N = cu_seqlens.numel() - 1
    else:
        N = 1 if q.dim() == 3 else q.shape[0]
    if out is None:
        out = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    if output_final_state and final_state is None:
        final_state = torch.empty(_state_shape(N, q, v, state_v_first, head_major),
                                  dtype=torch.float32, device=q.device)
    a = make_fwd_args(q, k, v, g, beta, scale=scale, eps=eps, a_log=a_log, dt_bias=dt_bias,
                      initial_state=initial_state, cu_seqlens=cu_seqlens, l2norm_qk=l2norm_qk,
                      beta_sigmoid=beta_sigmoid, gate_in_kernel=gate_in_kernel, use_exp2=use_exp2,
                      state_v_first=state_v_first, head_major=head_major, extra_flags=extra_flags,
                      out=out, final_state=final_state)
    _on_device(q, k, v, g, beta, a_log, dt_bias, initial_state, cu_seqlens, out, final_state)
    _check(lib.kda_chunk_fwd_static_scratch(ctypes.byref(a), _stream(stream)),
           "kda_chunk_fwd_static_scratch")
    return out, final_state


def kda_static_scratch_status(stream=None) -> int:
    """The device status of the last kda_chunk_fwd_static_scratch call on
    the current device (synchronises ``stream``): KDA_OK, or
    KDA_ERR_DEVICE_TIMEOUT when a bounded device wait gave up (the word is
    cleared)."""
    return load_library().kda_static_scratch_status(_stream(stream))


def prepare_chunk_fwd(q, k, v, g, beta, *, output_final_state=True, workspace=None, **kw):
    """Builds the ``kda_fwd_args`` of a forward once (outputs and workspace
    allocated), for callers that launch the same problem repeatedly through
    ``load_library().kda_chunk_fwd``.  Returns (args, out, final_state, ws)."""
    torch = _torch()
    lib = load_library()
    cu = kw.get("cu_seqlens")
    N = (cu.numel() - 1) if cu is not None else (1 if q.dim() == 3 else q.shape[0])
    out = kw.pop("out", None)
    if out is None:
        out = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    fin = kw.pop("final_state", None)
    if output_final_state and fin is None:
        fin = torch.empty(_state_shape(N, q, v, kw.get("state_v_first", False),
                                       kw.get("head_major", False)),
                          dtype=torch.float32, device=q.device)
    a = make_fwd_args(q, k, v, g, beta, out=out, final_state=fin, **kw)
    _on_device(q, k, v, g, beta, out, fin, workspace, *[kw.get(n) for n in _FWD_TENSOR_KW])
    ws = _workspace(lib.kda_chunk_fwd_workspace_size(ctypes.byref(a)), q.device, workspace)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    return a, out, fin, ws


def prepare_segment_summary(q, k, v, g, beta, seg_bounds, *, M=None, S_tilde=None,
                            workspace=None, **kw):
    """Builds the ``kda_fwd_args`` of a segment summary once (outputs and
    workspace allocated).  Returns (args, M, S_tilde, ws)."""
    torch = _torch()
    lib = load_library()
    S = seg_bounds.numel() - 1
    H, K, V = _heads(v, kw.get("head_major", False)), q.shape[-1], v.shape[-1]
    if M is None:
        M = torch.empty(S, H, K, K, dtype=torch.float32, device=q.device)
    if S_tilde is None:
        S_tilde = torch.empty(S, H, K, V, dtype=torch.float32, device=q.device)
    a = make_fwd_args(q, k, v, g, beta, **kw)
    _on_device(q, k, v, g, beta, seg_bounds, M, S_tilde, workspace, *[kw.get(n) for n in _FWD_TENSOR_KW])
    ws = _workspace(lib.kda_segment_summary_workspace_size(ctypes.byref(a), S), q.device, workspace)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    return a, M, S_tilde, ws


def kda_chunk_fwd_stages(args: kda_fwd_args) -> list:
    """Names of the kernels kda_chunk_fwd launches for ``args``, in order."""
    lib = load_library()
    names = (ctypes.c_char_p * 8)()
    n = lib.kda_chunk_fwd_stages(ctypes.byref(args), names, 8)
    return [names[i].decode() for i in range(n)]


def kda_chunk_fwd_profiled(args: kda_fwd_args, events, stream=None):
    """kda_chunk_fwd with ``events[i]`` (torch.cuda.Event, already recorded
    once so that they exist) recorded before stage i and after the last."""
    lib = load_library()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib.kda_chunk_fwd_profiled(ctypes.byref(args), _stream(stream), arr, len(events)),
           "kda_chunk_fwd_profiled")


def kda_segment_summary(q, k, v, g, beta, seg_bounds, *, scale=None, eps=1e-6, a_log=None,
                        dt_bias=None, l2norm_qk=True, beta_sigmoid=False, gate_in_kernel=False,
                        use_exp2=False, head_major=False, M=None, S_tilde=None, workspace=None,
                        stream=None):
    """(see below; pass ``workspace`` to keep the prepared chunks for a
    following kda_chunk_fwd with ``reuse_prep=True``)"""
    return _segment_summary(q, k, v, g, beta, seg_bounds, scale=scale, eps=eps, a_log=a_log,
                            dt_bias=dt_bias, l2norm_qk=l2norm_qk, beta_sigmoid=beta_sigmoid,
                            gate_in_kernel=gate_in_kernel, use_exp2=use_exp2,
                            head_major=head_major, M=M, S_tilde=S_tilde, workspace=workspace,
                            stream=stream)


def _segment_summary(q, k, v, g, beta, seg_bounds, *, scale=None, eps=1e-6, a_log=None,
                     dt_bias=None, l2norm_qk=True, beta_sigmoid=False, gate_in_kernel=False,
                     use_exp2=False, head_major=False, M=None, S_tilde=None, workspace=None,
                     stream=None):
    """Segment affine summary.  ``seg_bounds``: int32 device tensor [S+1] of
    token offsets on the flattened token axis.  Returns ``(M, S_tilde)``."""
    torch = _torch()
    lib = load_library()
    S = seg_bounds.numel() - 1
    H, K, V = _heads(v, head_major), q.shape[-1], v.shape[-1]
    if M is None:
        M = torch.empty(S, H, K, K, dtype=torch.float32, device=q.device)
    if S_tilde is None:
        S_tilde = torch.empty(S, H, K, V, dtype=torch.float32, device=q.device)
    _contig(seg_bounds, M, S_tilde)
    a = make_fwd_args(q, k, v, g, beta, scale=scale, eps=eps, a_log=a_log, dt_bias=dt_bias,
                      l2norm_qk=l2norm_qk, beta_sigmoid=beta_sigmoid,
                      gate_in_kernel=gate_in_kernel, use_exp2=use_exp2, head_major=head_major)
    _on_device(q, k, v, g, beta, seg_bounds, M, S_tilde, a_log, dt_bias, workspace)
    ws = _workspace(lib.kda_segment_summary_workspace_size(ctypes.byref(a), S), q.device, workspace)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    _check(lib.kda_segment_summary(ctypes.byref(a), seg_bounds.data_ptr(), S, M.data_ptr(),
                                   S_tilde.data_ptr(), _stream(stream)), "kda_segment_summary")
    return M, S_tilde


def kda_state_prefix_scan(M, S_tilde, S0=None, *, S_in=None, S_final=None, stream=None):
    """Ordered prefix scan.  M [C,S,H,K,K] or [S,H,K,K]; S_tilde likewise with
    V; S0 [C,H,K,V] / [H,K,V] or None.  Returns ``(S_in, S_final)``."""
    torch = _torch()
    lib = load_library()
    one = M.dim() == 4
    C = 1 if one else M.shape[0]
    S, H, K = M.shape[-4], M.shape[-3], M.shape[-1]
    V = S_tilde.shape[-1]
    if S_in is None:
        S_in = torch.empty(S_tilde.shape, dtype=torch.float32, device=M.device)
    if S_final is None:
        S_final = torch.empty(*(() if one else (C,)), H, K, V, dtype=torch.float32, device=M.device)
    _contig(M, S_tilde, S0, S_in, S_final)
    _on_device(M, S_tilde, S0, S_in, S_final)
    _check(lib.kda_state_prefix_scan(_ptr(M), _ptr(S_tilde), _ptr(S0), C, S, H, K, V, _ptr(S_in),
                                     _ptr(S_final), _stream(stream)), "kda_state_prefix_scan")
    return S_in, S_final


def _rows(cache):
    """(num_rows, row_stride_elems, payload_elems) of a pool whose dim 0 indexes
    rows and whose remaining dims are dense."""
    payload = 1
    for d in cache.shape[1:]:
        payload *= d
    inner = cache[0] if cache.shape[0] > 0 else cache
    if cache.dim() > 1 and not inner.is_contiguous():
        raise ValueError("the payload of a cache row must be dense")
    return cache.shape[0], cache.stride(0), payload


def _idx_code(idx) -> int:
    torch = _torch()
    if idx.dtype == torch.int32:
        return KDA_I32
    if idx.dtype == torch.int64:
        return KDA_I64
    raise TypeError("indices must be int32 or int64")


def kda_state_gather(cache, idx, flags=None, *, packed=None, stream=None):
    """packed[i] = cache[idx[i]] (zeros for invalid idx or false flag)."""
    torch = _torch()
    lib = load_library()
    n_rows, stride, payload = _rows(cache)
    n = idx.numel()
    if packed is None:
        packed = torch.empty(n, *cache.shape[1:], dtype=cache.dtype, device=cache.device)
    _contig(idx, flags, packed)
    if flags is not None and flags.dtype != torch.bool:
        raise TypeError("flags must be bool")
    _on_device(cache, idx, flags, packed)
    _check(lib.kda_state_gather(_ptr(cache), _dtype_code(cache), n_rows, stride, payload, _ptr(idx),
                                _idx_code(idx), _ptr(flags), n, _ptr(packed), _stream(stream)),
           "kda_state_gather")
    return packed


def kda_state_scatter(cache, idx, packed, *, stream=None):
    """cache[idx[i]] = packed[i] (converted to the cache dtype) for valid idx."""
    lib = load_library()
    n_rows, stride, payload = _rows(cache)
    _contig(idx, packed)
    _on_device(cache, idx, packed)
    _check(lib.kda_state_scatter(_ptr(cache), _dtype_code(cache), n_rows, stride, payload,
                                 _ptr(idx), _idx_code(idx), _ptr(packed), _dtype_code(packed),
                                 idx.numel(), _stream(stream)), "kda_state_scatter")
    return cache


def kda_recurrent_step(q, k, v, g, beta, cache, idx, init_flags=None, *, scale=None, eps=1e-6,
                       a_log=None, dt_bias=None, l2norm_qk=True, beta_sigmoid=False,
                       gate_in_kernel=False, state_v_first=False, out=None, stream=None):
    """Recurrent decode step on pool states, in place: q, k [N, T, Hk, dk]
    (Hk dividing H), g [N, T, H, dk], v [N, T, H, dv], beta [N, T, H];
    ``cache`` [rows, H, dk, dv] ([rows, H, dv, dk] with ``state_v_first``;
    any row stride); ``idx`` [N] rows of the pool.  Returns out [N, T, H, dv].  See ``kda_recurrent_step`` in
    include/kda.h."""
    torch = _torch()
    lib = load_library()
    if q.dim() != 4:
        raise ValueError("q/k/v are [N, T, H, D]")
    _contig(q, k, v, g, beta, idx, init_flags, a_log, dt_bias)
    if init_flags is not None and init_flags.dtype != torch.bool:
        raise TypeError("init_flags must be bool")
    if out is None:
        out = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    _contig(out)
    _on_device(q, k, v, g, beta, cache, idx, init_flags, a_log, dt_bias, out)
    n_rows, stride, _ = _rows(cache)
    a = kda_decode_args()
    _check_shapes(q, k, v, g, beta, out)
    a.N, a.T, a.H, a.Hk = q.shape[0], q.shape[1], v.shape[2], q.shape[2]
    a.dk, a.dv = q.shape[3], v.shape[3]
    a.qkv_dtype = _dtype_code(q)
    a.q, a.k, a.v, a.g, a.beta = _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta)
    a.a_log, a.dt_bias = _ptr(a_log), _ptr(dt_bias)
    a.scale = float(q.shape[-1] ** -0.5 if scale is None else scale)
    a.eps = float(eps)
    a.flags = ((KDA_L2NORM_QK if l2norm_qk else 0) | (KDA_BETA_SIGMOID if beta_sigmoid else 0)
               | (KDA_GATE_IN_KERNEL if gate_in_kernel else 0)
               | (KDA_STATE_V_FIRST if state_v_first else 0))
    a.out = _ptr(out)
    a.cache, a.cache_dtype, a.num_rows, a.row_stride_elems = _ptr(cache), _dtype_code(cache), n_rows, stride
    a.idx, a.idx_dtype, a.init_flags = _ptr(idx), _idx_code(idx), _ptr(init_flags)
    _check(lib.kda_recurrent_step(ctypes.byref(a), _stream(stream)), "kda_recurrent_step")
    return out


def prepare_chunk_bwd(q, k, v, g, beta, d_out, *, d_final_state=None, initial_state=None,
                      want_d_initial_state=None, workspace=None, **kw):
    """Builds the ``kda_bwd_args`` of a backward once (gradient tensors and
    workspace allocated).  ``kw`` are the forward's keyword arguments
    (scale, eps, a_log, dt_bias, cu_seqlens, l2norm_qk, beta_sigmoid,
    gate_in_kernel, use_exp2).  Returns (args, grads, ws) with grads a dict
    of dq, dk, dv, dg, dbeta, da_log, ddt_bias, d_initial_state."""
    torch = _torch()
    lib = load_library()
    cu = kw.get("cu_seqlens")
    N = (cu.numel() - 1) if cu is not None else (1 if q.dim() == 3 else q.shape[0])
    hm = kw.get("head_major", False)
    H, K, V = _heads(v, hm), q.shape[-1], v.shape[-1]
    dev = q.device
    if d_out is not None:
        if d_out.shape != v.shape or d_out.dtype != q.dtype:
            raise ValueError("d_out must have v's shape and q's dtype")
        _contig(d_out)
    if d_final_state is not None:
        if (tuple(d_final_state.shape) != _state_shape(N, q, v, kw.get("state_v_first", False), hm)
                or d_final_state.dtype != torch.float32):
            raise ValueError("d_final_state must be fp32 [N, H, dk, dv] ([N, H, dv, dk] V-first)")
        _contig(d_final_state)
    if want_d_initial_state is None:
        want_d_initial_state = initial_state is not None
    gate = kw.get("gate_in_kernel", False)
    grads = dict(
        dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
        dg=torch.empty(g.shape, dtype=torch.float32, device=dev),
        dbeta=torch.empty(beta.shape, dtype=torch.float32, device=dev),
        da_log=torch.empty(H, dtype=torch.float32, device=dev) if gate else None,
        ddt_bias=torch.empty(H, K, dtype=torch.float32, device=dev) if gate else None,
        d_initial_state=(torch.empty(_state_shape(N, q, v, kw.get("state_v_first", False), hm),
                                     dtype=torch.float32, device=dev)
                         if want_d_initial_state else None),
    )
    _on_device(q, k, v, g, beta, d_out, d_final_state, initial_state, workspace,
               *[kw.get(n) for n in _FWD_TENSOR_KW])
    b = kda_bwd_args()
    b.fwd = make_fwd_args(q, k, v, g, beta, initial_state=initial_state, **kw)
    b.d_out, b.d_final_state = _ptr(d_out), _ptr(d_final_state)
    b.dq, b.dk, b.dv = _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"])
    b.dg, b.dbeta = _ptr(grads["dg"]), _ptr(grads["dbeta"])
    b.da_log, b.ddt_bias = _ptr(grads["da_log"]), _ptr(grads["ddt_bias"])
    b.d_initial_state = _ptr(grads["d_initial_state"])
    ws = _workspace(lib.kda_chunk_bwd_workspace_size(ctypes.byref(b)), dev, workspace)
    b.workspace, b.workspace_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    return b, grads, ws


def kda_chunk_bwd(q, k, v, g, beta, d_out, *, stream=None, **kw):
    """Chunked KDA backward: gradients of <d_out, o> + <d_final_state,
    final_state> with respect to the forward's inputs as given (raw q, k;
    beta logits with ``beta_sigmoid``; raw gate input with
    ``gate_in_kernel``).  Takes the forward's tensors and keyword arguments
    plus ``d_final_state`` and ``want_d_initial_state``.  Returns a dict of
    dq, dk, dv (q's dtype), dg, dbeta, da_log, ddt_bias (None without
    ``gate_in_kernel``) and d_initial_state (fp32).  See ``kda_chunk_bwd`` in
    include/kda.h."""
    lib = load_library()
    b, grads, ws = prepare_chunk_bwd(q, k, v, g, beta, d_out, **kw)
    _check(lib.kda_chunk_bwd(ctypes.byref(b), _stream(stream)), "kda_chunk_bwd")
    return grads


def kda_segment_bwd_summary(q, k, v, g, beta, d_out, seg_bounds, *, E=None, workspace=None,
                            stream=None, **kw):
    """Backward segment summary: E [S, H, dk, dv], the gradient of
    <d_out, o> over each segment with respect to the state entering it.
    ``seg_bounds``: int32 device tensor [S+1] of token offsets on the
    flattened token axis; ``kw``: the forward's keyword arguments.  See
    ``kda_segment_bwd_summary`` in include/kda.h."""
    torch = _torch()
    lib = load_library()
    S = seg_bounds.numel() - 1
    H, K, V = _heads(v, kw.get("head_major", False)), q.shape[-1], v.shape[-1]
    if E is None:
        E = torch.empty(S, H, K, V, dtype=torch.float32, device=q.device)
    if d_out is not None and (d_out.shape != v.shape or d_out.dtype != q.dtype):
        raise ValueError("d_out must have v's shape and q's dtype")
    _contig(seg_bounds, E, d_out)
    kw.pop("initial_state", None)
    kw.pop("cu_seqlens", None)
    a = make_fwd_args(q, k, v, g, beta, **kw)
    _on_device(q, k, v, g, beta, d_out, seg_bounds, E, workspace, *[kw.get(n) for n in _FWD_TENSOR_KW])
    ws = _workspace(lib.kda_segment_bwd_summary_workspace_size(ctypes.byref(a), S), q.device,
                    workspace)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    _check(lib.kda_segment_bwd_summary(ctypes.byref(a), _ptr(d_out), seg_bounds.data_ptr(), S,
                                       E.data_ptr(), _stream(stream)), "kda_segment_bwd_summary")
    return E


def kda_state_grad_scan(M, E, dS_final=None, *, dS_out=None, dS_initial=None, stream=None):
    """Reverse-order state-gradient scan.  M [C,S,H,K,K] or [S,H,K,K]; E
    likewise with V; dS_final [C,H,K,V] / [H,K,V] or None.  Returns
    ``(dS_out, dS_initial)``."""
    torch = _torch()
    lib = load_library()
    one = M.dim() == 4
    C = 1 if one else M.shape[0]
    S, H, K = M.shape[-4], M.shape[-3], M.shape[-1]
    V = E.shape[-1]
    if dS_out is None:
        dS_out = torch.empty(E.shape, dtype=torch.float32, device=M.device)
    if dS_initial is None:
        dS_initial = torch.empty(*(() if one else (C,)), H, K, V, dtype=torch.float32, device=M.device)
    _contig(M, E, dS_final, dS_out, dS_initial)
    _on_device(M, E, dS_final, dS_out, dS_initial)
    _check(lib.kda_state_grad_scan(_ptr(M), _ptr(E), _ptr(dS_final), C, S, H, K, V, _ptr(dS_out),
                                   _ptr(dS_initial), _stream(stream)), "kda_state_grad_scan")
    return dS_out, dS_initial


def kda_get_device_status(workspace, stream=None) -> int:
    """Reads and clears the device error word of a workspace; returns the status."""
    return load_library().kda_get_device_status(workspace.data_ptr(), _stream(stream))
