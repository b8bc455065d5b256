"""fp64 CPU oracle for the chunked KDA forward, its backward, segment summary,
prefix scan and state-pool gather/scatter.

TEST INFRASTRUCTURE ONLY.  The product (the CUDA library under
``chunked_kimi_delta_gb300`` and its binding) never imports, links or calls
anything here; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` do.  The oracle shares no code with the CUDA path.

* ``chunk_fwd``, ``preprocess``, ``segment_summary``, ``state_prefix_scan``:
  the token-by-token recurrence in C (``kda_oracle.c``), fp64.
* ``chunk_bwd``: gradients of the same recurrence by reverse-mode
  differentiation, token by token, in C, fp64.
* ``segment_bwd_summary``, ``state_grad_scan``: the backward twins of the
  segment summary and the prefix scan (the local state gradient of each
  segment, composed in reverse time order with the transposed transitions).
* ``chunked.py``: an independent fp64 chunked form of the same forward (the
  WY representation), used only to pin the recurrence.
* ``state_copy.py``: gather/scatter as plain indexed copies.

Parity is pinned by ``tests/test_oracle_pins.py`` (closed forms, brute force,
invariants); see the header of each function for the passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .state_copy import state_gather, state_scatter, f32_to_bf16_bits, bf16_bits_to_f32  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

# Flag bits of the oracle's own C interface (kda_oracle.c).
_L2NORM_QK, _BETA_SIGMOID, _GATE_IN_KERNEL, _USE_EXP2 = 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile kda_oracle.c with gcc (no fast-math: IEEE fp64 throughout)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Problem(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int64),
        ("cu_seqlens", ctypes.POINTER(ctypes.c_int64)),
        ("H", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("a_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("beta", ctypes.c_void_p),
        ("scale", ctypes.c_double), ("eps", ctypes.c_double),
        ("flags", ctypes.c_uint32),
    ]


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER(_Problem)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.kdaref_chunk_fwd.argtypes = [P, vp, vp, vp, i32]
        lib.kdaref_preprocess.argtypes = [P, vp, vp, vp, vp]
        lib.kdaref_segment_summary.argtypes = [P, vp, i64, vp, vp, i32]
        lib.kdaref_state_prefix_scan.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32, vp, vp]
        lib.kdaref_max_threads.argtypes = [i32]
        lib.kdaref_chunk_bwd.argtypes = [P] + [vp] * 11 + [i32]
        for f in ("kdaref_chunk_fwd", "kdaref_preprocess", "kdaref_segment_summary",
                  "kdaref_state_prefix_scan", "kdaref_max_threads", "kdaref_chunk_bwd"):
            getattr(lib, f).restype = ctypes.c_int
        _lib_handle = lib
    return _lib_handle


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (bf16 is upcast exactly)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Problem:
    """Inputs of one forward problem as contiguous fp64 arrays.

    q, k: [T_total, H, dk]; v: [T_total, H, dv]; g: [T_total, H, dk] (raw gate
    input x when ``gate_in_kernel`` else natural-log decay); beta: [T_total, H]
    (logits when ``beta_sigmoid``); cu_seqlens: [N+1] token offsets.  A fixed
    length batch [B, T, H, D] is passed flattened with cu_seqlens = {0,T,2T..}.
    """

    def __init__(self, q, k, v, g, beta, *, cu_seqlens, scale, eps=1e-6, a_log=None,
                 dt_bias=None, l2norm=True, beta_sigmoid=False, gate_in_kernel=False,
                 use_exp2=False):
        self.q, self.k, self.v, self.g, self.beta = map(_f64, (q, k, v, g, beta))
        T = self.q.shape[0] if self.q.ndim == 3 else self.q.shape[0] * self.q.shape[1]
        H, dk = self.q.shape[-2], self.q.shape[-1]
        dv = self.v.shape[-1]
        self.q = self.q.reshape(T, H, dk)
        self.k = self.k.reshape(T, H, dk)
        self.v = self.v.reshape(T, H, dv)
        self.g = self.g.reshape(T, H, dk)
        self.beta = self.beta.reshape(T, H)
        cs = cu_seqlens.detach().cpu().numpy() if hasattr(cu_seqlens, "detach") else cu_seqlens
        self.cu = np.ascontiguousarray(np.asarray(cs, dtype=np.int64))
        if self.cu[0] != 0 or self.cu[-1] != T or np.any(np.diff(self.cu) < 0):
            raise ValueError("cu_seqlens must run from 0 to T_total, non-decreasing")
        self.a_log = _f64(a_log)
        self.dt_bias = _f64(dt_bias)
        if gate_in_kernel and self.a_log is None:
            raise ValueError("gate_in_kernel needs a_log")
        self.H, self.dk, self.dv, self.T = H, dk, dv, T
        self.scale, self.eps = float(scale), float(eps)
        self.flags = ((_L2NORM_QK if l2norm else 0) | (_BETA_SIGMOID if beta_sigmoid else 0)
                      | (_GATE_IN_KERNEL if gate_in_kernel else 0) | (_USE_EXP2 if use_exp2 else 0))

    def with_bounds(self, cu_seqlens):
        """The same inputs with other range bounds on the token axis (each
        range an independent sequence)."""
        import copy
        p = copy.copy(self)
        cs = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        if cs[0] != 0 or cs[-1] != self.T or np.any(np.diff(cs) < 0):
            raise ValueError("bounds must run from 0 to T_total, non-decreasing")
        p.cu = cs
        return p

    @property
    def num_seqs(self):
        return len(self.cu) - 1

    def _c(self):
        p = _Problem()
        p.num_seqs = self.num_seqs
        p.cu_seqlens = self.cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        p.H, p.dk, p.dv = self.H, self.dk, self.dv
        p.q, p.k, p.v, p.g = map(_ptr, (self.q, self.k, self.v, self.g))
        p.a_log, p.dt_bias, p.beta = _ptr(self.a_log), _ptr(self.dt_bias), _ptr(self.beta)
        p.scale, p.eps, p.flags = self.scale, self.eps, self.flags
        return p


def max_threads(nthreads: int = 0) -> int:
    return _lib().kdaref_max_threads(nthreads)


def chunk_fwd(prob: Problem, initial_state=None, *, want_out=True, nthreads=0):
    """Token-by-token recurrence; returns (out [T,H,dv], final_state [N,H,dk,dv])."""
    N, H, K, V = prob.num_seqs, prob.H, prob.dk, prob.dv
    S0 = _f64(initial_state)
    if S0 is not None:
        S0 = S0.reshape(N, H, K, V)
    out = np.zeros((prob.T, H, V)) if want_out else None
    fin = np.zeros((N, H, K, V))
    p = prob._c()
    rc = _lib().kdaref_chunk_fwd(ctypes.byref(p), _ptr(S0), _ptr(out), _ptr(fin), nthreads)
    if rc:
        raise MemoryError("oracle allocation failed")
    return out, fin


def preprocess(prob: Problem):
    """Returns (q_hat, k_hat, beta, g_natural_log) as fp64 arrays."""
    T, H, K = prob.T, prob.H, prob.dk
    qh, kh, g = np.zeros((T, H, K)), np.zeros((T, H, K)), np.zeros((T, H, K))
    b = np.zeros((T, H))
    p = prob._c()
    _lib().kdaref_preprocess(ctypes.byref(p), _ptr(qh), _ptr(kh), _ptr(b), _ptr(g))
    return qh, kh, b, g


def segment_summary(prob: Problem, seg_bounds, nthreads=0):
    """Per segment [a,b) of the token axis: (M [S,H,dk,dk], S_tilde [S,H,dk,dv])."""
    sb = np.ascontiguousarray(np.asarray(seg_bounds, dtype=np.int64))
    S = len(sb) - 1
    M = np.zeros((S, prob.H, prob.dk, prob.dk))
    St = np.zeros((S, prob.H, prob.dk, prob.dv))
    p = prob._c()
    rc = _lib().kdaref_segment_summary(ctypes.byref(p), _ptr(sb), S, _ptr(M), _ptr(St), nthreads)
    if rc:
        raise MemoryError("oracle allocation failed")
    return M, St


def state_prefix_scan(M, S_tilde, S0=None):
    """S_in[c, j] = state entering segment j of chain c; returns (S_in, S_final).

    M: [C, S, H, dk, dk] (or [S, H, dk, dk] for one chain); S_tilde likewise
    with dv; S0: [C, H, dk, dv] or None."""
    M = _f64(M)
    St = _f64(S_tilde)
    one = M.ndim == 4
    if one:
        M, St = M[None], St[None]
    C, S, H, K, _ = M.shape
    V = St.shape[-1]
    S0 = _f64(S0)
    if S0 is not None:
        S0 = S0.reshape(C, H, K, V)
    S_in = np.zeros((C, S, H, K, V))
    fin = np.zeros((C, H, K, V))
    _lib().kdaref_state_prefix_scan(_ptr(M), _ptr(St), _ptr(S0), C, S, H, K, V, _ptr(S_in), _ptr(fin))
    if one:
        return S_in[0], fin[0]
    return S_in, fin


def chunk_bwd(prob: Problem, initial_state=None, d_out=None, d_final=None, *, nthreads=0):
    """Gradients of L = sum(d_out * out) + sum(d_final * final_state) with
    respect to the inputs as given (raw q, k; beta logits with
    ``beta_sigmoid``; raw gate input x with ``gate_in_kernel``).  Returns a
    dict: dq, dk, dg [T,H,dk]; dv [T,H,dv]; dbeta [T,H]; da_log [H] and
    ddt_bias [H,dk] (zeros without ``gate_in_kernel``); d_initial
    [N,H,dk,dv]."""
    N, H, K, V, T = prob.num_seqs, prob.H, prob.dk, prob.dv, prob.T
    S0 = _f64(initial_state)
    if S0 is not None:
        S0 = S0.reshape(N, H, K, V)
    do = _f64(d_out)
    if do is not None:
        do = do.reshape(T, H, V)
    dfin = _f64(d_final)
    if dfin is not None:
        dfin = dfin.reshape(N, H, K, V)
    r = dict(dq=np.zeros((T, H, K)), dk=np.zeros((T, H, K)), dv=np.zeros((T, H, V)),
             dg=np.zeros((T, H, K)), dbeta=np.zeros((T, H)), d_initial=np.zeros((N, H, K, V)))
    dal = np.zeros((N, H))
    ddt = np.zeros((N, H, K))
    p = prob._c()
    rc = _lib().kdaref_chunk_bwd(ctypes.byref(p), _ptr(S0), _ptr(do), _ptr(dfin), _ptr(r["dq"]),
                                 _ptr(r["dk"]), _ptr(r["dv"]), _ptr(r["dg"]), _ptr(r["dbeta"]),
                                 _ptr(dal), _ptr(ddt), _ptr(r["d_initial"]), nthreads)
    if rc:
        raise MemoryError("oracle allocation failed")
    r["da_log"] = dal.sum(axis=0)
    r["ddt_bias"] = ddt.sum(axis=0)
    return r


def segment_bwd_summary(prob: Problem, seg_bounds, d_out=None, nthreads=0):
    """E[s, h]: the gradient of <d_out, o> restricted to segment s with
    respect to the state entering the segment ("Hyper-Parallel Chunk KDA
    current implementation design" section 5.2, bwd pre-process: the local
    backward summary; "KDA Chunk Backward - TPU/Pallas Kernel Design" section
    2.4, dS_ext).  The outputs of a segment are affine in its entering state,
    so E does not depend on that state: it is the initial-state gradient of
    the segment run alone, with no final-state cotangent.  [S, H, dk, dv]."""
    r = chunk_bwd(prob.with_bounds(seg_bounds), None, d_out, None, nthreads=nthreads)
    return r["d_initial"]


def state_grad_scan(M, E, dS_final=None):
    """Reverse-order scan of the state gradient across segments (same
    sections: summaries are exchanged in reverse time order).  For each chain
    c and head h, with g = dS_final[c, h] (zeros when None):
        for j = S-1 .. 0:  dS_out[c, j, h] = g;  g = M[c, j, h]^T g + E[c, j, h]
        dS_initial[c, h] = g
    M: [C, S, H, dk, dk] (or [S, H, dk, dk]); E: the same with dv.  Returns
    (dS_out, dS_initial); dS_out[c, j] is the gradient of the state leaving
    segment j."""
    M = _f64(M)
    E = _f64(E)
    one = M.ndim == 4
    if one:
        M, E = M[None], E[None]
    C, S, H, K, _ = M.shape
    V = E.shape[-1]
    g = np.zeros((C, H, K, V)) if dS_final is None else _f64(dS_final).reshape(C, H, K, V).copy()
    dS_out = np.zeros((C, S, H, K, V))
    for c in range(C):
        for h in range(H):
            for j in range(S - 1, -1, -1):
                dS_out[c, j, h] = g[c, h]
                g[c, h] = M[c, j, h].T @ g[c, h] + E[c, j, h]
    if one:
        return dS_out[0], g[0]
    return dS_out, g
