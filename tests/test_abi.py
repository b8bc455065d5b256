"""The C ABI on the host, without a GPU: the library builds and loads, exports
every entry point include/kda.h declares, and rejects bad arguments with the
documented status codes before launching anything."""
import ctypes
import os
import re

import pytest

import chunked_kimi_delta_gb300 as kda
from chunked_kimi_delta_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load_library()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "kda_chunk_fwd" in names and "kda_state_scatter" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for code, name in [(0, "KDA_OK"), (1, "KDA_ERR_INVALID_ARG"), (2, "KDA_ERR_UNSUPPORTED"),
                       (3, "KDA_ERR_ALIGNMENT"), (4, "KDA_ERR_WORKSPACE"), (5, "KDA_ERR_CUDA"),
                       (6, "KDA_ERR_DEVICE_TIMEOUT")]:
        assert kda.status_string(code) == name


def _args(**kw):
    a = kda.kda_fwd_args()
    a.B, a.T, a.H, a.dk, a.dv, a.chunk = 2, 100, 4, 128, 128, 64
    a.qkv_dtype = kda.KDA_BF16
    base = 1 << 20
    a.q, a.k, a.v, a.g, a.beta, a.out = (base * (i + 1) for i in range(6))
    a.scale, a.eps = 0.088, 1e-6
    for key, val in kw.items():
        setattr(a, key, val)
    return a


def test_fwd_argument_checks(lib):
    f = lambda a: lib.kda_chunk_fwd(ctypes.byref(a), None)
    assert f(_args(q=None)) == 1
    assert f(_args(out=None)) == 1
    assert f(_args(B=0)) == 1
    assert f(_args(dk=96)) == 2
    assert f(_args(dv=256)) == 2
    assert f(_args(chunk=32)) == 2
    assert f(_args(flags=kda.KDA_SAFE_GATE)) == 2
    assert f(_args(flags=kda.KDA_ALLOW_NEG_EIGVAL)) == 2
    assert f(_args(flags=kda.KDA_STATE_V_FIRST)) == 4           # V-first: taken (no workspace)
    assert f(_args(flags=1 << 20)) == 1
    assert f(_args(flags=kda.KDA_GATE_IN_KERNEL)) == 1          # a_log missing
    assert f(_args(q=(1 << 20) + 8)) == 3                        # misaligned
    assert f(_args(cu_seqlens=1 << 24, num_seqs=3)) == 1         # cu_seqlens needs B = 1
    assert f(_args(Hk=3)) == 1                                   # key heads must divide H
    assert f(_args(Hk=-1)) == 1
    assert f(_args(Hk=2)) == 4                                   # grouped keys: valid
    assert f(_args()) == 4                                       # no workspace
    a = _args()
    need = lib.kda_chunk_fwd_workspace_size(ctypes.byref(a))
    assert need > 0
    a.workspace, a.workspace_bytes = 1 << 30, need - 1
    assert f(a) == 4
    a.workspace, a.workspace_bytes = (1 << 30) + 16, need
    assert f(a) == 3                                             # workspace not 256-aligned
    assert lib.kda_chunk_fwd(None, None) == 1


def test_grouped_key_heads_shrink_host_staging(lib):
    """Hk = 0 reads as Hk = H; fewer key heads stage fewer q/k bytes."""
    size = lambda **kw: lib.kda_chunk_fwd_host_workspace_size(ctypes.byref(_args(**kw)))
    assert size(Hk=0) == size(Hk=4) > size(Hk=1) > 0
    dev = lambda **kw: lib.kda_chunk_fwd_workspace_size(ctypes.byref(_args(**kw)))
    assert dev(Hk=1) == dev(Hk=0) > 0                            # the packages are per value head


def test_workspace_grows_with_tokens(lib):
    small = lib.kda_chunk_fwd_workspace_size(ctypes.byref(_args(T=64)))
    big = lib.kda_chunk_fwd_workspace_size(ctypes.byref(_args(T=6400)))
    assert 0 < small < big
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(_args(dk=80))) == 0


def test_summary_and_scan_checks(lib):
    a = _args()
    assert lib.kda_segment_summary(ctypes.byref(a), None, 4, 1 << 20, 1 << 21, None) == 1
    assert lib.kda_segment_summary(ctypes.byref(a), 1 << 20, 0, 1 << 20, 1 << 21, None) == 1
    assert lib.kda_segment_summary_workspace_size(ctypes.byref(a), 0) == 0
    assert lib.kda_segment_summary_workspace_size(ctypes.byref(a), 4) > 0
    s = lib.kda_state_prefix_scan
    assert s(None, 1 << 20, None, 1, 4, 8, 128, 128, 1 << 21, None, None) == 1
    assert s(1 << 20, 1 << 20, None, 1, 0, 8, 128, 128, 1 << 21, None, None) == 1
    assert s(1 << 20, 1 << 20, None, 1, 4, 8, 96, 128, 1 << 21, None, None) == 2
    assert s(1 << 20, 1 << 20, None, 1, 4, 8, 128, 128, (1 << 21) + 4, None, None) == 3


def test_state_copy_checks(lib):
    g = lib.kda_state_gather
    # empty selection: OK, nothing launched (null pointers allowed)
    assert g(None, kda.KDA_F32, 4, 10, 10, None, kda.KDA_I32, None, 0, None, None) == 0
    assert g(1 << 20, kda.KDA_F32, 4, 5, 10, 1 << 21, kda.KDA_I32, None, 3, 1 << 22, None) == 1
    assert g(1 << 20, kda.KDA_F32, 0, 10, 10, 1 << 21, kda.KDA_I32, None, 3, 1 << 22, None) == 1
    assert g(1 << 20, kda.KDA_F32, 4, 10, 10, None, kda.KDA_I32, None, 3, 1 << 22, None) == 1
    assert g(1 << 20, kda.KDA_F32, 4, 10, 10, 1 << 21, kda.KDA_I32, None, -1, 1 << 22, None) == 1
    sc = lib.kda_state_scatter
    assert sc(None, kda.KDA_BF16, 4, 10, 10, None, kda.KDA_I64, None, kda.KDA_F32, 0, None) == 0
    assert sc(1 << 20, kda.KDA_BF16, 4, 10, 10, 1 << 21, 7, 1 << 22, kda.KDA_F32, 2, None) == 1


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        kda.load_library.__wrapped__(str(tmp_path / "nope.so")) if hasattr(kda.load_library, "__wrapped__") \
            else _load_fresh(str(tmp_path / "nope.so"))


def _load_fresh(path):
    saved = kda._lib
    kda._lib = None
    try:
        return kda.load_library(path)
    finally:
        kda._lib = saved


def test_host_io_checks(lib):
    """kda_chunk_fwd_host: block workspace independent of T beyond one block,
    and the unsupported options rejected before anything is launched."""
    f = lambda a: lib.kda_chunk_fwd_host(ctypes.byref(a), None)
    ws = lambda a: lib.kda_chunk_fwd_host_workspace_size(ctypes.byref(a))
    one = ws(_args(T=kda.KDA_HOST_BLOCK_TOKENS))
    assert one > 0 and ws(_args(T=8 * kda.KDA_HOST_BLOCK_TOKENS)) == one
    assert 0 < ws(_args(T=64)) < one
    assert ws(_args(T=100, final_state=1 << 26)) < ws(_args(T=100))  # no carried-state buffer
    assert ws(_args(cu_seqlens=1 << 24, num_seqs=2, B=1)) == 0
    assert f(_args(cu_seqlens=1 << 24, num_seqs=2, B=1)) == 2
    assert f(_args(h_out=1 << 24)) == 2
    assert f(_args(v_new_out=1 << 24)) == 2
    assert f(_args(flags=kda.KDA_REUSE_PREP)) == 2
    assert f(_args(q=None)) == 1
    assert f(_args()) == 4                                       # no workspace
    assert lib.kda_chunk_fwd_host(None, None) == 1


def test_decode_checks(lib):
    def args(**kw):
        a = kda.kda_decode_args()
        a.N, a.T, a.H, a.dk, a.dv = 4, 1, 2, 128, 128
        a.qkv_dtype, a.cache_dtype, a.idx_dtype = kda.KDA_BF16, kda.KDA_F32, kda.KDA_I32
        base = 1 << 20
        a.q, a.k, a.v, a.g, a.beta, a.out, a.cache, a.idx = (base * (i + 1) for i in range(8))
        a.num_rows, a.row_stride_elems = 8, 2 * 128 * 128
        a.scale, a.eps = 0.088, 1e-6
        for key, val in kw.items():
            setattr(a, key, val)
        return a
    f = lambda a: lib.kda_recurrent_step(ctypes.byref(a), None)
    assert f(args(T=0)) == 1
    assert f(args(N=-1)) == 1
    assert f(args(q=None)) == 1
    assert f(args(idx=None)) == 1
    assert f(args(row_stride_elems=100)) == 1
    assert f(args(num_rows=0)) == 1
    assert f(args(dk=96)) == 2
    assert f(args(flags=kda.KDA_REUSE_PREP)) == 2
    assert f(args(flags=kda.KDA_SAFE_GATE)) == 2
    assert f(args(flags=kda.KDA_GATE_IN_KERNEL)) == 1   # a_log missing
    assert f(args(flags=1 << 20)) == 1
    assert f(args(N=0, q=None, idx=None)) == 0           # nothing to do
    assert f(args(Hk=3, N=0)) == 1                       # key heads must divide H
    assert f(args(Hk=-2, N=0)) == 1
    assert f(args(Hk=1, N=0)) == 0
    assert lib.kda_recurrent_step(None, None) == 1


def test_binding_shapes_for_grouped_key_heads():
    """make_fwd_args reads H from v and Hk from q/k, and rejects shapes the
    kernels would read past (host logic only, no launch)."""
    import torch
    B, T, H, Hk, dk, dv = 2, 5, 6, 2, 64, 64
    q = torch.zeros(B, T, Hk, dk)
    v = torch.zeros(B, T, H, dv)
    g = torch.zeros(B, T, H, dk)
    beta = torch.zeros(B, T, H)
    a = kda.make_fwd_args(q, q, v, g, beta)
    assert (a.H, a.Hk, a.dk, a.dv) == (H, Hk, dk, dv)
    bad = [
        dict(q=torch.zeros(B, T, 4, dk), k=torch.zeros(B, T, 4, dk)),   # 4 does not divide 6
        dict(k=torch.zeros(B, T, H, dk)),                               # q, k differ
        dict(g=torch.zeros(B, T, Hk, dk)),                              # gate per value head
        dict(beta=torch.zeros(B, T, Hk)),
        dict(out=torch.zeros(B, T, Hk, dv)),                            # out is v-shaped
    ]
    for kw in bad:
        args = dict(q=q, k=q, v=v, g=g, beta=beta)
        out = kw.pop("out", None)
        args.update(kw)
        with pytest.raises(ValueError):
            kda.make_fwd_args(args["q"], args["k"], args["v"], args["g"], args["beta"], out=out)


def test_bwd_argument_checks(lib):
    def bargs(**kw):
        b = kda.kda_bwd_args()
        b.fwd = _args()
        base = 1 << 24
        b.dq, b.dk, b.dv, b.dg, b.dbeta = (base * (i + 1) for i in range(5))
        for key, val in kw.items():
            setattr(b, key, val)
        return b
    f = lambda b: lib.kda_chunk_bwd(ctypes.byref(b), None)
    size = lambda b: lib.kda_chunk_bwd_workspace_size(ctypes.byref(b))
    assert f(bargs()) == 4                                   # no workspace
    assert size(bargs()) > lib.kda_chunk_fwd_workspace_size(ctypes.byref(_args()))
    assert f(bargs(dq=None)) == 1
    assert f(bargs(dbeta=None)) == 1
    assert f(bargs(dv=(1 << 24) + 4)) == 3
    assert f(bargs(fwd=_args(flags=kda.KDA_REUSE_PREP))) == 2
    assert f(bargs(fwd=_args(dk=96))) == 2
    assert f(bargs(fwd=_args(Hk=3))) == 1
    assert size(bargs(fwd=_args(Hk=2))) > size(bargs())     # per-value-head dq/dk scratch
    assert size(bargs(dq=None)) == 0
    b = bargs()
    b.workspace, b.workspace_bytes = (1 << 30) + 16, size(b)
    assert f(b) == 3
    assert lib.kda_chunk_bwd(None, None) == 1


def test_backward_summary_and_grad_scan_checks(lib):
    a = _args()
    f = lambda *x: lib.kda_segment_bwd_summary(ctypes.byref(a), *x)
    assert f(None, 1 << 20, 0, 1 << 22, None) == 1                  # no segments
    assert f(None, None, 2, 1 << 22, None) == 1                     # no bounds
    assert f(None, 1 << 20, 2, None, None) == 1                     # no E
    assert f((1 << 24) + 2, 1 << 20, 2, 1 << 22, None) == 3        # d_out misaligned
    assert f(None, 1 << 20, 2, 1 << 22, None) == 4                  # no workspace
    assert lib.kda_segment_bwd_summary_workspace_size(ctypes.byref(a), 2) > 0
    assert lib.kda_segment_bwd_summary_workspace_size(ctypes.byref(a), 0) == 0
    g = lambda *x: lib.kda_state_grad_scan(*x)
    assert g(None, 1 << 20, None, 1, 2, 2, 64, 64, 1 << 21, None, None) == 1
    assert g(1 << 20, 1 << 21, None, 1, 0, 2, 64, 64, 1 << 22, None, None) == 1
    assert g(1 << 20, 1 << 21, None, 1, 2, 2, 96, 64, 1 << 22, None, None) == 2
    assert g(1 << 20, 1 << 21, (1 << 23) + 4, 1, 2, 2, 64, 64, 1 << 22, None, None) == 3


def test_v_first_workspace_and_rejections(lib):
    """V-first states need K-first copies in the workspace; the summaries are
    K-first only."""
    size = lambda **kw: lib.kda_chunk_fwd_workspace_size(ctypes.byref(_args(**kw)))
    vf = kda.KDA_STATE_V_FIRST
    assert size(flags=vf) == size()                               # no states: nothing to convert
    assert size(flags=vf, initial_state=1 << 20, final_state=1 << 21) > size(
        initial_state=1 << 20, final_state=1 << 21)
    a = _args(flags=vf)
    assert lib.kda_segment_summary(ctypes.byref(a), 1 << 20, 2, 1 << 21, 1 << 22, None) == 2
    assert lib.kda_segment_bwd_summary(ctypes.byref(a), None, 1 << 20, 2, 1 << 22, None) == 2


def test_head_major_layout_checks(lib):
    hmf = kda.KDA_LAYOUT_HEAD_MAJOR
    size = lambda **kw: lib.kda_chunk_fwd_workspace_size(ctypes.byref(_args(**kw)))
    assert size(flags=hmf) > size()                      # token-major copies of every tensor
    assert lib.kda_chunk_fwd_host_workspace_size(ctypes.byref(_args(flags=hmf))) == 0
    assert lib.kda_chunk_fwd_host(ctypes.byref(_args(flags=hmf)), None) == 2
    d = kda.kda_decode_args()
    d.N, d.T, d.H, d.dk, d.dv = 0, 1, 2, 128, 128
    d.qkv_dtype, d.cache_dtype, d.idx_dtype = kda.KDA_BF16, kda.KDA_F32, kda.KDA_I32
    d.num_rows, d.row_stride_elems, d.flags = 8, 2 * 128 * 128, hmf
    assert lib.kda_recurrent_step(ctypes.byref(d), None) == 2


def test_binding_head_major_shapes():
    """make_fwd_args reads B, T, H, Hk from head-major shapes."""
    import torch
    B, T, H, Hk, dk, dv = 2, 7, 4, 2, 64, 128
    q = torch.zeros(B, Hk, T, dk)
    v = torch.zeros(B, H, T, dv)
    g = torch.zeros(B, H, T, dk)
    beta = torch.zeros(B, H, T)
    a = kda.make_fwd_args(q, q, v, g, beta, head_major=True)
    assert (a.B, a.T, a.H, a.Hk, a.dk, a.dv) == (B, T, H, Hk, dk, dv)
    assert a.flags & kda.KDA_LAYOUT_HEAD_MAJOR
    with pytest.raises(ValueError):
        kda.make_fwd_args(q, q, v, g, beta)                 # read token-major: shapes disagree
    cu = torch.tensor([0, 3, 7], dtype=torch.int32)
    a = kda.make_fwd_args(q[0], q[0], v[0], g[0], beta[0], head_major=True, cu_seqlens=cu)
    assert (a.B, a.T, a.num_seqs) == (1, T, 2)


def test_launching_calls_reject_host_tensors(lib):
    """Every binding call that launches kernels refuses host tensors before
    reaching the library (the kernels would dereference host pointers);
    mixed devices are refused too."""
    import torch
    T, H, D = 64, 2, 64
    q = torch.randn(T, H, D)
    v = torch.randn(T, H, D)
    g = torch.randn(T, H, D)
    beta = torch.rand(T, H)
    with pytest.raises(ValueError, match="CUDA tensors"):
        kda.kda_chunk_fwd(q, q, v, g, beta)
    with pytest.raises(ValueError, match="CUDA tensors"):
        kda.kda_chunk_bwd(q, q, v, g, beta, v)
    with pytest.raises(ValueError, match="CUDA tensors"):
        kda.kda_segment_summary(q, q, v, g, beta, torch.tensor([0, T], dtype=torch.int32))
    M, St = torch.zeros(1, H, D, D), torch.zeros(1, H, D, D)
    with pytest.raises(ValueError, match="CUDA tensors"):
        kda.kda_state_prefix_scan(M, St)
    with pytest.raises(ValueError, match="CUDA tensors"):
        kda.kda_state_grad_scan(M, St)
    pool = torch.zeros(4, H, D, D)
    idx = torch.tensor([1, 2], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensors"):
        kda.kda_state_gather(pool, idx)
    with pytest.raises(ValueError, match="CUDA tensors"):
        kda.kda_state_scatter(pool, idx, torch.zeros(2, H, D, D))
    with pytest.raises(ValueError, match="CUDA tensors"):
        kda.kda_recurrent_step(q[None, :1], q[None, :1], v[None, :1], g[None, :1], beta[None, :1],
                               pool, idx[:1])


def test_device_check_refuses_other_gpus_and_mixtures():
    """The library launches on the current device: tensors of another GPU,
    or of several devices, are refused before any launch (checked on device
    objects, so it runs without a GPU)."""
    import torch
    d0, d1 = torch.device("cuda", 0), torch.device("cuda", 1)
    kda._check_devices([d0, None, d0], 0)  # all on the current device: accepted
    with pytest.raises(ValueError, match="current device"):
        kda._check_devices([d1, d1], 0)
    with pytest.raises(ValueError, match="one CUDA device"):
        kda._check_devices([d0, d1], 0)
    with pytest.raises(ValueError, match="CUDA tensors"):
        kda._check_devices([d0, torch.device("cpu")], 0)
