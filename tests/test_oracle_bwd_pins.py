"""Pins of the fp64 oracle's backward (``oracle.chunk_bwd``).

The backward is checked against central finite differences of the oracle's
forward, which is pinned on its own (test_oracle_pins.py): for a random
cotangent (d_out, d_final), every gradient the backward returns must equal
the numerical derivative of L = sum(d_out * out) + sum(d_final * final_state)
with respect to each input element.  Nothing here reuses the backward's
arithmetic.  The gradients are those "KDA Chunk Backward - TPU/Pallas Kernel
Design" sections 1-2 list (dq, dk, dv, dbeta, dg, dA_log, ddt_bias, dh0).
CPU only.
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(77)


def _inputs(T, H, K, V, *, gate_in_kernel, beta_sigmoid, l2norm, n_seqs_cu, s0=True):
    x = dict(
        q=RNG.standard_normal((T, H, K)),
        k=RNG.standard_normal((T, H, K)) * (1.0 if l2norm else 0.4),
        v=RNG.standard_normal((T, H, V)),
        g=(RNG.standard_normal((T, H, K)) if gate_in_kernel
           else -0.3 * np.abs(RNG.standard_normal((T, H, K)))),
        beta=(RNG.standard_normal((T, H)) if beta_sigmoid else RNG.uniform(0.1, 0.9, (T, H))),
        a_log=RNG.uniform(-2.0, 0.0, H),
        dt_bias=0.3 * RNG.standard_normal((H, K)),
    )
    N = len(n_seqs_cu) - 1
    if s0:
        x["S0"] = 0.2 * RNG.standard_normal((N, H, K, V))
    return x


def _prob(x, cu, flags):
    return oracle.Problem(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_seqlens=cu,
                          scale=1.0 / math.sqrt(x["q"].shape[-1]), eps=1e-6,
                          a_log=x["a_log"] if flags["gate_in_kernel"] else None,
                          dt_bias=x["dt_bias"] if flags["gate_in_kernel"] else None, **flags)


def _loss(x, cu, flags, do, dfin):
    out, fin = oracle.chunk_fwd(_prob(x, cu, flags), x.get("S0"))
    L = 0.0
    if do is not None:
        L += float(np.sum(do * out))
    if dfin is not None:
        L += float(np.sum(dfin * fin))
    return L


def _fd(x, cu, flags, do, dfin, name):
    """Central differences of the loss with respect to every element of x[name]."""
    base = x[name]
    grad = np.zeros_like(base)
    for idx in np.ndindex(base.shape):
        h = 1e-5 * max(1.0, abs(base[idx]))
        old = base[idx]
        base[idx] = old + h
        lp = _loss(x, cu, flags, do, dfin)
        base[idx] = old - h
        lm = _loss(x, cu, flags, do, dfin)
        base[idx] = old
        grad[idx] = (lp - lm) / (2 * h)
    return grad


def _check(x, cu, flags, do, dfin):
    r = oracle.chunk_bwd(_prob(x, cu, flags), x.get("S0"), do, dfin)
    names = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta"}
    if flags["gate_in_kernel"]:
        names.update(a_log="da_log", dt_bias="ddt_bias")
    if "S0" in x:
        names["S0"] = "d_initial"
    for inp, out in names.items():
        num = _fd(x, cu, flags, do, dfin, inp)
        got = r[out]
        scale = max(1.0, float(np.max(np.abs(num))))
        err = float(np.max(np.abs(got - num))) / scale
        assert err < 1e-6, f"{out}: max err {err:.2e} against finite differences"
    return r


FLAG_SETS = [
    dict(gate_in_kernel=True, beta_sigmoid=True, l2norm=True),
    dict(gate_in_kernel=False, beta_sigmoid=False, l2norm=False),
    dict(gate_in_kernel=True, beta_sigmoid=False, l2norm=True),
    dict(gate_in_kernel=False, beta_sigmoid=True, l2norm=False),
]


@pytest.mark.parametrize("flags", FLAG_SETS, ids=lambda f: "-".join(k for k, v in f.items() if v) or "plain")
def test_backward_matches_finite_differences(flags):
    """Two sequences and an empty one, d_k != d_v (a transposed state fails),
    initial states, both cotangents."""
    cu = [0, 3, 3, 7]
    T, H, K, V = 7, 2, 4, 3
    x = _inputs(T, H, K, V, n_seqs_cu=cu, **flags)
    do = RNG.standard_normal((T, H, V))
    dfin = RNG.standard_normal((3, H, K, V))
    _check(x, cu, {**flags, "use_exp2": False}, do, dfin)


def test_backward_matches_finite_differences_under_strong_decay():
    """Strong gate decay (a_log ~ U(1, 3): about -2 to -60 nats per token,
    "Hyper-Parallel Chunk KDA current implementation design" section 8.2):
    the backward still equals the derivative of the forward."""
    cu = [0, 3, 7]
    T, H, K, V = 7, 2, 4, 3
    flags = dict(gate_in_kernel=True, beta_sigmoid=True, l2norm=True)
    x = _inputs(T, H, K, V, n_seqs_cu=cu, **flags)
    x["a_log"] = RNG.uniform(1.0, 3.0, H)
    do = RNG.standard_normal((T, H, V))
    dfin = RNG.standard_normal((2, H, K, V))
    _check(x, cu, {**flags, "use_exp2": False}, do, dfin)


def test_backward_through_checkpoint_blocks():
    """A sequence longer than the oracle's 64-token checkpoint block."""
    cu = [0, 70]
    x = _inputs(70, 1, 3, 2, gate_in_kernel=True, beta_sigmoid=True, l2norm=True, n_seqs_cu=cu)
    flags = dict(gate_in_kernel=True, beta_sigmoid=True, l2norm=True)
    do = RNG.standard_normal((70, 1, 2))
    dfin = RNG.standard_normal((1, 1, 3, 2))
    r = oracle.chunk_bwd(_prob(x, cu, flags), x["S0"], do, dfin)
    # spot-check elements at the start, across the block edge and at the end
    for name, grad in (("v", "dv"), ("g", "dg")):
        base = x[name]
        for t in (0, 63, 64, 69):
            idx = (t, 0, 1)
            h = 1e-5
            old = base[idx]
            base[idx] = old + h
            lp = _loss(x, cu, flags, do, dfin)
            base[idx] = old - h
            lm = _loss(x, cu, flags, do, dfin)
            base[idx] = old
            num = (lp - lm) / (2 * h)
            assert abs(r[grad][idx] - num) < 1e-6 * max(1.0, abs(num)), (name, t)


def test_output_cotangent_only_and_state_cotangent_only():
    cu = [0, 5]
    flags = dict(gate_in_kernel=True, beta_sigmoid=True, l2norm=True)
    x = _inputs(5, 1, 3, 4, n_seqs_cu=cu, **flags)
    _check(x, cu, flags, RNG.standard_normal((5, 1, 4)), None)
    _check(x, cu, flags, None, RNG.standard_normal((1, 1, 3, 4)))


def test_zero_initial_state_gradient_still_returned():
    """Without an initial state the forward starts from zero; the gradient
    with respect to that zero state is still defined (d_initial)."""
    cu = [0, 4]
    flags = dict(gate_in_kernel=False, beta_sigmoid=False, l2norm=True)
    x = _inputs(4, 1, 3, 3, n_seqs_cu=cu, s0=False, **flags)
    do = RNG.standard_normal((4, 1, 3))
    r = oracle.chunk_bwd(_prob(x, cu, flags), None, do, None)
    x["S0"] = np.zeros((1, 1, 3, 3))
    num = _fd(x, cu, flags, do, None, "S0")
    assert np.max(np.abs(r["d_initial"] - num)) < 1e-6


def test_beta_zero_closed_form():
    """With beta = 0 the state only decays: S_t = Diag(exp(G_t)) S_0, so
    dS_0 = sum_t scale Diag(exp(G_t)) q^_t do_t^T + Diag(exp(G_T)) d_final,
    dv = 0 and dbeta_t = k^_t . (dS_t (v_t - S'_t^T k^_t)) is generally nonzero."""
    T, K, V = 6, 3, 2
    cu = [0, T]
    flags = dict(gate_in_kernel=False, beta_sigmoid=False, l2norm=True)
    x = _inputs(T, 1, K, V, n_seqs_cu=cu, **flags)
    x["beta"] = np.zeros((T, 1))
    do = RNG.standard_normal((T, 1, V))
    dfin = RNG.standard_normal((1, 1, K, V))
    r = oracle.chunk_bwd(_prob(x, cu, flags), x["S0"], do, dfin)
    qh = x["q"][:, 0] / np.sqrt(np.sum(x["q"][:, 0] ** 2, axis=-1, keepdims=True) + 1e-6)
    G = np.cumsum(x["g"][:, 0], axis=0)
    scale = 1.0 / math.sqrt(K)
    want = np.exp(G[-1])[:, None] * dfin[0, 0]
    for t in range(T):
        want += scale * np.outer(np.exp(G[t]) * qh[t], do[t, 0])
    np.testing.assert_allclose(r["d_initial"][0, 0], want, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(r["dv"], 0.0)


# ------------------------------------------- backward summary and reverse scan

def _segment_problem(T, H, K, V, seed_flags):
    cu = [0, T]
    x = _inputs(T, H, K, V, n_seqs_cu=cu, **seed_flags)
    return x, cu


@pytest.mark.parametrize("bounds", [(0, 5, 13, 20), (0, 1, 20), (0, 20)])
def test_segment_mode_backward_reproduces_unsplit_backward(bounds):
    """Forward summary -> scan -> backward summary -> reverse scan -> per-segment
    backward equals the backward of the whole sequence (fp64), for splits at
    any token.  A transposed or left-applied M, a forward-ordered scan or a
    wrong local term fails this."""
    flags = dict(gate_in_kernel=True, beta_sigmoid=True, l2norm=True)
    T, H, K, V = 20, 2, 4, 3
    x, cu = _segment_problem(T, H, K, V, flags)
    S0 = x["S0"]
    do = RNG.standard_normal((T, H, V))
    dfin = RNG.standard_normal((1, H, K, V))
    p = _prob(x, cu, flags)
    whole = oracle.chunk_bwd(p, S0, do, dfin)
    M, St = oracle.segment_summary(p, bounds)
    S_in, _ = oracle.state_prefix_scan(M, St, S0[0])
    E = oracle.segment_bwd_summary(p, bounds, do)
    dS_out, dS0 = oracle.state_grad_scan(M, E, dfin[0])
    seg = oracle.chunk_bwd(p.with_bounds(bounds), S_in, do, dS_out)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "da_log", "ddt_bias"):
        np.testing.assert_allclose(seg[name], whole[name], rtol=1e-10, atol=1e-12, err_msg=name)
    np.testing.assert_allclose(dS0, whole["d_initial"][0], rtol=1e-10, atol=1e-12)
    # the first segment's entering-state gradient is the whole initial-state gradient
    np.testing.assert_allclose(seg["d_initial"][0], whole["d_initial"][0], rtol=1e-10, atol=1e-12)


def test_backward_summary_is_the_affine_map_of_the_transition():
    """For one segment: d_initial(d_final) = M^T d_final + E, with M the
    forward transition of the segment (the gradient map is its adjoint)."""
    flags = dict(gate_in_kernel=False, beta_sigmoid=True, l2norm=True)
    T, H, K, V = 9, 1, 5, 3
    x, cu = _segment_problem(T, H, K, V, flags)
    do = RNG.standard_normal((T, H, V))
    p = _prob(x, cu, flags)
    M, _ = oracle.segment_summary(p, [0, T])
    E = oracle.segment_bwd_summary(p, [0, T], do)
    for _ in range(3):
        dfin = RNG.standard_normal((1, H, K, V))
        r = oracle.chunk_bwd(p, x["S0"], do, dfin)
        want = M[0, 0].T @ dfin[0, 0] + E[0, 0]
        np.testing.assert_allclose(r["d_initial"][0, 0], want, rtol=1e-11, atol=1e-12)


def test_state_grad_scan_small_closed_form():
    """Two segments, scalar-sized states: dS_out[1] = g, dS_out[0] = M1^T g + E1,
    dS0 = M0^T (M1^T g + E1) + E0."""
    rng = np.random.default_rng(3)
    M = rng.standard_normal((2, 1, 2, 2))
    E = rng.standard_normal((2, 1, 2, 3))
    g = rng.standard_normal((1, 2, 3))
    dS_out, dS0 = oracle.state_grad_scan(M, E, g)
    np.testing.assert_allclose(dS_out[1, 0], g[0])
    mid = M[1, 0].T @ g[0] + E[1, 0]
    np.testing.assert_allclose(dS_out[0, 0], mid)
    np.testing.assert_allclose(dS0[0], M[0, 0].T @ mid + E[0, 0])
