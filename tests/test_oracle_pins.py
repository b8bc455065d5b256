"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: closed
forms, special cases, dense brute force, the independent chunked (WY) form of
"KDA Chunk Backward - TPU/Pallas Kernel Design" section 1.2, the affine
composition of "KDA Context Parallelism (KCP)" and a worked example printed on
the pages.  A plausible slip in the oracle (a dropped decay, an update before
the decay, a sign, a transposed state, a wrong composition order) fails at
least one of them.  CPU only.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import chunked

RNG = np.random.default_rng(1234)
HERE = os.path.dirname(os.path.abspath(__file__))


def _prob(T, H, K, V, *, cu=None, g=None, beta=None, q=None, k=None, v=None, scale=None,
          **kw):
    cu = [0, T] if cu is None else cu
    q = RNG.standard_normal((T, H, K)) if q is None else q
    k = RNG.standard_normal((T, H, K)) if k is None else k
    v = RNG.standard_normal((T, H, V)) if v is None else v
    g = -0.3 * np.abs(RNG.standard_normal((T, H, K))) if g is None else g
    beta = RNG.uniform(0.05, 0.95, (T, H)) if beta is None else beta
    scale = 1.0 / math.sqrt(K) if scale is None else scale
    return oracle.Problem(q, k, v, g, beta, cu_seqlens=cu, scale=scale, **kw)


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# ---------------------------------------------------------------- preprocessing

def test_gate_activation_closed_forms():
    """g = -exp(a_log) softplus(x + dt_bias): softplus(0) = ln 2, softplus(z) -> z
    for large z, -> e^z for very negative z; dt_bias adds to x."""
    T, H, K = 1, 3, 4
    x = np.zeros((T, H, K))
    x[0, 0] = [0.0, 50.0, -50.0, 1.0]
    x[0, 1] = [0.0, 0.0, 0.0, 0.0]
    x[0, 2] = [2.0, -3.0, 0.5, 10.0]
    a_log = np.array([0.0, math.log(2.0), math.log(0.25)])
    dt_bias = np.zeros((H, K))
    dt_bias[0, 3] = -1.0                      # softplus(1 - 1) = ln 2
    dt_bias[2] = [-2.0, 3.0, -0.5, 0.0]       # all softplus(0) except the last
    p = _prob(T, H, K, K, g=x, a_log=a_log, dt_bias=dt_bias, gate_in_kernel=True)
    _, _, _, g = oracle.preprocess(p)
    ln2 = math.log(2.0)
    np.testing.assert_allclose(g[0, 0], [-ln2, -50.0, -math.exp(-50.0), -ln2], rtol=1e-14)
    np.testing.assert_allclose(g[0, 1], [-2 * ln2] * 4, rtol=1e-14)
    np.testing.assert_allclose(g[0, 2], [-0.25 * ln2] * 3 + [-0.25 * (10 + math.log1p(math.exp(-10)))],
                               rtol=1e-14)


def test_gate_passthrough_without_gate_flag():
    g = -np.abs(RNG.standard_normal((5, 2, 8)))
    p = _prob(5, 2, 8, 8, g=g)
    _, _, _, g2 = oracle.preprocess(p)
    np.testing.assert_array_equal(g2, g)


def test_l2norm_and_sigmoid():
    """rstd = (sum x^2 + eps)^(-1/2); a zero vector stays zero; sigma(0) = 1/2,
    sigma(ln 3) = 3/4."""
    T, H, K = 2, 1, 4
    q = np.zeros((T, H, K))
    q[0, 0] = [3.0, 4.0, 0.0, 0.0]
    k = np.zeros((T, H, K))
    k[0, 0] = [0.0, 0.0, 1e-4, 0.0]
    beta = np.array([[0.0], [math.log(3.0)]])
    p = _prob(T, H, K, K, q=q, k=k, beta=beta, eps=1e-6, beta_sigmoid=True)
    qh, kh, b, _ = oracle.preprocess(p)
    np.testing.assert_allclose(qh[0, 0], np.array([3, 4, 0, 0]) / math.sqrt(25 + 1e-6), rtol=1e-15)
    np.testing.assert_allclose(kh[0, 0, 2], 1e-4 / math.sqrt(1e-8 + 1e-6), rtol=1e-15)
    assert np.all(qh[1] == 0) and np.all(kh[1] == 0)
    np.testing.assert_allclose(b[:, 0], [0.5, 0.75], rtol=1e-15)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("K,V", [(4, 6), (8, 8)])
def test_beta_zero_is_pure_decay(K, V):
    """beta = 0 removes every write: S_t = Diag(e^{G_t}) S_0 with G_t the
    cumulative log-decay, o_t = scale S_t^T q_t."""
    T, H = 9, 2
    S0 = RNG.standard_normal((1, H, K, V))
    g = -np.abs(RNG.standard_normal((T, H, K)))
    p = _prob(T, H, K, V, g=g, beta=np.zeros((T, H)), l2norm=False)
    out, fin = oracle.chunk_fwd(p, S0)
    G = np.cumsum(g, axis=0)
    for h in range(H):
        for t in range(T):
            St = np.exp(G[t, h])[:, None] * S0[0, h]
            np.testing.assert_allclose(out[t, h], p.scale * St.T @ p.q[t, h], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(fin[0, h], np.exp(G[-1, h])[:, None] * S0[0, h], rtol=1e-12)


def test_alpha_one_beta_zero_keeps_state():
    T, H, K, V = 7, 1, 5, 3
    S0 = RNG.standard_normal((1, H, K, V))
    p = _prob(T, H, K, V, g=np.zeros((T, H, K)), beta=np.zeros((T, H)), l2norm=False)
    out, fin = oracle.chunk_fwd(p, S0)
    np.testing.assert_array_equal(fin, S0)
    for t in range(T):
        np.testing.assert_allclose(out[t, 0], p.scale * S0[0, 0].T @ p.q[t, 0], rtol=1e-13)


def test_orthogonal_keys_give_vanilla_linear_attention():
    """alpha = 1, orthonormal keys, S_0 = 0: the delta correction vanishes and
    o_t = scale sum_{j<=t} beta_j (q_t . k_j) v_j (linear attention)."""
    K, V, H = 8, 5, 1
    T = K
    Qm, _ = np.linalg.qr(RNG.standard_normal((K, K)))
    k = Qm.T[:, None, :].copy()               # rows orthonormal
    q = RNG.standard_normal((T, H, K))
    v = RNG.standard_normal((T, H, V))
    beta = RNG.uniform(0.1, 0.9, (T, H))
    p = _prob(T, H, K, V, q=q, k=k, v=v, beta=beta, g=np.zeros((T, H, K)), l2norm=False)
    out, _ = oracle.chunk_fwd(p)
    for t in range(T):
        ref = sum(beta[j, 0] * (q[t, 0] @ k[j, 0]) * v[j, 0] for j in range(t + 1))
        np.testing.assert_allclose(out[t, 0], p.scale * ref, rtol=1e-12, atol=1e-13)


def _dense_Mt(kh, beta, g):
    K = len(kh)
    return (np.eye(K) - beta * np.outer(kh, kh)) @ np.diag(np.exp(g))


@pytest.mark.parametrize("T,K,V", [(1, 4, 6), (5, 4, 6), (8, 7, 3)])
def test_brute_force_dense_expansion(T, K, V):
    """Tiny T: explicit dense M_t = (I - beta k k^T) Diag(alpha) matrices.
    S_T = M_T..M_1 S_0 + sum_j M_T..M_{j+1} beta_j k_j v_j^T, o_t = scale S_t^T q_t,
    and the segment summary M equals the dense product (later factors left)."""
    H = 2
    S0 = RNG.standard_normal((1, H, K, V))
    p = _prob(T, H, K, V, a_log=RNG.uniform(-2, 0, H), dt_bias=0.1 * RNG.standard_normal((H, K)),
              gate_in_kernel=True, beta_sigmoid=True, g=RNG.standard_normal((T, H, K)),
              beta=RNG.standard_normal((T, H)))
    qh, kh, b, g = oracle.preprocess(p)
    out, fin = oracle.chunk_fwd(p, S0)
    M, St = oracle.segment_summary(p, [0, T])
    for h in range(H):
        Ms = [_dense_Mt(kh[t, h], b[t, h], g[t, h]) for t in range(T)]
        for t in range(T):
            P = np.eye(K)
            for r in range(t + 1):
                P = Ms[r] @ P
            S = P @ S0[0, h]
            for j in range(t + 1):
                Pj = np.eye(K)
                for r in range(j + 1, t + 1):
                    Pj = Ms[r] @ Pj
                S = S + Pj @ (b[j, h] * np.outer(kh[j, h], p.v[j, h]))
            np.testing.assert_allclose(out[t, h], p.scale * S.T @ qh[t, h], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(fin[0, h], S, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(M[0, h], P, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(St[0, h], S - P @ S0[0, h], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- chunked = recurrent

@pytest.mark.parametrize("BT", [16, 32, 64])
@pytest.mark.parametrize("lens", [(130,), (1, 63, 65, 200)])
def test_chunked_form_equals_recurrence(BT, lens):
    """The WY chunked form (TPU design section 1.2) and the token loop agree."""
    H, K, V = 2, 16, 12
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    N = len(lens)
    S0 = 0.3 * RNG.standard_normal((N, H, K, V))
    p = _prob(T, H, K, V, cu=cu, a_log=RNG.uniform(-3, 0, H), dt_bias=0.1 * RNG.standard_normal((H, K)),
              gate_in_kernel=True, beta_sigmoid=True, g=RNG.standard_normal((T, H, K)),
              beta=RNG.standard_normal((T, H)))
    out, fin = oracle.chunk_fwd(p, S0)
    qh, kh, b, g = oracle.preprocess(p)
    out2, fin2 = chunked.chunk_fwd(qh, kh, p.v, b, g, cu, p.scale, BT=BT, initial_state=S0)
    assert _rel(out2, out) < 1e-12
    assert _rel(fin2, fin) < 1e-12


@pytest.mark.parametrize("pattern", ["a_log U(1,3)", "cliff", "fast uniform"])
def test_chunked_form_equals_recurrence_under_strong_decay(pattern):
    """Strong gate decay, the regime "Hyper-Parallel Chunk KDA current
    implementation design" section 8.2 singles out: the chunked form takes
    every decay as e^{G_r - G_j} of a difference, the token loop multiplies
    the per-token decays in turn; both stay exact in fp64 whatever the decay,
    so they agree.  Patterns: gate from a_log ~ U(1, 3) (about -2 to -60 nats
    per token); a precomputed gate of -0.01 per token with a -80-nat cliff
    inside a 16-token block on half the channels; -2.2 nats per token
    everywhere (about 141 nats per 64-token chunk)."""
    H, K, V = 2, 16, 12
    lens = (1, 63, 65, 200)
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    S0 = 0.3 * RNG.standard_normal((len(lens), H, K, V))
    if pattern == "a_log U(1,3)":
        p = _prob(T, H, K, V, cu=cu, a_log=RNG.uniform(1, 3, H), dt_bias=0.1 * RNG.standard_normal((H, K)),
                  gate_in_kernel=True, beta_sigmoid=True, g=RNG.standard_normal((T, H, K)),
                  beta=RNG.standard_normal((T, H)))
    else:
        g = np.full((T, H, K), -0.01)
        if pattern == "cliff":
            g[(np.arange(T) % 16) == 5, :, 1::2] = -80.0
        else:
            g[:] = -2.2
        p = _prob(T, H, K, V, cu=cu, g=g)
    qh, kh, b, gl = oracle.preprocess(p)
    assert gl.min() < -2.0  # the case decays strongly somewhere
    out, fin = oracle.chunk_fwd(p, S0)
    for BT in (16, 64):
        out2, fin2 = chunked.chunk_fwd(qh, kh, p.v, b, gl, cu, p.scale, BT=BT, initial_state=S0)
        assert _rel(out2, out) < 1e-11
        assert _rel(fin2, fin) < 1e-11


def test_golden_varlen_chunk_map():
    """Worked example of the TPU design, section 3.8: B=1, T=12, BT=4 with two
    sequences of lengths 8 and 4 -> chunk segment ids [1, 1, 2]."""
    with open(os.path.join(HERE, "golden", "varlen_segment_ids.json")) as f:
        gold = json.load(f)
    cu = np.concatenate([[0], np.cumsum(gold["seq_lens"])])
    chunks = chunked.chunk_list(cu, gold["BT"])
    assert [n + 1 for (n, _, _) in chunks] == gold["chunk_segment_ids"]
    tok = [0] * int(cu[-1])
    for (n, a, b) in chunks:
        for t in range(a, b):
            tok[t] = n + 1
    assert tok == gold["token_segment_ids"]


def test_exp2_flag_does_not_change_the_result():
    p1 = _prob(20, 2, 8, 8, gate_in_kernel=True, a_log=np.array([-1.0, -2.0]),
               g=RNG.standard_normal((20, 2, 8)))
    p2 = oracle.Problem(p1.q, p1.k, p1.v, p1.g, p1.beta, cu_seqlens=[0, 20], scale=p1.scale,
                        a_log=p1.a_log, gate_in_kernel=True, use_exp2=True)
    np.testing.assert_array_equal(oracle.chunk_fwd(p1)[0], oracle.chunk_fwd(p2)[0])


# ---------------------------------------------------------------- varlen and segments

def test_varlen_equals_separate_runs():
    lens = (3, 70, 1, 33)
    H, K, V = 2, 8, 6
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    S0 = RNG.standard_normal((len(lens), H, K, V))
    p = _prob(T, H, K, V, cu=cu)
    out, fin = oracle.chunk_fwd(p, S0)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        pn = oracle.Problem(p.q[a:b], p.k[a:b], p.v[a:b], p.g[a:b], p.beta[a:b], cu_seqlens=[0, b - a],
                            scale=p.scale)
        o_n, f_n = oracle.chunk_fwd(pn, S0[n:n + 1])
        np.testing.assert_array_equal(out[a:b], o_n)
        np.testing.assert_array_equal(fin[n], f_n[0])


@pytest.mark.parametrize("bounds", [(0, 64, 128, 192), (0, 1, 50, 51, 130, 192), (0, 192)])
def test_segment_composition_reproduces_full_run(bounds):
    """KCP: composing (M_j, S~_j) in order by S <- M_j S + S~_j reproduces the
    state entering every segment and the final state, for any split (also
    inside a chunk); finishing each segment from its incoming state gives the
    unsplit outputs."""
    T, H, K, V = 192, 2, 8, 6
    S0 = RNG.standard_normal((1, H, K, V))
    p = _prob(T, H, K, V)
    out, fin = oracle.chunk_fwd(p, S0)
    M, St = oracle.segment_summary(p, bounds)
    S_in, S_fin = oracle.state_prefix_scan(M, St, S0)
    assert _rel(S_fin, fin[0]) < 1e-12
    seg_out, seg_fin = oracle.chunk_fwd(
        oracle.Problem(p.q, p.k, p.v, p.g, p.beta, cu_seqlens=list(bounds), scale=p.scale),
        S_in.transpose(0, 1, 2, 3)[:, :, :, :])
    assert _rel(seg_out, out) < 1e-12
    for j in range(len(bounds) - 1):
        pre = oracle.Problem(p.q[:bounds[j + 1]], p.k[:bounds[j + 1]], p.v[:bounds[j + 1]],
                             p.g[:bounds[j + 1]], p.beta[:bounds[j + 1]],
                             cu_seqlens=[0, bounds[j + 1]], scale=p.scale)
        assert _rel(seg_fin[j], oracle.chunk_fwd(pre, S0)[1][0]) < 1e-12


def test_composition_is_ordered_not_commutative():
    """Swapping two segments' summaries changes the result (the composition
    is associative but not commutative)."""
    T, H, K, V = 40, 1, 6, 6
    p = _prob(T, H, K, V)
    M, St = oracle.segment_summary(p, [0, 20, 40])
    S0 = RNG.standard_normal((H, K, V))
    _, f1 = oracle.state_prefix_scan(M, St, S0)
    _, f2 = oracle.state_prefix_scan(M[::-1].copy(), St[::-1].copy(), S0)
    assert _rel(f2, f1) > 1e-3
    # associativity: composing the two summaries first gives the same map
    M01 = M[1, 0] @ M[0, 0]
    S01 = M[1, 0] @ St[0, 0] + St[1, 0]
    np.testing.assert_allclose(M01 @ S0[0] + S01, f1[0], rtol=1e-12)


def test_scan_chains_are_independent():
    T, H, K, V = 30, 2, 4, 5
    p = _prob(T, H, K, V)
    M, St = oracle.segment_summary(p, [0, 10, 20, 30])
    S0 = RNG.standard_normal((2, H, K, V))
    Sin2, fin2 = oracle.state_prefix_scan(np.stack([M, M]), np.stack([St, St]), S0)
    for c in range(2):
        Sin1, fin1 = oracle.state_prefix_scan(M, St, S0[c])
        np.testing.assert_array_equal(Sin2[c], Sin1)
        np.testing.assert_array_equal(fin2[c], fin1)


def test_transition_is_contractive():
    """With ||k^|| = 1, beta in (0,1) and alpha <= 1 each M_t has spectral
    norm <= 1, hence so does their product."""
    p = _prob(60, 2, 8, 8, beta_sigmoid=True, beta=RNG.standard_normal((60, 2)))
    M, _ = oracle.segment_summary(p, [0, 60])
    for h in range(2):
        assert np.linalg.norm(M[0, h], 2) <= 1.0 + 1e-12
