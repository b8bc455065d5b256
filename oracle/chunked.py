"""Independent fp64 chunked form of the KDA forward (the WY representation).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Used solely to pin the
token-by-token recurrence of ``kda_oracle.c``: the two must agree to rounding.

Follows "KDA Chunk Backward - TPU/Pallas Kernel Design":
  * section 1, the chunk output  o = s (q (.) e^{G}) h + tril(A_qk) v_new,
    the inter term reading the state at the chunk start and the intra term the
    earlier (and current) tokens of the chunk;
  * section 1.2, the WY representation
        L_rj = beta_r sum_c k_rc k_jc e^{G_rc - G_jc}   (j < r),
        A = (I + L)^{-1},  u = A (v (.) beta),  w = A (k (.) beta (.) e^{G}),
        v_new = u - w h,
    and the chunk-to-chunk state step
        h' = e^{G_C} (.) h + kg^T v_new,   kg = k (.) e^{G_C - G};
with G the inclusive cumulative log-decay inside the chunk and G_C its last
row.  Natural exponentials are used (the page's base-2 form only rescales G).
Chunks restart at every sequence start; the last chunk may be partial.
The triangular system is solved exactly (forward substitution).
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def chunk_list(cu_seqlens, BT):
    """Chunks as (sequence index, first token, end token): chunks restart at
    each sequence start and never straddle a boundary (section 3.8); the last
    chunk of a sequence may be partial."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = []
    for n in range(len(cu) - 1):
        for c0 in range(int(cu[n]), int(cu[n + 1]), BT):
            out.append((n, c0, min(c0 + BT, int(cu[n + 1]))))
    return out


def chunk_fwd(qh, kh, v, beta, g, cu_seqlens, scale, BT=64, initial_state=None):
    """qh, kh, g: [T,H,K] (already normalised / natural-log decay); v: [T,H,V];
    beta: [T,H]; returns (out [T,H,V], final [N,H,K,V])."""
    T, H, K = qh.shape
    V = v.shape[-1]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    out = np.zeros((T, H, V))
    fin = np.zeros((N, H, K, V))
    chunks = chunk_list(cu, BT)
    for n in range(N):
        for h in range(H):
            S = np.zeros((K, V)) if initial_state is None else np.array(initial_state[n, h], dtype=np.float64)
            for (_, c0, c1) in (c for c in chunks if c[0] == n):
                q_, k_, v_ = qh[c0:c1, h], kh[c0:c1, h], v[c0:c1, h]
                b_ = beta[c0:c1, h]
                G = np.cumsum(g[c0:c1, h], axis=0)            # [C, K]
                C = c1 - c0
                D = G[:, None, :] - G[None, :, :]               # D[r, j, c] = G_rc - G_jc
                low = np.tril(np.ones((C, C), dtype=bool), -1)  # j < r
                lowd = np.tril(np.ones((C, C), dtype=bool), 0)  # j <= r
                Ekk = np.where(low[:, :, None], np.exp(np.where(low[:, :, None], D, 0.0)), 0.0)
                Eqk = np.where(lowd[:, :, None], np.exp(np.where(lowd[:, :, None], D, 0.0)), 0.0)
                L = b_[:, None] * np.einsum("rc,jc,rjc->rj", k_, k_, Ekk)
                Aqk = scale * np.einsum("rc,jc,rjc->rj", q_, k_, Eqk)
                I_L = np.eye(C) + L
                u = solve_triangular(I_L, v_ * b_[:, None], lower=True, unit_diagonal=True)
                w = solve_triangular(I_L, k_ * b_[:, None] * np.exp(G), lower=True, unit_diagonal=True)
                v_new = u - w @ S
                out[c0:c1, h] = scale * (q_ * np.exp(G)) @ S + Aqk @ v_new
                GC = G[-1]
                kg = k_ * np.exp(GC[None, :] - G)
                S = np.exp(GC)[:, None] * S + kg.T @ v_new
            fin[n, h] = S
    return out, fin
