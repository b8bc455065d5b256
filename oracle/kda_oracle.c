/*
 * kda_oracle.c - plain, slow fp64 CPU oracle for the chunked Kimi Delta
 * Attention (KDA) forward pass, its segment affine summary and the state
 * prefix scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
 * Python binding) links, loads or calls this file.  Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark use it.  It shares no
 * code, header, table or helper with the CUDA path.
 *
 * Everything is computed token by token in IEEE double precision, in the
 * order the definitions below state, with no blocking, fusion or reordering.
 *
 * Sources (page title, section):
 *  [HP]   "Hyper-Parallel Chunk KDA current implementation design" (gitcode
 *         hyper-parallel issue 12): section 4 (npu_chunk_kda arguments: gate,
 *         Q/K L2 norm with epsilon, beta sigmoid, cu_seqlens, initial_state),
 *         section 5.1 (PreProcessFwd summary H_out = M @ H_in + E), section
 *         5.3 (merge), section 6.3 (composition in rank order), section 6.5
 *         (each packed sequence resets its state).
 *  [KCP]  "KDA Context Parallelism (KCP)": "Les notations" (cumulative
 *         transition M = prod M_r, zero-start state S~), "L'algorithme"
 *         (prefix scan S <- M_j S + S~_j over earlier fragments in order).
 *  [TPU]  "KDA Chunk Backward - TPU/Pallas Kernel Design", section 1.2 (the
 *         delta rule with per-channel gate; the public gate is a natural-log
 *         decay, exp2 is an internal base change, section 3.1).
 *
 * The per-token recurrence (the pages print it only garbled) is
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t,            alpha_t = exp(g_t)  (per channel)
 * with S a d_k x d_v matrix stored K-first (row c = key channel).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDAREF_L2NORM_QK      (1u << 0)
#define KDAREF_BETA_SIGMOID   (1u << 1)
#define KDAREF_GATE_IN_KERNEL (1u << 2)
#define KDAREF_USE_EXP2       (1u << 3)

/* One forward problem.  Token-major layout [T_total, H, D]; a fixed-length
 * batch [B, T, H, D] is the same memory with cu_seqlens = {0, T, 2T, ...}. */
typedef struct {
  int64_t num_seqs;          /* N                                              */
  const int64_t *cu_seqlens; /* [N+1] token offsets, non-decreasing            */
  int32_t H, dk, dv;
  const double *q, *k;       /* [T_total, H, dk]                               */
  const double *v;           /* [T_total, H, dv]                               */
  const double *g;           /* [T_total, H, dk] raw gate input x when         */
                             /* GATE_IN_KERNEL, else natural-log decay          */
  const double *a_log;       /* [H]      (GATE_IN_KERNEL only)                 */
  const double *dt_bias;     /* [H, dk] or NULL (= zeros)                      */
  const double *beta;        /* [T_total, H]: logits when BETA_SIGMOID          */
  double scale, eps;
  uint32_t flags;
} kdaref_problem;

/* softplus(z) = log(1 + e^z), written in the overflow-free form. */
static double softplus(double z) { return fmax(z, 0.0) + log1p(exp(-fabs(z))); }

/* Preprocess one (token, head): [HP] section 4 flags.
 *   q^ = q / sqrt(sum q^2 + eps), k^ likewise      (use_qk_l2norm_in_kernel)
 *   beta = 1 / (1 + e^{-b})                         (use_beta_sigmoid_in_kernel)
 *   g_c = -exp(a_log[h]) * softplus(x_c + dt_bias[h,c])   (use_gate_in_kernel)
 * The returned g is always the natural-log decay; use_exp2 only changes the
 * base a kernel works in ([TPU] section 3.1), not the value. */
static void preprocess_token(const kdaref_problem *p, int64_t t, int h, double *qh,
                             double *kh, double *beta_out, double *g_out) {
  const int K = p->dk;
  const int64_t row = t * p->H + h;
  const double *q = p->q + row * K;
  const double *k = p->k + row * K;
  double rq = 1.0, rk = 1.0;
  if (p->flags & KDAREF_L2NORM_QK) {
    double sq = 0.0, sk = 0.0;
    for (int c = 0; c < K; ++c) { sq += q[c] * q[c]; sk += k[c] * k[c]; }
    rq = 1.0 / sqrt(sq + p->eps);
    rk = 1.0 / sqrt(sk + p->eps);
  }
  for (int c = 0; c < K; ++c) { qh[c] = q[c] * rq; kh[c] = k[c] * rk; }
  double b = p->beta[row];
  if (p->flags & KDAREF_BETA_SIGMOID) b = 1.0 / (1.0 + exp(-b));
  *beta_out = b;
  const double *x = p->g + row * K;
  if (p->flags & KDAREF_GATE_IN_KERNEL) {
    const double A = exp(p->a_log[h]);
    for (int c = 0; c < K; ++c) {
      const double bias = p->dt_bias ? p->dt_bias[(int64_t)h * K + c] : 0.0;
      g_out[c] = -A * softplus(x[c] + bias);
    }
  } else {
    for (int c = 0; c < K; ++c) g_out[c] = x[c];
  }
}

/* One token of the recurrence on S (K x V, row-major, row = key channel). */
static void step(double *S, int K, int V, const double *kh, const double *v,
                 double beta, const double *g, double *delta) {
  /* S <- Diag(alpha) S */
  for (int c = 0; c < K; ++c) {
    const double a = exp(g[c]);
    for (int j = 0; j < V; ++j) S[(int64_t)c * V + j] *= a;
  }
  /* delta = v - S^T k   (the prediction error of the decayed state) */
  for (int j = 0; j < V; ++j) {
    double s = 0.0;
    for (int c = 0; c < K; ++c) s += S[(int64_t)c * V + j] * kh[c];
    delta[j] = v[j] - s;
  }
  /* S <- S + beta k delta^T  ==  (I - beta k k^T) Diag(alpha) S_prev + beta k v^T */
  for (int c = 0; c < K; ++c) {
    const double bk = beta * kh[c];
    for (int j = 0; j < V; ++j) S[(int64_t)c * V + j] += bk * delta[j];
  }
}

typedef struct {
  double *qh, *kh, *g, *delta;
} scratch_t;

static int scratch_alloc(scratch_t *s, int K, int V) {
  s->qh = (double *)malloc(sizeof(double) * K);
  s->kh = (double *)malloc(sizeof(double) * K);
  s->g = (double *)malloc(sizeof(double) * K);
  s->delta = (double *)malloc(sizeof(double) * (V > K ? V : K));
  return s->qh && s->kh && s->g && s->delta;
}
static void scratch_free(scratch_t *s) {
  free(s->qh); free(s->kh); free(s->g); free(s->delta);
}

/* Run tokens [t0, t1) of head h from state S (in/out).  Writes o when out. */
static void run_range(const kdaref_problem *p, int64_t t0, int64_t t1, int h, double *S,
                      double *out, scratch_t *w) {
  const int K = p->dk, V = p->dv;
  for (int64_t t = t0; t < t1; ++t) {
    double beta;
    preprocess_token(p, t, h, w->qh, w->kh, &beta, w->g);
    const double *v = p->v + (t * p->H + h) * V;
    step(S, K, V, w->kh, v, beta, w->g, w->delta);
    if (out) {
      double *o = out + (t * p->H + h) * V;
      for (int j = 0; j < V; ++j) {
        double s = 0.0;
        for (int c = 0; c < K; ++c) s += S[(int64_t)c * V + j] * w->qh[c];
        o[j] = p->scale * s;
      }
    }
  }
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
  return omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* Number of threads an OpenMP region will use (1 without OpenMP). */
int kdaref_max_threads(int nthreads) { return set_threads(nthreads); }

/* Preprocessed inputs, for tests of the preprocessing and of the chunked form.
 * qh, kh, g: [T_total, H, dk]; beta: [T_total, H]. */
int kdaref_preprocess(const kdaref_problem *p, double *qh, double *kh, double *beta,
                      double *g) {
  const int K = p->dk;
  const int64_t T = p->cu_seqlens[p->num_seqs];
  for (int64_t t = 0; t < T; ++t)
    for (int h = 0; h < p->H; ++h) {
      const int64_t row = t * p->H + h;
      preprocess_token(p, t, h, qh + row * K, kh + row * K, beta + row, g + row * K);
    }
  return 0;
}

/* Forward pass: out [T_total, H, dv]; initial_state / final_state
 * [N, H, dk, dv] or NULL.  Each sequence starts from its own initial state
 * ([HP] section 6.5). */
int kdaref_chunk_fwd(const kdaref_problem *p, const double *initial_state, double *out,
                     double *final_state, int nthreads) {
  const int K = p->dk, V = p->dv, H = p->H;
  const int64_t units = p->num_seqs * H;
  const int64_t SS = (int64_t)K * V;
  int err = 0;
  set_threads(nthreads);
#pragma omp parallel
  {
    scratch_t w;
    double *S = (double *)malloc(sizeof(double) * SS);
    if (!scratch_alloc(&w, K, V) || !S) {
#pragma omp atomic write
      err = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t u = 0; u < units; ++u) {
        const int64_t n = u / H;
        const int h = (int)(u % H);
        if (initial_state) memcpy(S, initial_state + u * SS, sizeof(double) * SS);
        else memset(S, 0, sizeof(double) * SS);
        run_range(p, p->cu_seqlens[n], p->cu_seqlens[n + 1], h, S, out, &w);
        if (final_state) memcpy(final_state + u * SS, S, sizeof(double) * SS);
      }
    }
    scratch_free(&w);
    free(S);
  }
  return err;
}

/* Segment affine summary ([HP] section 5.1, [KCP] "Les notations").
 * Segment s covers tokens [seg_bounds[s], seg_bounds[s+1]) of the token axis.
 *   M_s  = M_b ... M_{a+1}   with M_t = (I - beta_t k_t k_t^T) Diag(alpha_t),
 *          later factors on the left, so that S_out = M_s S_in + S~_s;
 *   S~_s = the recurrence run over the segment from S = 0.
 * M: [S, H, dk, dk], S_tilde: [S, H, dk, dv]. */
int kdaref_segment_summary(const kdaref_problem *p, const int64_t *seg_bounds,
                           int64_t num_segments, double *M, double *S_tilde,
                           int nthreads) {
  const int K = p->dk, V = p->dv, H = p->H;
  const int64_t units = num_segments * H;
  const int64_t SS = (int64_t)K * V, MM = (int64_t)K * K;
  int err = 0;
  set_threads(nthreads);
#pragma omp parallel
  {
    scratch_t w;
    double *kv = (double *)malloc(sizeof(double) * (K > V ? K : V));
    if (!scratch_alloc(&w, K, V) || !kv) {
#pragma omp atomic write
      err = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t u = 0; u < units; ++u) {
        const int64_t s = u / H;
        const int h = (int)(u % H);
        const int64_t a = seg_bounds[s], b = seg_bounds[s + 1];
        /* zero-start state */
        double *St = S_tilde + u * SS;
        memset(St, 0, sizeof(double) * SS);
        run_range(p, a, b, h, St, NULL, &w);
        /* cumulative transition: Mc <- M_t Mc, starting from the identity */
        double *Mc = M + u * MM;
        memset(Mc, 0, sizeof(double) * MM);
        for (int c = 0; c < K; ++c) Mc[(int64_t)c * K + c] = 1.0;
        for (int64_t t = a; t < b; ++t) {
          double beta;
          preprocess_token(p, t, h, w.qh, w.kh, &beta, w.g);
          /* Y = Diag(alpha) Mc */
          for (int c = 0; c < K; ++c) {
            const double al = exp(w.g[c]);
            for (int j = 0; j < K; ++j) Mc[(int64_t)c * K + j] *= al;
          }
          /* Mc = Y - beta k (k^T Y) */
          for (int j = 0; j < K; ++j) {
            double sum = 0.0;
            for (int c = 0; c < K; ++c) sum += w.kh[c] * Mc[(int64_t)c * K + j];
            kv[j] = sum;
          }
          for (int c = 0; c < K; ++c) {
            const double bk = beta * w.kh[c];
            for (int j = 0; j < K; ++j) Mc[(int64_t)c * K + j] -= bk * kv[j];
          }
        }
      }
    }
    scratch_free(&w);
    free(kv);
  }
  return err;
}

/* Prefix scan over segments in order ([KCP] "L'algorithme", [HP] 5.3/6.3):
 *   S = S0 (or 0);  for j: S_in[j] = S;  S = M_j S + S~_j;   S_final = S.
 * Independent chains (one per sequence) are laid out one after another.
 * M: [C, S, H, dk, dk]; S_tilde, S_in: [C, S, H, dk, dv];
 * S0, S_final: [C, H, dk, dv] (S0 and S_final may be NULL). */
int kdaref_state_prefix_scan(const double *M, const double *S_tilde, const double *S0,
                             int64_t num_chains, int64_t num_segments, int H, int dk,
                             int dv, double *S_in, double *S_final) {
  const int64_t SS = (int64_t)dk * dv, MM = (int64_t)dk * dk;
  double *S = (double *)malloc(sizeof(double) * SS);
  double *T = (double *)malloc(sizeof(double) * SS);
  if (!S || !T) { free(S); free(T); return 1; }
  for (int64_t ch = 0; ch < num_chains; ++ch)
    for (int h = 0; h < H; ++h) {
      const int64_t st = ch * H + h;
      if (S0) memcpy(S, S0 + st * SS, sizeof(double) * SS);
      else memset(S, 0, sizeof(double) * SS);
      for (int64_t j = 0; j < num_segments; ++j) {
        const int64_t u = (ch * num_segments + j) * H + h;
        memcpy(S_in + u * SS, S, sizeof(double) * SS);
        const double *Mj = M + u * MM;
        const double *Sj = S_tilde + u * SS;
        for (int r = 0; r < dk; ++r)
          for (int c = 0; c < dv; ++c) {
            double sum = 0.0;
            for (int m = 0; m < dk; ++m) sum += Mj[(int64_t)r * dk + m] * S[(int64_t)m * dv + c];
            T[(int64_t)r * dv + c] = sum + Sj[(int64_t)r * dv + c];
          }
        memcpy(S, T, sizeof(double) * SS);
      }
      if (S_final) memcpy(S_final + st * SS, S, sizeof(double) * SS);
    }
  free(S);
  free(T);
  return 0;
}

/* ------------------------------------------------------------------------
 * Backward pass: gradients of  L = sum(d_out . out) + sum(d_final . final)
 * with respect to every input of kdaref_chunk_fwd, by reverse-mode
 * differentiation of the token recurrence above ([TPU] sections 1 and 2 list
 * the same gradients: dq, dk, dv, dbeta, dg, dA_log, ddt_bias and the
 * initial-state gradient dh0; [HP] section 5.2 npu_chunk_kda_bwd_finalize
 * returns the same seven plus dh0 from bwd_dhu).
 *
 * Per token, with S' = Diag(alpha) S_{t-1}, delta = v - S'^T k^,
 * S_t = S' + beta k^ delta^T and o_t = scale S_t^T q^, going backwards with
 * dS = dL/dS_t (d_final at the last token of a sequence):
 *   dS    += scale q^ do^T          dq^  = scale S_t do
 *   ddelta = beta dS^T k^           dbeta = k^T dS delta     dk^ = beta dS delta
 *   dv     = ddelta                 dS'  = dS - k^ ddelta^T  dk^ -= S' ddelta
 *   dg_c   = alpha_c sum_j dS'_cj S_{t-1,cj}                 dS_{t-1} = Diag(alpha) dS'
 * then through the preprocessing:
 *   L2 norm (x^ = x r, r = (sum x^2 + eps)^-1/2):  dx = r dx^ - r^3 (x . dx^) x
 *   sigmoid:  db = dbeta beta (1 - beta)
 *   gate g = -exp(a_log) softplus(z), z = x + dt_bias:
 *             dz = -exp(a_log) sigmoid(z) dg;  dx = dz;  ddt_bias += dz;  da_log += g dg
 * The states S_{t-1} of a sequence are recomputed forward from checkpoints
 * kept every KDAREF_CKPT tokens.
 * ------------------------------------------------------------------------ */
#define KDAREF_CKPT 64

/* Raw-input gradients of one token from the gradients of its preprocessed
 * values (dqh, dkh over K channels, dbeta, dgn = gradient of the natural-log
 * decay).  dq, dk, dg are rows of [T, H, dk]; *db the token's beta gradient;
 * dalog / ddtb accumulate this head's parameter gradients. */
static void preprocess_bwd(const kdaref_problem *p, int64_t t, int h, const double *dqh,
                           const double *dkh, double dbeta, const double *dgn, double *dq,
                           double *dk, double *db, double *dg, double *dalog, double *ddtb) {
  const int K = p->dk;
  const int64_t row = t * p->H + h;
  const double *q = p->q + row * K;
  const double *k = p->k + row * K;
  if (p->flags & KDAREF_L2NORM_QK) {
    double sq = 0.0, sk = 0.0, pq = 0.0, pk = 0.0;
    for (int c = 0; c < K; ++c) {
      sq += q[c] * q[c];
      sk += k[c] * k[c];
      pq += q[c] * dqh[c];
      pk += k[c] * dkh[c];
    }
    const double rq = 1.0 / sqrt(sq + p->eps), rk = 1.0 / sqrt(sk + p->eps);
    for (int c = 0; c < K; ++c) {
      dq[c] = rq * dqh[c] - rq * rq * rq * pq * q[c];
      dk[c] = rk * dkh[c] - rk * rk * rk * pk * k[c];
    }
  } else {
    for (int c = 0; c < K; ++c) { dq[c] = dqh[c]; dk[c] = dkh[c]; }
  }
  double b = p->beta[row];
  if (p->flags & KDAREF_BETA_SIGMOID) {
    const double s = 1.0 / (1.0 + exp(-b));
    *db = dbeta * s * (1.0 - s);
  } else {
    *db = dbeta;
  }
  const double *x = p->g + row * K;
  if (p->flags & KDAREF_GATE_IN_KERNEL) {
    const double A = exp(p->a_log[h]);
    for (int c = 0; c < K; ++c) {
      const double z = x[c] + (p->dt_bias ? p->dt_bias[(int64_t)h * K + c] : 0.0);
      const double sig = 1.0 / (1.0 + exp(-z));
      const double dz = -A * sig * dgn[c];
      dg[c] = dz;
      ddtb[c] += dz;
      *dalog += -A * softplus(z) * dgn[c];
    }
  } else {
    for (int c = 0; c < K; ++c) dg[c] = dgn[c];
  }
}

/* Gradients.  d_out [T_total, H, dv] (NULL = zeros); d_final [N, H, dk, dv]
 * (NULL = zeros); outputs dq, dk, dg [T_total, H, dk], dv [T_total, H, dv],
 * dbeta [T_total, H] (with respect to the inputs as given: logits, raw gate
 * input), da_log_part [N, H] and ddt_bias_part [N, H, dk] (per-sequence
 * parts of the parameter gradients, to be summed over N), d_initial
 * [N, H, dk, dv] (may be NULL). */
int kdaref_chunk_bwd(const kdaref_problem *p, const double *initial_state,
                     const double *d_out, const double *d_final, double *dq, double *dk,
                     double *dv, double *dg, double *dbeta, double *da_log_part,
                     double *ddt_bias_part, double *d_initial, int nthreads) {
  const int K = p->dk, V = p->dv, H = p->H;
  const int64_t units = p->num_seqs * H;
  const int64_t SS = (int64_t)K * V;
  int err = 0;
  set_threads(nthreads);
#pragma omp parallel
  {
    scratch_t w;
    int64_t maxlen = 0;
    for (int64_t n = 0; n < p->num_seqs; ++n) {
      const int64_t len = p->cu_seqlens[n + 1] - p->cu_seqlens[n];
      if (len > maxlen) maxlen = len;
    }
    const int64_t nck = maxlen / KDAREF_CKPT + 1;
    double *ck = (double *)malloc(sizeof(double) * SS * nck);              /* checkpoints */
    double *blk = (double *)malloc(sizeof(double) * SS * (KDAREF_CKPT + 1)); /* a block's states */
    double *dS = (double *)malloc(sizeof(double) * SS);
    double *dSd = (double *)malloc(sizeof(double) * SS);
    double *Sd = (double *)malloc(sizeof(double) * SS);
    double *vec = (double *)malloc(sizeof(double) * (5 * K + 2 * V));
    if (!scratch_alloc(&w, K, V) || !ck || !blk || !dS || !dSd || !Sd || !vec) {
#pragma omp atomic write
      err = 1;
    } else {
      double *dqh = vec, *dkh = vec + K, *dgn = vec + 2 * K, *alpha = vec + 3 * K;
      double *ddelta = vec + 5 * K, *delta = vec + 5 * K + V;
#pragma omp for schedule(dynamic, 1)
      for (int64_t u = 0; u < units; ++u) {
        const int64_t n = u / H;
        const int h = (int)(u % H);
        const int64_t a = p->cu_seqlens[n], b = p->cu_seqlens[n + 1];
        double *dalog = da_log_part + u, *ddtb = ddt_bias_part + u * K;
        *dalog = 0.0;
        memset(ddtb, 0, sizeof(double) * K);
        /* forward: checkpoint the state entering every KDAREF_CKPT-th token */
        double *S = blk;
        if (initial_state) memcpy(S, initial_state + u * SS, sizeof(double) * SS);
        else memset(S, 0, sizeof(double) * SS);
        for (int64_t t = a; t < b; ++t) {
          if ((t - a) % KDAREF_CKPT == 0)
            memcpy(ck + ((t - a) / KDAREF_CKPT) * SS, S, sizeof(double) * SS);
          run_range(p, t, t + 1, h, S, NULL, &w);
        }
        /* backward, block by block from the end */
        if (d_final) memcpy(dS, d_final + u * SS, sizeof(double) * SS);
        else memset(dS, 0, sizeof(double) * SS);
        for (int64_t c0 = b > a ? (b - 1 - a) / KDAREF_CKPT * KDAREF_CKPT : 0; b > a && c0 >= 0;
             c0 -= KDAREF_CKPT) {
          const int64_t t0 = a + c0, t1 = (t0 + KDAREF_CKPT < b) ? t0 + KDAREF_CKPT : b;
          /* blk[i] = state entering token t0 + i, i = 0 .. t1 - t0 */
          memcpy(blk, ck + (c0 / KDAREF_CKPT) * SS, sizeof(double) * SS);
          for (int64_t t = t0; t < t1; ++t) {
            memcpy(blk + (t - t0 + 1) * SS, blk + (t - t0) * SS, sizeof(double) * SS);
            run_range(p, t, t + 1, h, blk + (t - t0 + 1) * SS, NULL, &w);
          }
          for (int64_t t = t1 - 1; t >= t0; --t) {
            const double *Sp = blk + (t - t0) * SS;   /* S_{t-1} */
            const double *St = blk + (t - t0 + 1) * SS; /* S_t */
            double beta;
            preprocess_token(p, t, h, w.qh, w.kh, &beta, w.g);
            const double *v = p->v + (t * H + h) * V;
            const double *dov = d_out ? d_out + (t * H + h) * V : NULL;
            for (int c = 0; c < K; ++c) alpha[c] = exp(w.g[c]);
            for (int c = 0; c < K; ++c)
              for (int j = 0; j < V; ++j) Sd[(int64_t)c * V + j] = alpha[c] * Sp[(int64_t)c * V + j];
            for (int j = 0; j < V; ++j) {
              double s = 0.0;
              for (int c = 0; c < K; ++c) s += Sd[(int64_t)c * V + j] * w.kh[c];
              delta[j] = v[j] - s;
            }
            /* o_t = scale S_t^T q^ */
            for (int c = 0; c < K; ++c) {
              double s = 0.0;
              if (dov)
                for (int j = 0; j < V; ++j) s += St[(int64_t)c * V + j] * dov[j];
              dqh[c] = p->scale * s;
              if (dov)
                for (int j = 0; j < V; ++j) dS[(int64_t)c * V + j] += p->scale * w.qh[c] * dov[j];
            }
            /* S_t = S' + beta k^ delta^T */
            double dbt = 0.0;
            for (int j = 0; j < V; ++j) {
              double s = 0.0;
              for (int c = 0; c < K; ++c) s += dS[(int64_t)c * V + j] * w.kh[c];
              ddelta[j] = beta * s;
              dbt += s * delta[j];
            }
            for (int c = 0; c < K; ++c) {
              double s = 0.0;
              for (int j = 0; j < V; ++j) s += dS[(int64_t)c * V + j] * delta[j];
              dkh[c] = beta * s;
            }
            /* delta = v - S'^T k^ */
            double *dvr = dv + (t * H + h) * V;
            for (int j = 0; j < V; ++j) dvr[j] = ddelta[j];
            for (int c = 0; c < K; ++c) {
              double s = 0.0;
              for (int j = 0; j < V; ++j) {
                dSd[(int64_t)c * V + j] = dS[(int64_t)c * V + j] - w.kh[c] * ddelta[j];
                s += Sd[(int64_t)c * V + j] * ddelta[j];
              }
              dkh[c] -= s;
            }
            /* S' = Diag(alpha) S_{t-1} */
            for (int c = 0; c < K; ++c) {
              double s = 0.0;
              for (int j = 0; j < V; ++j) s += dSd[(int64_t)c * V + j] * Sp[(int64_t)c * V + j];
              dgn[c] = alpha[c] * s;
              for (int j = 0; j < V; ++j) dS[(int64_t)c * V + j] = alpha[c] * dSd[(int64_t)c * V + j];
            }
            const int64_t row = t * H + h;
            preprocess_bwd(p, t, h, dqh, dkh, dbt, dgn, dq + row * K, dk + row * K, dbeta + row,
                           dg + row * K, dalog, ddtb);
          }
        }
        if (d_initial) memcpy(d_initial + u * SS, dS, sizeof(double) * SS);
      }
    }
    scratch_free(&w);
    free(ck); free(blk); free(dS); free(dSd); free(Sd); free(vec);
  }
  return err;
}
