// kda_generic.cu - CUDA-core (fp32 arithmetic) chunked KDA forward.
//
// This is the exact-arithmetic path: fp32 FMAs, exponentials of the exact
// differences of cumulative gates (no factorisation), a fp32 triangular
// solve.  It serves fp32 inputs, where the forward must match the fp64
// recurrence to 1e-4, and every shape the tensor-core path does not take.
//
// Chunk formulas ("KDA Chunk Backward - TPU/Pallas Kernel Design", sections 1
// and 1.2), per chunk of up to 64 tokens with G the inclusive cumulative
// log-decay inside the chunk and h the state entering it:
//   L_rj  = beta_r sum_c k_rc k_jc e^{G_rc - G_jc}      (j < r)
//   A     = (I + L)^-1,   u = A (v . beta),   w = A (k . beta . e^{G})
//   Aqk_rj = scale sum_c q_rc k_jc e^{G_rc - G_jc}     (j <= r)
//   v_new = u - w h,   o = scale (q . e^{G}) h + Aqk v_new
//   h'    = e^{G_C} . h + (k . e^{G_C - G})^T v_new
// With KDA_USE_EXP2 the gates are carried in base 2 and exponentiated with
// exp2 (section 3.1); the result is the same up to rounding.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex(float x, bool base2) { return base2 ? exp2f(x) : expf(x); }

// ---------------------------------------------------------------------------
// chunk_off[n] = number of chunks in ranges [0, n); one block.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) chunk_map_kernel(SeqInfo s, int32_t *chunk_off) {
  __shared__ long long part[1024];
  const int tid = threadIdx.x;
  const int per = (s.N + 1023) / 1024;
  const int a = min(tid * per, s.N), b = min(a + per, s.N);
  long long sum = 0;
  for (int n = a; n < b; ++n) {
    int64_t t0, t1;
    seq_range(s, n, t0, t1);
    sum += (t1 - t0 + BT - 1) / BT;
  }
  part[tid] = sum;
  __syncthreads();
  if (tid == 0) {
    long long acc = 0;
    for (int i = 0; i < 1024; ++i) {
      const long long x = part[i];
      part[i] = acc;
      acc += x;
    }
    chunk_off[s.N] = (int32_t)acc;
  }
  __syncthreads();
  long long acc = part[tid];
  for (int n = a; n < b; ++n) {
    chunk_off[n] = (int32_t)acc;
    int64_t t0, t1;
    seq_range(s, n, t0, t1);
    acc += (t1 - t0 + BT - 1) / BT;
  }
}

// ---------------------------------------------------------------------------
// Intra-chunk stage: one CTA per (chunk, head).
// ---------------------------------------------------------------------------
template <typename Tin, int K, int V>
__global__ void __launch_bounds__(256)
generic_intra_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                     const Tin *__restrict__ v, const float *__restrict__ g,
                     const float *__restrict__ beta, GateParams gp, SeqInfo s, int H, int Hk,
                     float *__restrict__ w_out, float *__restrict__ u_out,
                     float *__restrict__ qg_out, float *__restrict__ kg_out,
                     float *__restrict__ aqk_out, float *__restrict__ gc_out) {
  constexpr int KP = K + 1;
  constexpr int XP = (K > V ? K : V) + 1;
  extern __shared__ float smem[];
  float *sQ = smem;          // [64][XP]  q^ ; later v.beta
  float *sK = sQ + 64 * XP;  // [64][KP]  k^ ; later k^.beta.e^G
  float *sG = sK + 64 * KP;  // [64][KP]  cumulative gate
  float *sL = sG + 64 * KP;  // [64][65]  L
  float *sA = sL + 64 * 65;  // [64][65]  Aqk, then (I+L)^-1
  float *sB = sA + 64 * 65;  // [64]      beta

  const int64_t c = blockIdx.x;
  const int h = blockIdx.y;
  int n, len;
  int64_t t0;
  if (!chunk_lookup(s, c, n, t0, len)) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool base2 = (gp.flags & KDA_USE_EXP2) != 0;
  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;

  // 1. q, k, gate (rows past the chunk end are zero).
  const float A_h = gate ? expf(gp.a_log[h]) : 0.f;
  for (int i = tid; i < BT * K; i += 256) {
    const int r = i / K, cc = i % K;
    float qv = 0.f, kv = 0.f, gv = 0.f;
    if (r < len) {
      const int64_t off = ((t0 + r) * H + h) * (int64_t)K + cc;
      const int64_t offk = ((t0 + r) * Hk + h / (H / Hk)) * (int64_t)K + cc;  // grouped key heads
      qv = to_f32(q[offk]);
      kv = to_f32(k[offk]);
      gv = g[off];
      if (gate) {
        const float z = gv + (gp.dt_bias ? gp.dt_bias[h * K + cc] : 0.f);
        const float sp = fmaxf(z, 0.f) + log1pf(expf(-fabsf(z)));  // softplus
        gv = -A_h * sp;
      }
      if (base2) gv *= kLog2e;
    }
    sQ[r * XP + cc] = qv;
    sK[r * KP + cc] = kv;
    sG[r * KP + cc] = gv;
  }
  if (tid < BT) {
    float b = 0.f;
    if (tid < len) {
      b = beta[(t0 + tid) * H + h];
      if (gp.flags & KDA_BETA_SIGMOID) b = 1.f / (1.f + expf(-b));
    }
    sB[tid] = b;
  }
  __syncthreads();

  // 2. L2 norm of q and k rows; chunk-local inclusive cumsum of the gate.
  if (gp.flags & KDA_L2NORM_QK) {
    for (int r = warp; r < BT; r += 8) {
      float sq = 0.f, sk = 0.f;
      for (int cc = lane; cc < K; cc += 32) {
        const float a = sQ[r * XP + cc], b = sK[r * KP + cc];
        sq += a * a;
        sk += b * b;
      }
      for (int o = 16; o; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      const float rq = rsqrtf(sq + gp.eps), rk = rsqrtf(sk + gp.eps);
      for (int cc = lane; cc < K; cc += 32) {
        sQ[r * XP + cc] *= rq;
        sK[r * KP + cc] *= rk;
      }
    }
  }
  if (tid < K) {
    float acc = 0.f;
    for (int r = 0; r < BT; ++r) {
      acc += sG[r * KP + tid];
      sG[r * KP + tid] = acc;
    }
  }
  __syncthreads();

  // 3. L (strictly lower, beta-weighted) and Aqk (lower with diagonal, scaled)
  //    over the 2080 pairs j <= r, with exact exponentials of differences.
  for (int p = tid; p < BT * (BT + 1) / 2; p += 256) {
    int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
    while ((r + 1) * (r + 2) / 2 <= p) ++r;
    while (r * (r + 1) / 2 > p) --r;
    const int j = p - r * (r + 1) / 2;
    float kk = 0.f, qk = 0.f;
    for (int cc = 0; cc < K; ++cc) {
      const float e = ex(sG[r * KP + cc] - sG[j * KP + cc], base2);
      const float kj = sK[j * KP + cc] * e;
      kk = fmaf(sK[r * KP + cc], kj, kk);
      qk = fmaf(sQ[r * XP + cc], kj, qk);
    }
    sL[r * 65 + j] = (j < r) ? sB[r] * kk : 0.f;
    sA[r * 65 + j] = gp.scale * qk;
  }
  for (int i = tid; i < BT * BT; i += 256) {
    const int r = i / BT, j = i % BT;
    if (j > r) {
      sL[r * 65 + j] = 0.f;
      sA[r * 65 + j] = 0.f;
    }
  }
  __syncthreads();

  // 4. qg = scale q^ e^G, kg = k^ e^{G_C - G}, Aqk, gC = e^{G_C}.
  const float *GC = sG + (len - 1) * KP;
  for (int i = tid; i < len * K; i += 256) {
    const int r = i / K, cc = i % K;
    const int64_t off = ((t0 + r) * H + h) * (int64_t)K + cc;
    const float G = sG[r * KP + cc];
    qg_out[off] = gp.scale * sQ[r * XP + cc] * ex(G, base2);
    kg_out[off] = sK[r * KP + cc] * ex(GC[cc] - G, base2);
  }
  for (int i = tid; i < len * BT; i += 256) {
    const int r = i / BT, j = i % BT;
    aqk_out[((t0 + r) * H + h) * BT + j] = sA[r * 65 + j];
  }
  if (tid < K) gc_out[(c * H + h) * K + tid] = ex(GC[tid], base2);
  __syncthreads();

  // 5. v.beta into sQ, k^.beta.e^G into sK.
  for (int i = tid; i < BT * V; i += 256) {
    const int r = i / V, cc = i % V;
    const float vv = (r < len) ? to_f32(v[((t0 + r) * H + h) * (int64_t)V + cc]) : 0.f;
    sQ[r * XP + cc] = vv * sB[r];
  }
  for (int i = tid; i < BT * K; i += 256) {
    const int r = i / K, cc = i % K;
    sK[r * KP + cc] = sK[r * KP + cc] * sB[r] * ex(sG[r * KP + cc], base2);
  }

  // 6. (I + L)^-1 by forward substitution, four lanes per column.
  {
    const int col = tid >> 2, part = tid & 3;
    for (int i = 0; i < BT; ++i) {
      float acc = 0.f;
      for (int m = col + part; m < i; m += 4) acc = fmaf(sL[i * 65 + m], sA[m * 65 + col], acc);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (part == 0) sA[i * 65 + col] = (i == col) ? 1.f : (i > col ? -acc : 0.f);
      __syncwarp();
    }
  }
  __syncthreads();

  // 7. w = A (k^.beta.e^G), u = A (v.beta): one thread per output column.
  for (int col = tid; col < K + V; col += 256) {
    const bool isw = col < K;
    const int cc = isw ? col : col - K;
    const float *src = isw ? (sK + cc) : (sQ + cc);
    const int stride = isw ? KP : XP;
    for (int r = 0; r < len; ++r) {
      float acc = 0.f;
      for (int j = 0; j <= r; ++j) acc = fmaf(sA[r * 65 + j], src[j * stride], acc);
      if (isw) w_out[((t0 + r) * H + h) * (int64_t)K + cc] = acc;
      else u_out[((t0 + r) * H + h) * (int64_t)V + cc] = acc;
    }
  }
}

// ---------------------------------------------------------------------------
// Inter-chunk chain: one CTA per (range, head, 32-column tile of the state).
// In summary mode the state is the augmented [S~ | M] (d_v + d_k columns):
// the M columns start from the identity and see u = 0, so that after the
// range they hold the product of the per-chunk transitions.
// ---------------------------------------------------------------------------
constexpr int VT = 32;

template <typename Tout, int K>
__global__ void __launch_bounds__(256)
generic_inter_kernel(bool summary, SeqInfo s, int H, int V, const float *__restrict__ w,
                     const float *__restrict__ u, const float *__restrict__ qg,
                     const float *__restrict__ kg, const float *__restrict__ aqk,
                     const float *__restrict__ gc, InterOut io) {
  extern __shared__ float smem[];
  float *sH = smem;              // [K][VT]
  float *sW = sH + K * VT;       // [64][K]
  float *sQg = sW + BT * K;      // [64][K]
  float *sKg = sQg + BT * K;     // [64][K]
  float *sU = sKg + BT * K;      // [64][VT]
  float *sVn = sU + BT * VT;     // [64][VT]
  float *sA = sVn + BT * VT;     // [64][64]
  float *sGc = sA + BT * BT;     // [K]

  const int n = blockIdx.x / H, h = blockIdx.x % H;
  const int tid = threadIdx.x, j = tid & (VT - 1), rb = tid >> 5;
  const int col = blockIdx.y * VT + j;  // column of the (augmented) state
  int64_t t0, t1;
  seq_range(s, n, t0, t1);
  const int64_t c0 = seq_first_chunk(s, n);
  const int64_t unit = (int64_t)n * H + h;

  for (int cc = rb; cc < K; cc += 8) {
    float x;
    if (summary) x = (col >= V && cc == col - V) ? 1.f : 0.f;
    else x = io.initial_state ? io.initial_state[(unit * K + cc) * V + col] : 0.f;
    sH[cc * VT + j] = x;
  }

  int64_t ci = c0;
  for (int64_t t = t0; t < t1; t += BT, ++ci) {
    const int len = (int)((t1 - t) < BT ? (t1 - t) : BT);
    __syncthreads();  // previous chunk done with the tiles
    for (int i = tid; i < BT * K; i += 256) {
      const int r = i / K, cc = i % K;
      const bool in = r < len;
      const int64_t off = ((t + r) * H + h) * (int64_t)K + cc;
      sW[i] = in ? w[off] : 0.f;
      sKg[i] = in ? kg[off] : 0.f;
      if (!summary) sQg[i] = in ? qg[off] : 0.f;
    }
    for (int r = rb; r < BT; r += 8)
      sU[r * VT + j] = (r < len && col < V) ? u[((t + r) * H + h) * (int64_t)V + col] : 0.f;
    if (!summary)
      for (int i = tid; i < BT * BT; i += 256) {
        const int r = i / BT;
        sA[i] = r < len ? aqk[((t + r) * H + h) * BT + (i % BT)] : 0.f;
      }
    for (int cc = tid; cc < K; cc += 256) sGc[cc] = gc[(ci * H + h) * K + cc];
    if (!summary && io.h_out)
      for (int cc = rb; cc < K; cc += 8)
        io.h_out[((ci * H + h) * K + cc) * V + col] = sH[cc * VT + j];
    __syncthreads();

    // v_new = u - w h
    for (int r = rb; r < BT; r += 8) {
      float acc = sU[r * VT + j];
      for (int cc = 0; cc < K; ++cc) acc = fmaf(-sW[r * K + cc], sH[cc * VT + j], acc);
      sVn[r * VT + j] = acc;
    }
    __syncthreads();

    // o = qg h + Aqk v_new
    if (!summary) {
      for (int r = rb; r < len; r += 8) {
        float acc = 0.f;
        for (int cc = 0; cc < K; ++cc) acc = fmaf(sQg[r * K + cc], sH[cc * VT + j], acc);
        for (int s2 = 0; s2 <= r; ++s2) acc = fmaf(sA[r * BT + s2], sVn[s2 * VT + j], acc);
        const int64_t off = ((t + r) * H + h) * (int64_t)V + col;
        if (io.out) static_cast<Tout *>(io.out)[off] = from_f32<Tout>(acc);
        if (io.v_new_out) io.v_new_out[off] = sVn[r * VT + j];
      }
      __syncthreads();
    }

    // h' = e^{G_C} h + kg^T v_new
    for (int cc = rb; cc < K; cc += 8) {
      float acc = sGc[cc] * sH[cc * VT + j];
      for (int r = 0; r < len; ++r) acc = fmaf(sKg[r * K + cc], sVn[r * VT + j], acc);
      sH[cc * VT + j] = acc;
    }
  }
  __syncthreads();
  for (int cc = rb; cc < K; cc += 8) {
    const float x = sH[cc * VT + j];
    if (summary) {
      if (col < V) io.S_tilde[(unit * K + cc) * V + col] = x;
      else io.M[(unit * K + cc) * K + (col - V)] = x;
    } else if (io.final_state) {
      io.final_state[(unit * K + cc) * V + col] = x;
    }
  }
}

template <typename Tin, int K, int V>
cudaError_t intra_dispatch(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, const GateParams &gp, const SeqInfo &s,
                           const FwdPlan &p, char *ws, cudaStream_t st) {
  constexpr int KP = K + 1, XP = (K > V ? K : V) + 1;
  const size_t smem = sizeof(float) * (64 * XP + 2 * 64 * KP + 2 * 64 * 65 + 64);
  auto kern = generic_intra_kernel<Tin, K, V>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (p.nchunks == 0) return cudaSuccess;
  dim3 grid((unsigned)p.nchunks, p.H);
  kern<<<grid, 256, smem, st>>>(
      static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v), g,
      beta, gp, s, p.H, p.Hk, reinterpret_cast<float *>(ws + p.off_w),
      reinterpret_cast<float *>(ws + p.off_u), reinterpret_cast<float *>(ws + p.off_qg),
      reinterpret_cast<float *>(ws + p.off_kg), reinterpret_cast<float *>(ws + p.off_aqk),
      reinterpret_cast<float *>(ws + p.off_gc));
  return cudaGetLastError();
}

template <typename Tout, int K>
cudaError_t inter_dispatch(bool summary, const InterOut &io, const SeqInfo &s, const FwdPlan &p,
                           const char *ws, cudaStream_t st) {
  const size_t smem = sizeof(float) * (K * VT + 3 * BT * K + 2 * BT * VT + BT * BT + K);
  auto kern = generic_inter_kernel<Tout, K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int cols = summary ? p.V + K : p.V;
  dim3 grid((unsigned)((int64_t)p.N * p.H), cols / VT);
  if (grid.x == 0) return cudaSuccess;
  kern<<<grid, 256, smem, st>>>(
      summary, s, p.H, p.V, reinterpret_cast<const float *>(ws + p.off_w),
      reinterpret_cast<const float *>(ws + p.off_u), reinterpret_cast<const float *>(ws + p.off_qg),
      reinterpret_cast<const float *>(ws + p.off_kg), reinterpret_cast<const float *>(ws + p.off_aqk),
      reinterpret_cast<const float *>(ws + p.off_gc), io);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_map(const SeqInfo &s, int32_t *chunk_off, cudaStream_t st) {
  chunk_map_kernel<<<1, 1024, 0, st>>>(s, chunk_off);
  return cudaGetLastError();
}

cudaError_t launch_generic_intra(kda_dtype dt, const void *q, const void *k, const void *v,
                                 const float *g, const float *beta, const GateParams &gp,
                                 const SeqInfo &s, const FwdPlan &p, char *ws, cudaStream_t st) {
#define KDA_INTRA(T_, K_, V_) \
  if (p.K == K_ && p.V == V_) return intra_dispatch<T_, K_, V_>(q, k, v, g, beta, gp, s, p, ws, st);
  if (dt == KDA_F32) {
    KDA_INTRA(float, 64, 64) KDA_INTRA(float, 64, 128) KDA_INTRA(float, 128, 64) KDA_INTRA(float, 128, 128)
  } else {
    KDA_INTRA(__nv_bfloat16, 64, 64) KDA_INTRA(__nv_bfloat16, 64, 128)
    KDA_INTRA(__nv_bfloat16, 128, 64) KDA_INTRA(__nv_bfloat16, 128, 128)
  }
#undef KDA_INTRA
  return cudaErrorInvalidValue;
}

cudaError_t launch_generic_inter(kda_dtype dt, bool summary, const InterOut &io, const SeqInfo &s,
                                 const FwdPlan &p, const char *ws, cudaStream_t st) {
  if (dt == KDA_F32) {
    if (p.K == 64) return inter_dispatch<float, 64>(summary, io, s, p, ws, st);
    if (p.K == 128) return inter_dispatch<float, 128>(summary, io, s, p, ws, st);
  } else {
    if (p.K == 64) return inter_dispatch<__nv_bfloat16, 64>(summary, io, s, p, ws, st);
    if (p.K == 128) return inter_dispatch<__nv_bfloat16, 128>(summary, io, s, p, ws, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kda
