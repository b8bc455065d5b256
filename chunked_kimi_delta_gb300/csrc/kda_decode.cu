// kda_decode.cu - recurrent decode step on states kept in a cache pool.
//
// The token-by-token form of the KDA recurrence ("KDA Chunk Backward -
// TPU/Pallas Kernel Design" section 1; the decode path named in the
// vllm-ascend KDA prefill state copy article, "背景"), run in place on the
// rows of a state pool: for each selected sequence i and head h,
//   S = row idx[i] of the pool (zero if the row is invalid or its flag false)
//   for each new token t:  S = Diag(alpha_t) S;  delta = v_t - S^T k^_t;
//                          S += beta_t k^_t delta^T;  o_t = scale S^T q^_t
//   row idx[i] = S  (when the row is valid)
// with alpha, k^, q^, beta from the same gate / L2 norm / sigmoid as the
// chunked forward.  All arithmetic in fp32.
//
// One CTA per (sequence, head): each thread holds 4 adjacent columns of the
// state for a group of rows in registers (16-byte loads and stores when the
// pool allows); the two dot products per token (S^T k^, S^T q^) reduce
// inside each thread and then across the row groups through shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecThreads = 256;
constexpr int kMaxD = 128;

template <typename T> __device__ __forceinline__ float ldf(const T *p) { return to_f32<T>(*p); }

// 4 consecutive state elements of a row: 16-byte (fp32) or 8-byte (bf16) access.
__device__ __forceinline__ void ld4(const float *p, float (&x)[4]) {
  const float4 v = *reinterpret_cast<const float4 *>(p);
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void ld4(const __nv_bfloat16 *p, float (&x)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2 *>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}
__device__ __forceinline__ void st4(float *p, const float (&x)[4]) {
  *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ void st4(__nv_bfloat16 *p, const float (&x)[4]) {
  __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
  uint2 raw;
  raw.x = *reinterpret_cast<uint32_t *>(&a);
  raw.y = *reinterpret_cast<uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p) = raw;
}

// Element-wise forms for states that are not 16-byte aligned.
template <typename Tc>
__device__ __forceinline__ void ld4_any(const Tc *p, float (&x)[4], bool vec) {
  if (vec) {
    ld4(p, x);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = to_f32<Tc>(p[j]);
  }
}
template <typename Tc>
__device__ __forceinline__ void st4_any(Tc *p, const float (&x)[4], bool vec) {
  if (vec) {
    st4(p, x);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) p[j] = from_f32<Tc>(x[j]);
  }
}

// One CTA per (sequence, head, slice of VS value columns): the columns of
// the state evolve independently (the gate acts on rows, k^ and q^ are
// shared), so splitting them spreads a state over several CTAs, each with
// fewer registers, and more CTAs stay resident per SM.
// Thread = (column quad cq: slice columns 4 cq .. 4 cq + 3, row group rg: R
// rows).  VEC: the pool base and row stride are 16-byte aligned, so each
// thread's 4 elements move as one 16-byte (fp32) or 8-byte (bf16) access.
template <typename Tin, typename Tc, typename Tidx, int K, int V, int VS, bool VEC>
__global__ void __launch_bounds__(kDecThreads, 2)
decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
              const float *__restrict__ g, const float *__restrict__ beta, GateParams gp,
              Tin *__restrict__ out, Tc *cache, int64_t num_rows, int64_t row_stride,
              const Tidx *__restrict__ idx, const bool *__restrict__ init_flags, int T, int H,
              int Hk, bool vfirst) {
  constexpr int NQ = VS / 4;                // column quads of the slice
  constexpr int RG = kDecThreads / NQ;      // row groups
  constexpr int R = K / RG;                 // rows per thread
  constexpr int NS = V / VS;                // slices per state
  static_assert(R >= 1 && R * RG == K && 2 * K <= kDecThreads && VS <= kDecThreads, "thread layout");
  __shared__ float s_k[kMaxD], s_q[kMaxD], s_a[kMaxD], s_v[kMaxD];
  __shared__ __align__(16) float s_part[RG][VS];
  __shared__ float s_red[2][8];
  __shared__ float s_beta;

  const int tid = threadIdx.x;
  const int cq = tid % NQ, rg = tid / NQ;
  const int64_t unit = blockIdx.x / NS;
  const int c0 = (int)(blockIdx.x % NS) * VS;  // first value column of the slice
  const int n = (int)(unit / H), h = (int)(unit % H);
  const int64_t row = (int64_t)idx[n];
  const bool valid = row >= 0 && row < num_rows;
  const bool load = valid && (!init_flags || init_flags[n]);
  Tc *state = cache + (valid ? row * row_stride : 0) + (int64_t)h * K * V;
  Tc *mine = state + (int64_t)(R * rg) * V + c0 + 4 * cq;  // this thread's first element
  // V-first pool states ([V, K] per head): element (row, column) at column * K + row
  Tc *mine_vf = state + (int64_t)(c0 + 4 * cq) * K + R * rg;

  float s[R][4];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (!load) {
      s[r][0] = s[r][1] = s[r][2] = s[r][3] = 0.f;
    } else if (vfirst) {
#pragma unroll
      for (int j = 0; j < 4; ++j) s[r][j] = to_f32<Tc>(mine_vf[(int64_t)j * K + r]);
    } else {
      ld4_any(mine + (int64_t)r * V, s[r], VEC);
    }
  }

  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;
  const bool l2n = (gp.flags & KDA_L2NORM_QK) != 0;
  const bool sig = (gp.flags & KDA_BETA_SIGMOID) != 0;
  const float A_h = gate ? expf(gp.a_log[h]) : 0.f;
  const int warp = tid >> 5, lane = tid & 31;

  // Column sums of the RG partials in s_part for this thread's 4 columns.
  auto col_sums = [&](float (&sum)[4]) {
    sum[0] = sum[1] = sum[2] = sum[3] = 0.f;
#pragma unroll
    for (int x = 0; x < RG; ++x) {
      const float4 pv = *reinterpret_cast<const float4 *>(&s_part[x][4 * cq]);
      sum[0] += pv.x; sum[1] += pv.y; sum[2] += pv.z; sum[3] += pv.w;
    }
  };

  for (int t = 0; t < T; ++t) {
    const int64_t tok = ((int64_t)n * T + t) * H + h;              // token-head index
    const int64_t tokk = ((int64_t)n * T + t) * Hk + h / (H / Hk);  // and of q, k
    // ---- stage the token: gate, raw q / k (norms below), this slice of v, beta
    float kq2 = 0.f;  // k^2 (threads < K) or q^2 (threads K .. 2K-1)
    if (tid < K) {
      const float kc = ldf(k + tokk * K + tid);
      s_k[tid] = kc;
      kq2 = kc * kc;
      float gv = g[tok * K + tid];
      if (gate) {
        const float z = gv + (gp.dt_bias ? gp.dt_bias[h * K + tid] : 0.f);
        gv = -A_h * (fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))));  // -exp(a_log) softplus(z)
      }
      s_a[tid] = expf(gv);
    } else if (tid < 2 * K) {
      const float qc = ldf(q + tokk * K + (tid - K));
      s_q[tid - K] = qc;
      kq2 = qc * qc;
    }
    if (tid < VS) s_v[tid] = ldf(v + tok * V + c0 + tid);
    if (tid == 0) {
      const float b = beta[tok];
      s_beta = sig ? 1.f / (1.f + expf(-b)) : b;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) kq2 += __shfl_xor_sync(0xffffffffu, kq2, o);
    if (lane == 0 && warp < 2 * K / 32) s_red[warp * 32 < K ? 0 : 1][warp % (K / 32)] = kq2;
    __syncthreads();
    float nk = 0.f, nq = 0.f;
#pragma unroll
    for (int w = 0; w < K / 32; ++w) {
      nk += s_red[0][w];
      nq += s_red[1][w];
    }
    const float rk = l2n ? rsqrtf(nk + gp.eps) : 1.f;
    const float rq = (l2n ? rsqrtf(nq + gp.eps) : 1.f) * gp.scale;
    const float bt = s_beta;

    // ---- S = Diag(alpha) S; partial (S^T k^) over this thread's rows
    {
      float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int kr = R * rg + r;
        const float a = s_a[kr], kk = s_k[kr] * rk;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s[r][j] *= a;
          p[j] = fmaf(s[r][j], kk, p[j]);
        }
      }
      *reinterpret_cast<float4 *>(&s_part[rg][4 * cq]) = make_float4(p[0], p[1], p[2], p[3]);
    }
    __syncthreads();
    // ---- delta = v - S^T k^; S += beta k^ delta^T; partial (S^T q^)
    {
      float sk[4];
      col_sums(sk);
      float bd[4], po[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j) bd[j] = bt * (s_v[4 * cq + j] - sk[j]);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int kr = R * rg + r;
        const float kk = s_k[kr] * rk, qq = s_q[kr];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s[r][j] = fmaf(bd[j], kk, s[r][j]);
          po[j] = fmaf(s[r][j], qq, po[j]);
        }
      }
      __syncthreads();  // every read of s_part (delta) is done
      *reinterpret_cast<float4 *>(&s_part[rg][4 * cq]) = make_float4(po[0], po[1], po[2], po[3]);
    }
    __syncthreads();
    if (rg == 0) {
      float so[4];
      col_sums(so);
#pragma unroll
      for (int j = 0; j < 4; ++j) out[tok * V + c0 + 4 * cq + j] = from_f32<Tin>(rq * so[j]);
    }
    __syncthreads();  // staging buffers are rewritten by the next token
  }

  if (valid) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (vfirst) {
#pragma unroll
        for (int j = 0; j < 4; ++j) mine_vf[(int64_t)j * K + r] = from_f32<Tc>(s[r][j]);
      } else {
        st4_any(mine + (int64_t)r * V, s[r], VEC);
      }
    }
  }
}

// Value columns per CTA: the whole state (measured on the 64 x 32 pool step:
// 58 us with one CTA per state, 76 us with two, 117 us with four - each
// slice repeats the token staging and its barriers).

template <typename Tin, typename Tc, typename Tidx>
cudaError_t dispatch_kv(int dk, int dv, bool aligned, int64_t units, cudaStream_t st, const void *q,
                        const void *k, const void *v, const float *g, const float *beta,
                        const GateParams &gp, void *out, void *cache, int64_t num_rows,
                        int64_t row_stride, const void *idx, const bool *init_flags, int T, int H,
                        int Hk, bool vfirst) {
  const Tin *qq = static_cast<const Tin *>(q), *kk = static_cast<const Tin *>(k),
            *vv = static_cast<const Tin *>(v);
#define KDA_DEC(KK, VV, VEC)                                                                      \
  decode_kernel<Tin, Tc, Tidx, KK, VV, VV, VEC>                                                   \
      <<<(unsigned)units, kDecThreads, 0, st>>>(                                                  \
          qq, kk, vv, g, beta, gp, static_cast<Tin *>(out), static_cast<Tc *>(cache), num_rows,     \
          row_stride, static_cast<const Tidx *>(idx), init_flags, T, H, Hk, vfirst)
#define KDA_DEC2(KK, VV)              \
  if (aligned) KDA_DEC(KK, VV, true); \
  else KDA_DEC(KK, VV, false)
  if (dk == 128 && dv == 128) { KDA_DEC2(128, 128); }
  else if (dk == 128 && dv == 64) { KDA_DEC2(128, 64); }
  else if (dk == 64 && dv == 128) { KDA_DEC2(64, 128); }
  else { KDA_DEC2(64, 64); }
#undef KDA_DEC2
#undef KDA_DEC
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(kda_dtype qkv_dtype, kda_dtype cache_dtype, kda_index_dtype idx_dtype,
                          int dk, int dv, int N, int T, int H, int Hk, const void *q, const void *k,
                          const void *v, const float *g, const float *beta, const GateParams &gp,
                          void *out, void *cache, int64_t num_rows, int64_t row_stride,
                          const void *idx, const bool *init_flags, bool vfirst, cudaStream_t st) {
  const int64_t units = (int64_t)N * H;
  if (units == 0) return cudaSuccess;
  // vector accesses need 16-byte aligned states: the pool base and the row
  // stride (a state's offset inside a row, h*dk*dv elements, and each
  // thread's column quad are multiples of 16 bytes)
  const size_t esz = cache_dtype == KDA_BF16 ? 2 : 4;
  const bool aligned = !vfirst && (reinterpret_cast<uintptr_t>(cache) & 15u) == 0 &&
                       ((size_t)row_stride * esz) % 16 == 0;
#define KDA_DEC_IDX(TI, TC, TX)                                                                     \
  return dispatch_kv<TI, TC, TX>(dk, dv, aligned, units, st, q, k, v, g, beta, gp, out, cache,       \
                                 num_rows, row_stride, idx, init_flags, T, H, Hk, vfirst)
  const bool ibf = qkv_dtype == KDA_BF16, cbf = cache_dtype == KDA_BF16, i64 = idx_dtype == KDA_I64;
  if (ibf && cbf && i64) KDA_DEC_IDX(__nv_bfloat16, __nv_bfloat16, int64_t);
  if (ibf && cbf) KDA_DEC_IDX(__nv_bfloat16, __nv_bfloat16, int32_t);
  if (ibf && i64) KDA_DEC_IDX(__nv_bfloat16, float, int64_t);
  if (ibf) KDA_DEC_IDX(__nv_bfloat16, float, int32_t);
  if (cbf && i64) KDA_DEC_IDX(float, __nv_bfloat16, int64_t);
  if (cbf) KDA_DEC_IDX(float, __nv_bfloat16, int32_t);
  if (i64) KDA_DEC_IDX(float, float, int64_t);
  KDA_DEC_IDX(float, float, int32_t);
#undef KDA_DEC_IDX
}

}  // namespace kda
