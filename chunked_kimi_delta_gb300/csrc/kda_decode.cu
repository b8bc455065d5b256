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
// One CTA per (sequence, head): thread (v, half) holds column v of the
// state for the 64 key channels of its half in registers; the two dot
// products per token (S^T k^, S^T q^) reduce inside each thread and then
// across the two halves through shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecThreads = 256;
constexpr int kMaxD = 128;

template <typename T> __device__ __forceinline__ float ldf(const T *p) { return to_f32<T>(*p); }

template <typename Tin, typename Tc, typename Tidx, int K, int V>
__global__ void __launch_bounds__(kDecThreads)
decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
              const float *__restrict__ g, const float *__restrict__ beta, GateParams gp,
              Tin *__restrict__ out, Tc *cache, int64_t num_rows, int64_t row_stride,
              const Tidx *__restrict__ idx, const bool *__restrict__ init_flags, int T, int H) {
  static_assert(2 * V <= kDecThreads && K % 2 == 0, "thread layout");
  __shared__ float s_k[kMaxD], s_q[kMaxD], s_a[kMaxD], s_v[kMaxD];
  __shared__ float s_part[2][kMaxD];
  __shared__ float s_red[2][8];
  __shared__ float s_beta;

  const int tid = threadIdx.x;
  const int cv = tid % V, half = tid / V;        // column of the state, half of its rows
  const bool active = half < 2;                  // V = 64: threads 128..255 hold nothing
  constexpr int R = K / 2;                        // rows per thread
  const int n = blockIdx.x / H, h = blockIdx.x % H;
  const int64_t row = (int64_t)idx[n];
  const bool valid = row >= 0 && row < num_rows;
  const bool load = valid && (!init_flags || init_flags[n]);
  Tc *state = cache + (valid ? row * row_stride : 0) + (int64_t)h * K * V;

  float s[R];
#pragma unroll
  for (int r = 0; r < R; ++r)
    s[r] = (active && load) ? to_f32<Tc>(state[(int64_t)(R * half + r) * V + cv]) : 0.f;

  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;
  const bool l2n = (gp.flags & KDA_L2NORM_QK) != 0;
  const bool sig = (gp.flags & KDA_BETA_SIGMOID) != 0;
  const float A_h = gate ? expf(gp.a_log[h]) : 0.f;
  const int warp = tid >> 5, lane = tid & 31;

  for (int t = 0; t < T; ++t) {
    const int64_t tok = ((int64_t)n * T + t) * H + h;  // token-head index
    // ---- stage the token: gate, raw q / k (norms below), v, beta
    float kq2 = 0.f;  // k^2 (threads < K) or q^2 (threads K .. 2K-1)
    if (tid < K) {
      const float kc = ldf(k + tok * K + tid);
      s_k[tid] = kc;
      kq2 = kc * kc;
      float gv = g[tok * K + tid];
      if (gate) {
        const float z = gv + (gp.dt_bias ? gp.dt_bias[h * K + tid] : 0.f);
        gv = -A_h * (fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))));  // -exp(a_log) softplus(z)
      }
      s_a[tid] = expf(gv);
    } else if (tid < 2 * K) {
      const float qc = ldf(q + tok * K + (tid - K));
      s_q[tid - K] = qc;
      kq2 = qc * qc;
    }
    if (tid < V) s_v[tid] = ldf(v + tok * V + tid);
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

    // ---- S = Diag(alpha) S; partial (S^T k^)[cv] over this thread's rows
    float p = 0.f;
    if (active) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int kr = R * half + r;
        s[r] *= s_a[kr];
        p = fmaf(s[r], s_k[kr] * rk, p);
      }
      s_part[half][cv] = p;
    }
    __syncthreads();
    // ---- delta = v - S^T k^; S += beta k^ delta^T; partial (S^T q^)[cv]
    float po = 0.f;
    if (active) {
      const float delta = s_v[cv] - (s_part[0][cv] + s_part[1][cv]);
      const float bd = bt * delta;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int kr = R * half + r;
        s[r] = fmaf(bd, s_k[kr] * rk, s[r]);
        po = fmaf(s[r], s_q[kr], po);
      }
    }
    __syncthreads();  // every read of s_part (delta) is done
    if (active) s_part[half][cv] = po;
    __syncthreads();
    if (active && half == 0) out[tok * V + cv] = from_f32<Tin>(rq * (s_part[0][cv] + s_part[1][cv]));
    __syncthreads();  // staging buffers are rewritten by the next token
  }

  if (active && valid) {
#pragma unroll
    for (int r = 0; r < R; ++r) state[(int64_t)(R * half + r) * V + cv] = from_f32<Tc>(s[r]);
  }
}

template <typename Tin, typename Tc, typename Tidx>
cudaError_t dispatch_kv(int dk, int dv, dim3 grid, cudaStream_t st, const void *q, const void *k,
                        const void *v, const float *g, const float *beta, const GateParams &gp, void *out,
                        void *cache, int64_t num_rows, int64_t row_stride, const void *idx,
                        const bool *init_flags, int T, int H) {
#define KDA_DEC(KK, VV)                                                                            \
  decode_kernel<Tin, Tc, Tidx, KK, VV><<<grid, kDecThreads, 0, st>>>(                              \
      static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v), g, beta, \
      gp, static_cast<Tin *>(out), static_cast<Tc *>(cache), num_rows, row_stride,                  \
      static_cast<const Tidx *>(idx), init_flags, T, H)
  if (dk == 128 && dv == 128) KDA_DEC(128, 128);
  else if (dk == 128 && dv == 64) KDA_DEC(128, 64);
  else if (dk == 64 && dv == 128) KDA_DEC(64, 128);
  else KDA_DEC(64, 64);
#undef KDA_DEC
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(kda_dtype qkv_dtype, kda_dtype cache_dtype, kda_index_dtype idx_dtype,
                          int dk, int dv, int N, int T, int H, const void *q, const void *k,
                          const void *v, const float *g, const float *beta, const GateParams &gp,
                          void *out, void *cache, int64_t num_rows, int64_t row_stride,
                          const void *idx, const bool *init_flags, cudaStream_t st) {
  const dim3 grid((unsigned)((int64_t)N * H));
  if (grid.x == 0) return cudaSuccess;
#define KDA_DEC_IDX(TI, TC, TX)                                                                     \
  return dispatch_kv<TI, TC, TX>(dk, dv, grid, st, q, k, v, g, beta, gp, out, cache, num_rows,     \
                                 row_stride, idx, init_flags, T, H)
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
