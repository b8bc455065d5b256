// kda_tc_exact.cu - exact intra-chunk stage for chunks under strong decay.
//
// The tensor-core prep (kda_tc_prep.cu) factors every decay 2^{G_r - G_j}
// of the A_kk / A_qk products into a row part 2^{G_r - b} and a column part
// 2^{b - G_j} around a reference gate b per 16-token sub-block ("KDA Chunk
// Backward - TPU/Pallas Kernel Design", section 3.7).  Inside a sub-block the
// two parts grow with the sub-block's own decay; past about 2^126 they leave
// the fp32 / bf16 range, and the product, whose true value may be anywhere up
// to 1 (the diagonal of A_qk is exactly 1 before scaling), is lost.  The
// prep therefore lists every (chunk, head) in which some channel's
// chunk-local gate moves by more than STRONG_DECAY_LOG2 inside one sub-block
// (far inside the range, so that the parts it builds for the other items
// are exact up to rounding).  This kernel recomputes each listed item from
// exponentials of exact gate differences on the CUDA cores, in fp32, and
// overwrites the item's whole package and, for the backward, its
// A = (I + L)^-1.  Formulas (same design, sections 1 and 1.2), with G the
// chunk-local inclusive cumulative gate in log2 units:
//   L_rj   = beta_r sum_c k^_rc k^_jc 2^{G_rc - G_jc}         (j < r)
//   Aqk_rj = scale sum_c q^_rc k^_jc 2^{G_rc - G_jc}         (j <= r)
//   A = (I + L)^-1,  w = A (k^ . beta . 2^G),  u = A (v . beta)
//   qg = scale q^ . 2^G,  kg = k^ . 2^{G_C - G},  gC = 2^{G_C}
#include <cuda_bf16.h>

#include "kda_tc.cuh"

namespace kda {
namespace tcp {
namespace {

constexpr int NT = 256;
constexpr int RS = 129;  // fp32 row stride of the [64][128] tiles
constexpr int AS = 65;   // fp32 row stride of the [64][64] tiles
constexpr float kLog2e = 1.4426950408889634f;

// shared memory, in floats
constexpr int O_Q = 0;              // scale q^ [64][RS]
constexpr int O_K = O_Q + 64 * RS;  // k^, later k^ beta 2^G
constexpr int O_G = O_K + 64 * RS;  // G (log2) [64][RS]
constexpr int O_V = O_G + 64 * RS;  // v, later v beta
constexpr int O_L = O_V + 64 * RS;  // L [64][AS]
constexpr int O_A = O_L + 64 * AS;  // (I + L)^-1
constexpr int O_P = O_A + 64 * AS;  // Aqk
constexpr int O_B = O_P + 64 * AS;  // beta [64]
constexpr int SMEM_FLOATS = O_B + 64;
constexpr size_t SMEM_BYTES = sizeof(float) * SMEM_FLOATS;

__device__ __forceinline__ void st_bf16(char *pk, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16 *>(pk + off) = __float2bfloat16_rn(x);
}

__global__ void __launch_bounds__(NT, 1)
tc_prep_exact_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                     const __nv_bfloat16 *__restrict__ v, const float *__restrict__ x,
                     const float *__restrict__ beta, GateParams gp, SeqInfo s, int H, int Hk,
                     const uint32_t *__restrict__ count, const uint32_t *__restrict__ list,
                     char *__restrict__ pkg, float *__restrict__ a_out) {
  extern __shared__ float sm[];
  float *sQ = sm + O_Q, *sK = sm + O_K, *sG = sm + O_G, *sV = sm + O_V;
  float *sL = sm + O_L, *sA = sm + O_A, *sP = sm + O_P, *sB = sm + O_B;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;
  const bool l2n = (gp.flags & KDA_L2NORM_QK) != 0;
  const bool sig = (gp.flags & KDA_BETA_SIGMOID) != 0;
  const uint32_t n_items = *count;

  for (uint32_t idx = blockIdx.x; idx < n_items; idx += gridDim.x) {
    __syncthreads();  // the previous item is done with shared memory
    const uint32_t wi = list[idx];
    const int64_t gc = wi / (uint32_t)H;
    const int h = (int)(wi % (uint32_t)H), hk = h / (H / Hk);
    int n, len;
    int64_t t0;
    if (!chunk_lookup(s, gc, n, t0, len)) continue;  // uniform over the CTA
    char *pk = pkg + (size_t)(gc * H + h) * PK_BYTES;

    // 1. inputs; the gate in log2 units (rows past the chunk end: zero)
    const float A_h = gate ? expf(gp.a_log[h]) : 0.f;
    for (int i = tid; i < BT * K; i += NT) {
      const int r = i >> 7, c = i & 127;
      float qv = 0.f, kv = 0.f, vv = 0.f, g = 0.f;
      if (r < len) {
        const int64_t tk = ((t0 + r) * Hk + hk) * (int64_t)K + c;
        const int64_t tv = ((t0 + r) * H + h) * (int64_t)K + c;
        qv = __bfloat162float(q[tk]);
        kv = __bfloat162float(k[tk]);
        vv = __bfloat162float(v[tv]);
        g = x[tv];
        if (gate) {
          const float z = g + (gp.dt_bias ? gp.dt_bias[h * K + c] : 0.f);
          g = -A_h * (fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))));
        }
        g *= kLog2e;
      }
      sQ[r * RS + c] = qv;
      sK[r * RS + c] = kv;
      sV[r * RS + c] = vv;
      sG[r * RS + c] = g;
    }
    if (tid < BT) {
      float b = 0.f;
      if (tid < len) {
        b = beta[(t0 + tid) * H + h];
        if (sig) b = 1.f / (1.f + expf(-b));
      }
      sB[tid] = b;
    }
    __syncthreads();

    // 2. row norms (the attention scale rides on q^), chunk-local cumsum
    for (int r = warp; r < BT; r += NT / 32) {
      float sq = 0.f, sk = 0.f;
      for (int c = lane; c < K; c += 32) {
        sq = fmaf(sQ[r * RS + c], sQ[r * RS + c], sq);
        sk = fmaf(sK[r * RS + c], sK[r * RS + c], sk);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      const float rq = (l2n ? rsqrtf(sq + gp.eps) : 1.f) * gp.scale;
      const float rk = l2n ? rsqrtf(sk + gp.eps) : 1.f;
      for (int c = lane; c < K; c += 32) {
        sQ[r * RS + c] *= rq;
        sK[r * RS + c] *= rk;
      }
    }
    if (tid < K) {
      float acc = 0.f;
      for (int r = 0; r < BT; ++r) {
        acc += sG[r * RS + tid];
        sG[r * RS + tid] = acc;
      }
    }
    __syncthreads();

    // 3. L and Aqk over the 2080 pairs j <= r, exponentials of the exact
    //    differences (every factor <= 1 for a decaying gate)
    for (int p = tid; p < BT * (BT + 1) / 2; p += NT) {
      int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
      while ((r + 1) * (r + 2) / 2 <= p) ++r;
      while (r * (r + 1) / 2 > p) --r;
      const int j = p - r * (r + 1) / 2;
      float kk = 0.f, qk = 0.f;
      for (int c = 0; c < K; ++c) {
        const float kj = sK[j * RS + c] * exp2f(sG[r * RS + c] - sG[j * RS + c]);
        kk = fmaf(sK[r * RS + c], kj, kk);
        qk = fmaf(sQ[r * RS + c], kj, qk);
      }
      sL[r * AS + j] = j < r ? sB[r] * kk : 0.f;
      sP[r * AS + j] = qk;
    }
    for (int i = tid; i < BT * BT; i += NT) {
      const int r = i >> 6, j = i & 63;
      if (j > r) {
        sL[r * AS + j] = 0.f;
        sP[r * AS + j] = 0.f;
      }
    }
    __syncthreads();

    // 4. the package parts that need q^, k^ and G as they are: qg, kg
    //    (rows past the end are zero), Aqk, gC
    for (int i = tid; i < BT * K; i += NT) {
      const int r = i >> 7, c = i & 127;
      const float G = sG[r * RS + c], GC = sG[(BT - 1) * RS + c];
      st_bf16(pk, PK_WQ + kmaj_off(128, r, c), sQ[r * RS + c] * exp2f(G));
      st_bf16(pk, PK_KG + mnmaj_off(64, r, c), sK[r * RS + c] * exp2f(GC - G));
    }
    for (int i = tid; i < BT * BT; i += NT) {
      const int r = i >> 6, j = i & 63;
      st_bf16(pk, PK_AQK + kmaj_off(64, r, j), sP[r * AS + j]);
    }
    if (tid < K)
      reinterpret_cast<float *>(pk + PK_GC)[tid] = exp2f(sG[(BT - 1) * RS + tid]);
    __syncthreads();

    // 5. right-hand sides k^ beta 2^G and v beta, in place
    for (int i = tid; i < BT * K; i += NT) {
      const int r = i >> 7, c = i & 127;
      sK[r * RS + c] *= sB[r] * exp2f(sG[r * RS + c]);
      sV[r * RS + c] *= sB[r];
    }
    // 6. (I + L)^-1 by forward substitution, four lanes per column
    {
      const int col = tid >> 2, part = tid & 3;
      for (int i = 0; i < BT; ++i) {
        float acc = 0.f;
        for (int m = col + part; m < i; m += 4) acc = fmaf(sL[i * AS + m], sA[m * AS + col], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        if (part == 0) sA[i * AS + col] = (i == col) ? 1.f : (i > col ? -acc : 0.f);
        __syncwarp();
      }
    }
    __syncthreads();

    // 7. w = A (k^ beta 2^G) -> WQ rows 64..127, u = A (v beta) -> U: one
    //    thread per output column; rows past the end come out zero (their
    //    beta and k^ are zero)
    {
      const bool isw = tid < K;
      const int c = tid & 127;
      const float *src = isw ? sK : sV;
      for (int r = 0; r < BT; ++r) {
        float acc = 0.f;
        for (int j = 0; j <= r; ++j) acc = fmaf(sA[r * AS + j], src[j * RS + c], acc);
        if (isw) st_bf16(pk, PK_WQ + kmaj_off(128, 64 + r, c), acc);
        else st_bf16(pk, PK_U + u_offset(r, c), acc);
      }
    }
    if (a_out) {
      float *dst = a_out + (size_t)(gc * H + h) * (BT * BT);
      for (int i = tid; i < BT * BT; i += NT) {
        const int r = i >> 6, j = i & 63;
        dst[i] = (r < len && j <= r) ? sA[r * AS + j] : 0.f;
      }
    }
  }
}

}  // namespace

cudaError_t launch_tc_prep_exact(const void *q, const void *k, const void *v, const float *x,
                                 const float *beta, const GateParams &gp, const SeqInfo &s,
                                 int64_t nitems, int H, int Hk, const uint32_t *flag_count,
                                 const uint32_t *flag_list, char *pkg, float *a_out, cudaStream_t st) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  cudaError_t e = cudaFuncSetAttribute(tc_prep_exact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (nitems == 0) return cudaSuccess;
  const int grid = (int)(nitems < sms ? nitems : sms);
  tc_prep_exact_kernel<<<grid, NT, SMEM_BYTES, st>>>(
      static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
      static_cast<const __nv_bfloat16 *>(v), x, beta, gp, s, H, Hk, flag_count, flag_list, pkg, a_out);
  return cudaGetLastError();
}

}  // namespace tcp
}  // namespace kda
