// kda_scan.cu - ordered prefix scan of segment affine summaries.
//
// "KDA Context Parallelism (KCP)", "L'algorithme": the state entering segment
// j is rebuilt from the earlier segments' summaries in order,
//     S <- M_j S + S~_j,
// and "Hyper-Parallel Chunk KDA current implementation design" sections 5.3
// and 6.3 compose forward summaries in time (rank) order, in fp32.
//
// One CTA per (chain, head, 16-column tile of the state): the columns of S
// evolve independently (every M_j acts on the left).  The segment loop is
// sequential.  Thread (half, r) owns state row r and the 8 columns of its
// half of the tile in registers; per segment it reads its own row of M_j
// (its column, in the reverse form) straight from L2 four entries at a time
// and the tile's rows from shared memory as warp-wide broadcasts (every lane
// of a warp reads the same row), so one M entry feeds 8 FMAs and one
// broadcast feeds 4 x 8 - in fp32 on the CUDA cores throughout.
//
// The reverse form is the backward twin ("Hyper-Parallel Chunk KDA current
// implementation design" section 5.2; "KDA Chunk Backward - TPU/Pallas Kernel
// Design" section 2.4): the state gradient runs from the last segment to the
// first through the transposed transitions, g <- M_j^T g + E_j.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int CT = 16;  // state columns per CTA

template <int K, bool REVERSE>
__global__ void __launch_bounds__(2 * K)
prefix_scan_kernel(const float *__restrict__ M, const float *__restrict__ St,
                   const float *__restrict__ S0, int S, int H, int V, float *__restrict__ S_in,
                   float *__restrict__ S_final) {
  __shared__ __align__(16) float sS[K * CT];  // the state tile entering the step
  const int ch = blockIdx.x / H, h = blockIdx.x % H;
  const int tid = threadIdx.x;
  const int r = tid % K, half = tid / K;  // a warp shares `half`: broadcast reads
  const int col0 = blockIdx.y * CT + 8 * half;
  const int64_t st0 = (int64_t)ch * H + h;

  float acc[8];
  if (S0) {
    const float4 *src = reinterpret_cast<const float4 *>(S0 + (st0 * K + r) * V + col0);
    const float4 a = src[0], b = src[1];
    acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
    acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
  } else {
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;
  }
  for (int step = 0; step < S; ++step) {
    const int seg = REVERSE ? S - 1 - step : step;
    const int64_t u = ((int64_t)ch * S + seg) * H + h;
    float4 *sin = reinterpret_cast<float4 *>(S_in + (u * K + r) * V + col0);
    sin[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    sin[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    __syncthreads();  // the previous step is done reading sS
    float4 *mine = reinterpret_cast<float4 *>(sS + r * CT + 8 * half);
    mine[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    mine[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    __syncthreads();
    {
      const float4 *st = reinterpret_cast<const float4 *>(St + (u * K + r) * V + col0);
      const float4 a = st[0], b = st[1];
      acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
      acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
    }
    const float *Mu = M + u * K * K;
#pragma unroll 8
    for (int m0 = 0; m0 < K; m0 += 4) {
      float mv[4];
      if (REVERSE) {  // row r of M^T = column r of M: lanes read consecutive entries
#pragma unroll
        for (int i = 0; i < 4; ++i) mv[i] = __ldg(Mu + (m0 + i) * K + r);
      } else {
        const float4 t = __ldg(reinterpret_cast<const float4 *>(Mu + r * K + m0));
        mv[0] = t.x; mv[1] = t.y; mv[2] = t.z; mv[3] = t.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 a = *reinterpret_cast<const float4 *>(sS + (m0 + i) * CT + 8 * half);
        const float4 b = *reinterpret_cast<const float4 *>(sS + (m0 + i) * CT + 8 * half + 4);
        acc[0] = fmaf(mv[i], a.x, acc[0]); acc[1] = fmaf(mv[i], a.y, acc[1]);
        acc[2] = fmaf(mv[i], a.z, acc[2]); acc[3] = fmaf(mv[i], a.w, acc[3]);
        acc[4] = fmaf(mv[i], b.x, acc[4]); acc[5] = fmaf(mv[i], b.y, acc[5]);
        acc[6] = fmaf(mv[i], b.z, acc[6]); acc[7] = fmaf(mv[i], b.w, acc[7]);
      }
    }
  }
  if (S_final) {
    float4 *dst = reinterpret_cast<float4 *>(S_final + (st0 * K + r) * V + col0);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

template <int K>
cudaError_t scan_dispatch(const float *M, const float *St, const float *S0, int C, int S, int H,
                          int V, float *S_in, float *S_final, cudaStream_t st, bool reverse) {
  if (V % CT != 0) return cudaErrorInvalidValue;
  dim3 grid((unsigned)((int64_t)C * H), V / CT);
  if (reverse)
    prefix_scan_kernel<K, true><<<grid, 2 * K, 0, st>>>(M, St, S0, S, H, V, S_in, S_final);
  else
    prefix_scan_kernel<K, false><<<grid, 2 * K, 0, st>>>(M, St, S0, S, H, V, S_in, S_final);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefix_scan(const float *M, const float *S_tilde, const float *S0, int C, int S,
                               int H, int K, int V, float *S_in, float *S_final, cudaStream_t st,
                               bool reverse) {
  if (K == 64) return scan_dispatch<64>(M, S_tilde, S0, C, S, H, V, S_in, S_final, st, reverse);
  if (K == 128) return scan_dispatch<128>(M, S_tilde, S0, C, S, H, V, S_in, S_final, st, reverse);
  return cudaErrorInvalidValue;
}

}  // namespace kda
