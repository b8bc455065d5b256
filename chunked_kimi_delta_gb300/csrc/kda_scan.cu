// kda_scan.cu - ordered prefix scan of segment affine summaries.
//
// "KDA Context Parallelism (KCP)", "L'algorithme": the state entering segment
// j is rebuilt from the earlier segments' summaries in order,
//     S <- M_j S + S~_j,
// and "Hyper-Parallel Chunk KDA current implementation design" sections 5.3
// and 6.3 compose forward summaries in time (rank) order, in fp32.
//
// One CTA per (chain, head, 32-column tile of the state): the columns of S
// evolve independently (every M_j acts on the left).  The segment loop is
// sequential; each step is a K x K by K x 32 product on CUDA cores in fp32,
// with M_j staged in shared memory and the running state held in registers
// (each warp owns K/8 rows of the tile, one column per lane).
//
// The reverse form is the backward twin ("Hyper-Parallel Chunk KDA current
// implementation design" section 5.2; "KDA Chunk Backward - TPU/Pallas Kernel
// Design" section 2.4): the state gradient runs from the last segment to the
// first through the transposed transitions, g <- M_j^T g + E_j.
#include "kda_internal.cuh"

namespace kda {

namespace {

template <int K>
__global__ void __launch_bounds__(256)
prefix_scan_kernel(const float *__restrict__ M, const float *__restrict__ St,
                   const float *__restrict__ S0, int S, int H, int V, float *__restrict__ S_in,
                   float *__restrict__ S_final, bool reverse) {
  constexpr int R = K / 8;  // rows of the tile per warp
  extern __shared__ float smem[];
  float *sM = smem;                // [K][K+1]
  float *sS = sM + K * (K + 1);    // [K][32]
  const int ch = blockIdx.x / H, h = blockIdx.x % H;
  const int tid = threadIdx.x, j = tid & 31, rb = tid >> 5;
  const int col = blockIdx.y * 32 + j;
  const int64_t st0 = (int64_t)ch * H + h;

  float reg[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int r = rb + 8 * i;
    reg[i] = S0 ? S0[(st0 * K + r) * V + col] : 0.f;
  }
  for (int step = 0; step < S; ++step) {
    const int seg = reverse ? S - 1 - step : step;
    const int64_t u = ((int64_t)ch * S + seg) * H + h;
    __syncthreads();  // previous step done with sM / sS
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int r = rb + 8 * i;
      sS[r * 32 + j] = reg[i];
      S_in[(u * K + r) * V + col] = reg[i];
    }
    const float *Mu = M + u * K * K;
    if (reverse)  // sM = M^T
      for (int x = tid; x < K * K; x += 256) sM[(x % K) * (K + 1) + (x / K)] = Mu[x];
    else
      for (int x = tid; x < K * K; x += 256) sM[(x / K) * (K + 1) + (x % K)] = Mu[x];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int r = rb + 8 * i;
      float acc = St[(u * K + r) * V + col];
      for (int m = 0; m < K; ++m) acc = fmaf(sM[r * (K + 1) + m], sS[m * 32 + j], acc);
      reg[i] = acc;
    }
  }
  if (S_final) {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int r = rb + 8 * i;
      S_final[(st0 * K + r) * V + col] = reg[i];
    }
  }
}

template <int K>
cudaError_t scan_dispatch(const float *M, const float *St, const float *S0, int C, int S, int H,
                          int V, float *S_in, float *S_final, cudaStream_t st, bool reverse) {
  const size_t smem = sizeof(float) * (K * (K + 1) + K * 32);
  auto kern = prefix_scan_kernel<K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((int64_t)C * H), V / 32);
  kern<<<grid, 256, smem, st>>>(M, St, S0, S, H, V, S_in, S_final, reverse);
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
