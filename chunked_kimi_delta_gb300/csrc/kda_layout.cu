// kda_layout.cu - state layout conversion at the boundary.
//
// "Hyper-Parallel Chunk KDA current implementation design", section 4.1
// (state_v_first): a caller may hand over and receive recurrent states with
// their last two dimensions as [V, K]; the library works K-first ([K, V])
// internally and converts at the boundary.  A state is a dense fp32 matrix,
// states follow one another.
#include "kda_internal.cuh"

namespace kda {

namespace {

// dst[m][c][r] = src[m][r][c] for every matrix m of R x C; 32 x 32 tiles
// through shared memory, both sides coalesced.  Matrix ids start at m_base;
// when count_ptr is given only ids below (*count_ptr) * per_count are
// converted (the others are left untouched).
__global__ void __launch_bounds__(256)
transpose_kernel(const float *__restrict__ src, float *__restrict__ dst, int R, int C,
                 int64_t m_base, const int32_t *__restrict__ count_ptr, int per_count) {
  __shared__ float tile[32][33];
  const int64_t m = m_base + blockIdx.z;
  if (count_ptr && m >= (int64_t)(*count_ptr) * per_count) return;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  const float *s = src + m * R * C;
  float *d = dst + m * R * C;
  for (int y = ty; y < 32; y += 8) {
    const int r = r0 + y, c = c0 + tx;
    if (r < R && c < C) tile[y][tx] = s[(int64_t)r * C + c];
  }
  __syncthreads();
  for (int y = ty; y < 32; y += 8) {
    const int c = c0 + y, r = r0 + tx;
    if (r < R && c < C) d[(int64_t)c * R + r] = tile[tx][y];
  }
}

}  // namespace

cudaError_t launch_transpose_states(const float *src, float *dst, int64_t n, int R, int C,
                                    const int32_t *count_ptr, int per_count, cudaStream_t st) {
  for (int64_t m0 = 0; m0 < n; m0 += 65535) {  // grid z is at most 65535
    const int64_t nz = (n - m0) < 65535 ? (n - m0) : 65535;
    dim3 grid((C + 31) / 32, (R + 31) / 32, (unsigned)nz);
    transpose_kernel<<<grid, 256, 0, st>>>(src, dst, R, C, m0, count_ptr, per_count);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kda
