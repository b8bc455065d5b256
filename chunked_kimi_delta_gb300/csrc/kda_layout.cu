// kda_layout.cu - state layout conversion at the boundary.
//
// "Hyper-Parallel Chunk KDA current implementation design", section 4.1
// (state_v_first): a caller may hand over and receive recurrent states with
// their last two dimensions as [V, K]; the library works K-first ([K, V])
// internally and converts at the boundary.  A state is a dense fp32 matrix,
// states follow one another.
//
// Section 4.2 of the same design lists the token layouts BSND [B, T, H, D],
// TND [T, H, D] and the head-major BNSD [B, H, T, D], NTD [H, T, D].  The
// kernels work token-major; head-major tensors are converted at the
// boundary by swapping the token and head axes, row by row (a row is the D
// elements of one (token, head)).  Heads narrower than the tensor-core
// kernels' 128 channels are widened into zero-padded copies and the outputs
// cut back (window copies).
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

// One unit = U bytes (16 when a row's bytes are a multiple of 16, else the
// element size); thread = unit of the destination.
template <typename Unit>
__global__ void __launch_bounds__(256)
swap_token_head_kernel(const Unit *__restrict__ src, Unit *__restrict__ dst, int64_t B, int H,
                       int64_t T, int units_per_row, bool to_token_major, int64_t total) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int u = (int)(i % units_per_row);
  const int64_t row = i / units_per_row;  // destination row
  int64_t b, t;
  int h;
  if (to_token_major) {  // destination [B][T][H]
    h = (int)(row % H);
    const int64_t bt = row / H;
    t = bt % T;
    b = bt / T;
    dst[i] = src[(((b * H + h) * T) + t) * units_per_row + u];
  } else {  // destination [B][H][T]
    t = row % T;
    const int64_t bh = row / T;
    h = (int)(bh % H);
    b = bh / H;
    dst[i] = src[(((b * T + t) * H) + h) * units_per_row + u];
  }
}

// Window copy between stacks of matrices of different shapes, in 16-byte
// units: dst[m][r][u] = src[m][r][u] where r < Rs and u < Us, else `fill`
// (m < n; dst is Rd x Ud units per matrix).  With count_ptr only matrices
// below (*count_ptr) * per_count are written.
__global__ void __launch_bounds__(256)
window_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int Rs, int Us, int Rd, int Ud,
              uint4 fill, const int32_t *__restrict__ count_ptr, int per_count, int64_t total) {
  const int64_t limit = count_ptr ? (int64_t)(*count_ptr) * per_count * Rd * Ud : total;
  const int64_t end = limit < total ? limit : total;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < end;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int u = (int)(i % Ud);
    const int64_t mr = i / Ud;
    const int r = (int)(mr % Rd);
    const int64_t m = mr / Rd;
    dst[i] = (r < Rs && u < Us) ? src[(m * Rs + r) * Us + u] : fill;
  }
}

}  // namespace

cudaError_t launch_window_copy(const void *src, void *dst, int64_t n, int rows_src, int row_bytes_src,
                               int rows_dst, int row_bytes_dst, uint32_t fill, const int32_t *count_ptr,
                               int per_count, cudaStream_t st) {
  if (row_bytes_src % 16 || row_bytes_dst % 16 || rows_src < 1 || rows_dst < 1) return cudaErrorInvalidValue;
  const int64_t total = n * rows_dst * (row_bytes_dst / 16);
  if (total == 0) return cudaSuccess;
  const int64_t want = (total + 255) / 256;
  const unsigned blocks = (unsigned)(want < 4096 ? want : 4096);
  window_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), rows_src,
                                        row_bytes_src / 16, rows_dst, row_bytes_dst / 16,
                                        make_uint4(fill, fill, fill, fill), count_ptr, per_count, total);
  return cudaGetLastError();
}

cudaError_t launch_swap_token_head(const void *src, void *dst, int64_t B, int H, int64_t T,
                                   int row_bytes, bool to_token_major, cudaStream_t st) {
  const int64_t rows = B * H * T;
  if (rows == 0) return cudaSuccess;
  if (row_bytes % 16 == 0) {
    const int upr = row_bytes / 16;
    const int64_t total = rows * upr;
    swap_token_head_kernel<uint4><<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
        static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), B, H, T, upr, to_token_major, total);
  } else {
    if (row_bytes % 4 != 0) return cudaErrorInvalidValue;
    const int upr = row_bytes / 4;
    const int64_t total = rows * upr;
    swap_token_head_kernel<uint32_t><<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
        static_cast<const uint32_t *>(src), static_cast<uint32_t *>(dst), B, H, T, upr, to_token_major,
        total);
  }
  return cudaGetLastError();
}

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
