// kda_state_copy.cu - gather / scatter of per-request recurrent states between
// a cache pool and packed rows.
//
// Contract (vllm-ascend KDA prefill state copy article, section "数值契约",
// numerical contract): a gather of an invalid index (negative, out of range)
// or of a row whose flag is false writes zeros; duplicate gather indices are
// legal; every packed row is written.  A scatter skips invalid indices,
// ignores flags, and converts the packed row to the cache dtype first.  Only
// the payload of a row is touched: the gap between the payload and the next
// row stays as it was.  Row addresses are 64-bit element offsets, so rows
// more than 4 GiB apart are reached with 32-bit indices.
//
// One CTA row-slice per (selected row, slice of the payload); 16-byte vector
// accesses whenever the payload, the row stride and both base pointers allow
// it, element accesses otherwise.  Same-dtype copies move raw bits (NaN
// payloads survive); fp32 -> bf16 rounds to nearest even.
#include <type_traits>

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;

template <typename Ts, typename Td>
__device__ __forceinline__ void copy8(const Ts *s, Td *d) {
  if constexpr (std::is_same<Ts, Td>::value) {
    constexpr int n16 = (int)(8 * sizeof(Ts) / 16);
#pragma unroll
    for (int i = 0; i < n16; ++i) reinterpret_cast<uint4 *>(d)[i] = reinterpret_cast<const uint4 *>(s)[i];
  } else if constexpr (std::is_same<Ts, float>::value) {  // fp32 -> bf16
    const float4 a = reinterpret_cast<const float4 *>(s)[0];
    const float4 b = reinterpret_cast<const float4 *>(s)[1];
    __nv_bfloat162 o[4] = {__floats2bfloat162_rn(a.x, a.y), __floats2bfloat162_rn(a.z, a.w),
                           __floats2bfloat162_rn(b.x, b.y), __floats2bfloat162_rn(b.z, b.w)};
    *reinterpret_cast<uint4 *>(d) = *reinterpret_cast<const uint4 *>(o);
  } else {  // bf16 -> fp32 (exact)
    const uint4 raw = *reinterpret_cast<const uint4 *>(s);
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&raw);
    float2 f0 = __bfloat1622float2(p[0]), f1 = __bfloat1622float2(p[1]);
    float2 f2 = __bfloat1622float2(p[2]), f3 = __bfloat1622float2(p[3]);
    reinterpret_cast<float4 *>(d)[0] = make_float4(f0.x, f0.y, f1.x, f1.y);
    reinterpret_cast<float4 *>(d)[1] = make_float4(f2.x, f2.y, f3.x, f3.y);
  }
}

template <typename Ts, typename Td>
__device__ __forceinline__ void copy1(const Ts *s, Td *d) {
  if constexpr (std::is_same<Ts, Td>::value) *d = *s;
  else *d = from_f32<Td>(to_f32<Ts>(*s));
}

template <typename Td>
__device__ __forceinline__ void zero8(Td *d) {
  constexpr int n16 = (int)(8 * sizeof(Td) / 16);
#pragma unroll
  for (int i = 0; i < n16; ++i) reinterpret_cast<uint4 *>(d)[i] = make_uint4(0, 0, 0, 0);
}

// gather: src = cache rows, dst = packed; scatter: src = packed, dst = cache rows.
template <bool GATHER, bool VEC, typename Tidx, typename Ts, typename Td>
__global__ void __launch_bounds__(kThreads)
state_copy_kernel(const Ts *__restrict__ src, Td *__restrict__ dst, const Tidx *__restrict__ idx,
                  const bool *__restrict__ flags, int64_t num_rows, int64_t row_stride,
                  int64_t payload) {
  const int64_t i = blockIdx.x;
  const int64_t row = (int64_t)idx[i];
  bool valid = row >= 0 && row < num_rows;
  if (GATHER && flags && !flags[i]) valid = false;
  if (!GATHER && !valid) return;
  const Ts *s = GATHER ? src + (valid ? row * row_stride : 0) : src + i * payload;
  Td *d = GATHER ? dst + i * payload : dst + row * row_stride;
  const int64_t stride = (int64_t)gridDim.y * kThreads;
  if (VEC) {
    const int64_t groups = payload / 8;
    for (int64_t gi = (int64_t)blockIdx.y * kThreads + threadIdx.x; gi < groups; gi += stride) {
      if (valid) copy8(s + 8 * gi, d + 8 * gi);
      else zero8(d + 8 * gi);
    }
  } else {
    for (int64_t e = (int64_t)blockIdx.y * kThreads + threadIdx.x; e < payload; e += stride) {
      if (valid) copy1(s + e, d + e);
      else d[e] = from_f32<Td>(0.f);
    }
  }
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <bool GATHER, typename Ts, typename Td>
cudaError_t launch_typed(const void *src, void *dst, const void *idx, kda_index_dtype it,
                         const bool *flags, int64_t num_rows, int64_t row_stride, int64_t payload,
                         int64_t n_sel, cudaStream_t st) {
  const bool vec = payload % 8 == 0 && row_stride % 8 == 0 && aligned16(src) && aligned16(dst);
  const int64_t work = vec ? payload / 8 : payload;
  int64_t slices = (work + kThreads - 1) / kThreads;
  if (slices > 1024) slices = 1024;
  if (slices < 1) slices = 1;
  const dim3 grid((unsigned)n_sel, (unsigned)slices);
  const Ts *s = static_cast<const Ts *>(src);
  Td *d = static_cast<Td *>(dst);
#define KDA_COPY(V_, TI_)                                                                   \
  state_copy_kernel<GATHER, V_, TI_, Ts, Td><<<grid, kThreads, 0, st>>>(                    \
      s, d, static_cast<const TI_ *>(idx), flags, num_rows, row_stride, payload)
  if (it == KDA_I32) {
    if (vec) KDA_COPY(true, int32_t); else KDA_COPY(false, int32_t);
  } else {
    if (vec) KDA_COPY(true, int64_t); else KDA_COPY(false, int64_t);
  }
#undef KDA_COPY
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state_gather(const void *cache, kda_dtype dt, int64_t num_rows,
                                int64_t row_stride, int64_t payload, const void *idx,
                                kda_index_dtype it, const bool *flags, int64_t n_sel,
                                void *packed, cudaStream_t st) {
  if (dt == KDA_F32)
    return launch_typed<true, float, float>(cache, packed, idx, it, flags, num_rows, row_stride,
                                            payload, n_sel, st);
  return launch_typed<true, __nv_bfloat16, __nv_bfloat16>(cache, packed, idx, it, flags, num_rows,
                                                          row_stride, payload, n_sel, st);
}

cudaError_t launch_state_scatter(void *cache, kda_dtype dt, int64_t num_rows, int64_t row_stride,
                                 int64_t payload, const void *idx, kda_index_dtype it,
                                 const void *packed, kda_dtype pdt, int64_t n_sel,
                                 cudaStream_t st) {
#define KDA_SCAT(TS_, TD_)                                                                 \
  return launch_typed<false, TS_, TD_>(packed, cache, idx, it, nullptr, num_rows, row_stride, \
                                       payload, n_sel, st)
  if (dt == KDA_F32 && pdt == KDA_F32) KDA_SCAT(float, float);
  if (dt == KDA_F32 && pdt == KDA_BF16) KDA_SCAT(__nv_bfloat16, float);
  if (dt == KDA_BF16 && pdt == KDA_F32) KDA_SCAT(float, __nv_bfloat16);
  KDA_SCAT(__nv_bfloat16, __nv_bfloat16);
#undef KDA_SCAT
}

}  // namespace kda
