// kda_tc_host.cu - host side of the tensor-core path: TMA descriptors for the
// inputs, encoded through the driver entry point (no link-time libcuda).
#include <cudaTypedefs.h>
#include <string.h>

#include "kda_tc.cuh"

namespace kda {
namespace tcp {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Token-major [T_tot, H, D] tensor seen as 3-D (D, H, T_tot); a box covers
// `box0` channels of one head over 64 tokens.
bool encode3(CUtensorMap *m, CUtensorMapDataType dt, uint32_t esize, const void *ptr, int D, int H,
             int64_t T, uint32_t box0, CUtensorMapSwizzle sw) {
  auto fn = encoder();
  if (!fn) return false;
  memset(m, 0, sizeof(*m));
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)H * D * esize};
  cuuint32_t box[3] = {box0, 1, (cuuint32_t)BT};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_input_maps(const void *q, const void *k, const void *v, const float *x, int64_t T_tot,
                     int dk, int dv, int H, int Hk, TcMaps &maps) {
  if (T_tot <= 0 || (dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return false;
  return encode3(&maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, dk, Hk, T_tot, (uint32_t)dk,
                 CU_TENSOR_MAP_SWIZZLE_NONE) &&
         encode3(&maps.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, dk, Hk, T_tot, (uint32_t)dk,
                 CU_TENSOR_MAP_SWIZZLE_NONE) &&
         encode3(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, v, dv, H, T_tot, 64,
                 CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode3(&maps.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, x, dk, H, T_tot, (uint32_t)dk,
                 CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool make_out_map(const void *o, int64_t T_tot, int H, int dv, CUtensorMap &map) {
  if (T_tot <= 0 || (dv != 64 && dv != 128)) return false;
  return encode3(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o, dv, H, T_tot, 64, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_value_map(const void *x, int64_t T_tot, int H, CUtensorMap &map) {
  if (T_tot <= 0) return false;
  return encode3(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, V, H, T_tot, 64,
                 CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace tcp
}  // namespace kda
