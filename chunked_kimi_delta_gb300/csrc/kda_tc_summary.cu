// kda_tc_summary.cu - segment affine summary on the tensor cores.
//
// For each (segment, head) the chunks of the segment are walked in order on
// the augmented state X = [S~ | M] (128 x 256), started from [0 | I]
// ("Hyper-Parallel Chunk KDA current implementation design" section 5.1,
// PreProcessFwd: H_out = M H_in + E; "KDA Context Parallelism (KCP)", "Les
// notations").  Per chunk, with the prep kernel's package:
//   P   = [w; w] X                     (tcgen05, M=128, N=256, K=128)
//   V'  = [u - P_S~ | -P_M]            (the values of the two parts; bf16)
//   U   = kg^T V'                      (tcgen05, M=128, N=256, K=64)
//   X  <- e^{G_C} X + U                (fp32, registers)
// Both parts share one CTA and one copy of each package; only the w rows,
// u, kg and e^{G_C} of a package are loaded (qg and A_qk serve the output,
// which a summary does not produce).  The w rows are stacked twice, so that
// the product fills all 128 TMEM lanes (an M=64 product would leave half of
// every warp's lanes idle in the readout) at no extra tensor time: the
// warps of lane quarters 0, 1 and 2, 3 read the two copies and split the
// columns.
#include <cuda_bf16.h>

#include "kda_tc.cuh"

namespace kda {
namespace tcp {
namespace {

constexpr int NT = 512;  // 16 warps: (TMEM lane quarter) x (64-column quarter of X)

// One package buffer (bytes): [w; w] (K-major, two 64-channel panels of 128
// rows), u, kg (as in the package) and e^{G_C}.
constexpr uint32_t B_W = 0;
constexpr uint32_t B_U = 32768;
constexpr uint32_t B_KG = 49152;
constexpr uint32_t B_GC = 65536;
constexpr uint32_t B_BYTES = 66048;
constexpr uint32_t BUF_STRIDE = 66560;           // 1024-aligned
constexpr uint32_t S_BAR = B_BYTES;              // full[2], bar_ma, bar_mc, tslot, abort: in the
                                                 // alignment gap after buffer 0
constexpr uint32_t S_XB = 2 * BUF_STRIDE;        // X bf16, MN-major (K = 128 channels, N = 256)
constexpr uint32_t S_VN = S_XB + 65536;          // V' bf16, MN-major (K = 64 tokens, N = 256)
constexpr uint32_t SMEM_BYTES = S_VN + 32768 + 1024;
static_assert(S_BAR + 64 <= BUF_STRIDE && SMEM_BYTES <= 232448, "shared memory layout");
constexpr uint32_t TMEM_COLS = 512;              // P (256, M=64 layout) and U (256)

// NARROW: heads of 64 channels (dk or dv), whose M and S~ are the windows
// of the 128-wide ones (the 128-wide instantiation keeps constant addressing,
// and so its registers).
template <bool NARROW>
__global__ void __launch_bounds__(NT, 1) tc_summary_kernel(const char *__restrict__ pkg, float *S_tilde,
                                                           float *Mout, SeqInfo s, int H, int dk_arg,
                                                           int dv_arg, uint32_t *err) {
  const int dk = NARROW ? dk_arg : 128, dv = NARROW ? dv_arg : 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + S_BAR);  // [2]
  uint64_t *bar_ma = full + 2;
  uint64_t *bar_mc = full + 3;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(full + 4);
  volatile uint32_t *abort_flag = tslot + 1;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q4 = warp & 3, cq = warp >> 2;
  const int kr = 32 * q4 + lane;  // row of X (key channel) owned by this thread
  const int n = blockIdx.x / H, h = blockIdx.x % H;
  int64_t t0, t1;
  seq_range(s, n, t0, t1);
  const int64_t c0 = seq_first_chunk(s, n);
  const int64_t nch = (t1 - t0 + BT - 1) / BT;
  const int64_t unit = (int64_t)n * H + h;

  if (warp == 0) {
    tc::tmem_alloc(tslot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(full, 1);
    tc::mbar_init(full + 1, 1);
    tc::mbar_init(bar_ma, 1);
    tc::mbar_init(bar_mc, 1);
    tc::mbar_fence_init();
    *abort_flag = 0;
  }

  // X = [0 | I]: columns 64 cq .. 64 cq + 63 of row kr
  float hr[64];
#pragma unroll
  for (int x = 0; x < 64; ++x) hr[x] = (cq >= 2 && kr == 64 * (cq - 2) + x) ? 1.f : 0.f;
  auto store_xb = [&]() {
#pragma unroll
    for (int x = 0; x < 64; x += 8) {
      const uint4 v = make_uint4(pack_bf16(hr[x], hr[x + 1]), pack_bf16(hr[x + 2], hr[x + 3]),
                                 pack_bf16(hr[x + 4], hr[x + 5]), pack_bf16(hr[x + 6], hr[x + 7]));
      *reinterpret_cast<uint4 *>(sm + S_XB + mnmaj_off(128, kr, 64 * cq + x)) = v;
    }
  };
  store_xb();
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tP = tmem, tU = tmem + 256;

  // thread 0 starts the copies and the MMAs and keeps count, for the drain
  int64_t loads_issued = 0, loads_done = 0;
  bool ma_pending = false, mc_pending = false;
  uint32_t ma_par = 0, mc_par = 0;
  auto load = [&](int64_t cc) {
    const int bb = (int)(cc & 1);
    uint8_t *dst = sm + bb * BUF_STRIDE;
    const char *src = pkg + (size_t)((c0 + cc) * H + h) * PK_BYTES;
    tc::mbar_arrive_expect_tx(full + bb, B_BYTES);
    // the package's w rows (rows 64..127 of each [qg; w] panel; their swizzle
    // phase repeats every 8 rows) into rows 0..63 and 64..127 of each panel
    for (int pn = 0; pn < 2; ++pn)
      for (int cp = 0; cp < 2; ++cp)
        bulk_load(dst + B_W + pn * 16384 + cp * 8192, src + PK_WQ + pn * 16384 + 8192, 8192, full + bb);
    bulk_load(dst + B_U, src + PK_U, 16384, full + bb);
    bulk_load(dst + B_KG, src + PK_KG, 16384, full + bb);
    bulk_load(dst + B_GC, src + PK_GC, 512, full + bb);
    ++loads_issued;
  };
  if (tid == 0)
    for (int64_t c = 0; c < 2 && c < nch; ++c) load(c);

  for (int64_t c = 0; c < nch; ++c) {
    const int b = (int)(c & 1);
    uint8_t *buf = sm + b * BUF_STRIDE;
    bool ok = wait_or_flag(full + b, (uint32_t)((c >> 1) & 1), err);
    if (!ok) *abort_flag = 1;
    else if (tid == 0) loads_done = c + 1;
    __syncthreads();  // X (bf16) of this chunk and its package are in place
    if (*abort_flag) break;

    // ---- P = [w; w] X; the buffer of chunk c - 1 takes chunk c + 1
    if (tid == 0) {
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(128, 256, false, true);
      const uint32_t a0 = tc::smem_u32(buf + B_W), b0 = tc::smem_u32(sm + S_XB);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc::mma_bf16(tP, tc::smem_desc_sw128(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                     tc::smem_desc_sw128(b0 + kk * 2048, 16384, 1024), idesc, kk > 0);
      tc::mma_commit(bar_ma);
      ma_pending = true;
      ma_par = (uint32_t)(c & 1);
      if (c >= 1 && c + 1 < nch) load(c + 1);
    }
    __syncwarp();
    ok = __all_sync(0xffffffffu, wait_or_flag(bar_ma, (uint32_t)(c & 1), err));
    if (tid == 0 && ok) ma_pending = false;
    if (!ok) *abort_flag = 1;
    tc::tc_fence_after();

    // ---- V' = [u - P | -P]: row r of P in TMEM lanes r and 64 + r; the
    //      warps of lane quarters 0, 1 take the first 32 columns of their
    //      64-column quarter, those of quarters 2, 3 the last 32
    if (ok) {
      const int r = 32 * (q4 & 1) + lane;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float d[16];
        const int col = 64 * cq + 32 * (q4 >> 1) + 16 * cc;  // column of X
        __syncwarp();
        tc::tmem_ld16(tP + ((uint32_t)(32 * q4) << 16) + col, d);
        tc::tmem_ld_wait();
        {
          float vn[16];
          if (cq >= 2) {
#pragma unroll
            for (int x = 0; x < 16; ++x) vn[x] = -d[x];
          } else {
            const uint4 ua = *reinterpret_cast<const uint4 *>(buf + B_U + u_offset(r, col));
            const uint4 ub = *reinterpret_cast<const uint4 *>(buf + B_U + u_offset(r, col + 8));
            const uint32_t uw[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const float2 u2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&uw[x]));
              vn[2 * x] = u2.x - d[2 * x];
              vn[2 * x + 1] = u2.y - d[2 * x + 1];
            }
          }
          *reinterpret_cast<uint4 *>(sm + S_VN + mnmaj_off(64, r, col)) =
              make_uint4(pack_bf16(vn[0], vn[1]), pack_bf16(vn[2], vn[3]), pack_bf16(vn[4], vn[5]),
                         pack_bf16(vn[6], vn[7]));
          *reinterpret_cast<uint4 *>(sm + S_VN + mnmaj_off(64, r, col + 8)) =
              make_uint4(pack_bf16(vn[8], vn[9]), pack_bf16(vn[10], vn[11]), pack_bf16(vn[12], vn[13]),
                         pack_bf16(vn[14], vn[15]));
        }
      }
    }
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (*abort_flag) break;

    // ---- U = kg^T V'
    if (tid == 0) {
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(128, 256, true, true);
      const uint32_t g0 = tc::smem_u32(buf + B_KG), v0 = tc::smem_u32(sm + S_VN);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_bf16(tU, tc::smem_desc_sw128(g0 + kk * 2048, 8192, 1024),
                     tc::smem_desc_sw128(v0 + kk * 2048, 8192, 1024), idesc, kk > 0);
      tc::mma_commit(bar_mc);
      mc_pending = true;
      mc_par = (uint32_t)(c & 1);
    }
    __syncwarp();
    ok = __all_sync(0xffffffffu, wait_or_flag(bar_mc, (uint32_t)(c & 1), err));
    if (tid == 0 && ok) mc_pending = false;
    if (!ok) {
      *abort_flag = 1;
    } else {
      tc::tc_fence_after();
      // ---- X <- e^{G_C} X + U
      const float gcv = reinterpret_cast<const float *>(buf + B_GC)[kr];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float d[16];
        tc::tmem_ld16(tU + ((uint32_t)(32 * q4) << 16) + 64 * cq + 16 * cc, d);
        tc::tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 16; ++x) hr[16 * cc + x] = fmaf(gcv, hr[16 * cc + x], d[x]);
      }
      store_xb();
    }
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();
  }
  __syncthreads();

  // the caller's windows: S~ rows < dk, columns < dv; M rows and columns < dk
  // (narrow heads: the padded channels' part of M is the identity, of S~ zero)
  const int lim = cq < 2 ? dv : dk;  // columns of this thread's part
  if (*abort_flag == 0 && kr < dk && 64 * (cq & 1) < lim) {
    float *base = (cq < 2 ? S_tilde : Mout) + (unit * dk + kr) * lim + 64 * (cq & 1);
    float4 *dst = reinterpret_cast<float4 *>(base);
#pragma unroll
    for (int x = 0; x < 16; ++x) dst[x] = make_float4(hr[4 * x], hr[4 * x + 1], hr[4 * x + 2], hr[4 * x + 3]);
  }
  if (*abort_flag != 0 && tid == 0) {
    // a wait gave up: let the MMAs and copies this CTA started finish (each
    // wait bounded) before its tensor and shared memory are released
    if (ma_pending) drain_wait(bar_ma, ma_par);
    if (mc_pending) drain_wait(bar_mc, mc_par);
    for (int64_t c = loads_done; c < loads_issued; ++c) drain_wait(full + (c & 1), (uint32_t)((c >> 1) & 1));
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_tc_summary(const char *pkg, float *S_tilde, float *M, const SeqInfo &s, int H, int dk,
                              int dv, uint32_t *err, cudaStream_t st) {
  const int64_t units = (int64_t)s.N * H;
  if (units == 0) return cudaSuccess;
  auto kern = (dk == 128 && dv == 128) ? tc_summary_kernel<false> : tc_summary_kernel<true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)units, NT, SMEM_BYTES, st>>>(pkg, S_tilde, M, s, H, dk, dv, err);
  return cudaGetLastError();
}

}  // namespace tcp
}  // namespace kda
