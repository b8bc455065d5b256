// kda_tc_chain.cu - inter-chunk stage of the tensor-core KDA forward.
//
// One CTA per (sequence, head) walks the chunks in order ("KDA Chunk Backward
// - TPU/Pallas Kernel Design" sections 1 and 1.2; "Hyper-Parallel Chunk KDA
// current implementation design" section 5.1, FwdH and FwdFinalize):
//   [qg; w] h        -> P           (tcgen05, M=128, N=128, K=128)
//   v_new = u - w h                 (CUDA cores, fp32, stored bf16 for the MMAs)
//   P[0:64] += Aqk v_new            (tcgen05; o = qg h + Aqk v_new)
//   kg^T v_new       -> U           (tcgen05, M=128, N=128, K=64)
//   h' = e^{G_C} h + U              (fp32, registers)
// The fp32 state lives in registers (thread = one key channel x 64 value
// channels); a bf16 copy in shared memory is the MMA operand.  Packages are
// double-buffered with bulk copies issued two chunks ahead.
//
// Summary mode ("Hyper-Parallel ..." section 5.1, PreProcessFwd; "KDA Context
// Parallelism (KCP)"): the same chain on the augmented state [S~ | M] with
// X_0 = [0 | I] and values [u | 0]; blockIdx.y = 0 carries the S~ columns,
// blockIdx.y = 1 the M columns; nothing else is written.
#include <cuda_bf16.h>

#include "kda_tc.cuh"

namespace kda {
namespace tcp {
namespace {

constexpr int NT = 256;
constexpr uint32_t S_BUF0 = 0;
constexpr uint32_t S_BAR = PK_BYTES;         // 3 mbarriers in the gap before buffer 1
constexpr uint32_t S_BUF1 = 91136;           // 1024-aligned
constexpr uint32_t S_HB = 182272;            // h bf16, MN-major (K = 128 channels)
constexpr uint32_t S_VN = 215040;            // v_new bf16, MN-major (K = 64 tokens)
constexpr uint32_t SMEM_BYTES = 231424 + 1024;
constexpr uint32_t BUF_STRIDE = S_BUF1 - S_BUF0;

template <int MODE>
__global__ void __launch_bounds__(NT, 1) tc_chain_kernel(ChainArgs a, SeqInfo s, int H) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + S_BAR);  // [2]
  uint64_t *bar_mma = full + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(full + 3);
  volatile uint32_t *abort_flag = tslot + 1;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q4 = warp & 3, hf = warp >> 2;
  const int kr = 32 * q4 + lane;  // key channel (state row) owned by this thread
  const int n = blockIdx.x / H, h = blockIdx.x % H;
  const int part = blockIdx.y;
  int64_t t0, t1;
  seq_range(s, n, t0, t1);
  const int64_t c0 = seq_first_chunk(s, n);
  const int64_t nch = (t1 - t0 + BT - 1) / BT;
  const int64_t unit = (int64_t)n * H + h;

  if (warp == 0) {
    tc::tmem_alloc(tslot, 256);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(full, 1);
    tc::mbar_init(full + 1, 1);
    tc::mbar_init(bar_mma, 1);
    tc::mbar_fence_init();
    *abort_flag = 0;
  }

  // initial state -> registers and the bf16 operand
  float hr[64];
  if (MODE == CHAIN_FWD) {
    if (a.initial_state) {
      const float4 *src = reinterpret_cast<const float4 *>(a.initial_state + (unit * K + kr) * V + 64 * hf);
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const float4 v = src[x];
        hr[4 * x] = v.x; hr[4 * x + 1] = v.y; hr[4 * x + 2] = v.z; hr[4 * x + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int x = 0; x < 64; ++x) hr[x] = 0.f;
    }
  } else {
#pragma unroll
    for (int x = 0; x < 64; ++x) hr[x] = (part == 1 && kr == 64 * hf + x) ? 1.f : 0.f;
  }
  auto store_hb = [&]() {
#pragma unroll
    for (int x = 0; x < 64; x += 8) {
      const uint4 v = make_uint4(pack_bf16(hr[x], hr[x + 1]), pack_bf16(hr[x + 2], hr[x + 3]),
                                 pack_bf16(hr[x + 4], hr[x + 5]), pack_bf16(hr[x + 6], hr[x + 7]));
      *reinterpret_cast<uint4 *>(sm + S_HB + mnmaj_off(128, kr, 64 * hf + x)) = v;
    }
  };
  store_hb();
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tP = tmem, tU = tmem + 128;

  // thread 0 keeps count of the copies and MMAs it started, for the drain
  int64_t loads_issued = 0, loads_done = 0;
  bool mma_pending = false;
  if (tid == 0) {
    for (int64_t c = 0; c < 2 && c < nch; ++c) {
      ++loads_issued;
      tc::mbar_arrive_expect_tx(full + c, PK_BYTES);
      bulk_load(sm + S_BUF0 + c * BUF_STRIDE, a.pkg + (size_t)((c0 + c) * H + h) * PK_BYTES, PK_BYTES,
                full + c);
    }
  }

  uint32_t mph = 0;
  for (int64_t c = 0; c < nch; ++c) {
    const int b = (int)(c & 1);
    uint8_t *buf = sm + S_BUF0 + b * BUF_STRIDE;
    const int64_t tc0 = t0 + c * BT;
    const int len = (int)((t1 - tc0) < BT ? (t1 - tc0) : BT);
    bool ok = wait_or_flag(full + b, (uint32_t)((c >> 1) & 1), a.err);
    if (!ok) *abort_flag = 1;
    else loads_done = c + 1;
    if (MODE == CHAIN_FWD && a.h_out) {
      float4 *dst = reinterpret_cast<float4 *>(a.h_out + (((c0 + c) * H + h) * K + kr) * V + 64 * hf);
#pragma unroll
      for (int x = 0; x < 16; ++x) dst[x] = make_float4(hr[4 * x], hr[4 * x + 1], hr[4 * x + 2], hr[4 * x + 3]);
    }
    __syncthreads();
    if (*abort_flag) break;

    // ---- [qg; w] h -> P
    if (tid == 0) {
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(128, 128, false, true);
      const uint32_t a0 = tc::smem_u32(buf + PK_WQ), b0 = tc::smem_u32(sm + S_HB);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc::mma_bf16(tP, tc::smem_desc_sw128(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                     tc::smem_desc_sw128(b0 + kk * 2048, 16384, 1024), idesc, kk > 0);
      tc::mma_commit(bar_mma);
      mma_pending = true;
    }
    __syncwarp();
    ok = wait_or_flag(bar_mma, mph, a.err);
    if (ok) { mma_pending = false; mph ^= 1; }
    else *abort_flag = 1;
    tc::tc_fence_after();
    __syncthreads();
    if (*abort_flag) break;

    // ---- v_new = u - w h  (P rows 64..127 live in TMEM lanes 64..127)
    if (q4 >= 2) {
      const int r = 32 * (q4 - 2) + lane;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float d[16];
        __syncwarp();
        tc::tmem_ld16(tP + ((uint32_t)(32 * q4) << 16) + 64 * hf + 16 * cc, d);
        tc::tmem_ld_wait();
        const int col = 64 * hf + 16 * cc;
        float vn[16];
#pragma unroll
        for (int x = 0; x < 16; x += 4) {
          float4 u4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (!(MODE == CHAIN_SUMMARY && part == 1))
            u4 = *reinterpret_cast<const float4 *>(buf + PK_U + u_offset(r, col + x));
          vn[x] = u4.x - d[x];
          vn[x + 1] = u4.y - d[x + 1];
          vn[x + 2] = u4.z - d[x + 2];
          vn[x + 3] = u4.w - d[x + 3];
        }
        *reinterpret_cast<uint4 *>(sm + S_VN + mnmaj_off(64, r, col)) =
            make_uint4(pack_bf16(vn[0], vn[1]), pack_bf16(vn[2], vn[3]), pack_bf16(vn[4], vn[5]),
                       pack_bf16(vn[6], vn[7]));
        *reinterpret_cast<uint4 *>(sm + S_VN + mnmaj_off(64, r, col + 8)) =
            make_uint4(pack_bf16(vn[8], vn[9]), pack_bf16(vn[10], vn[11]), pack_bf16(vn[12], vn[13]),
                       pack_bf16(vn[14], vn[15]));
        if (MODE == CHAIN_FWD && a.v_new_out && r < len) {
          float4 *dst = reinterpret_cast<float4 *>(a.v_new_out + ((tc0 + r) * H + h) * V + col);
#pragma unroll
          for (int x = 0; x < 4; ++x) dst[x] = make_float4(vn[4 * x], vn[4 * x + 1], vn[4 * x + 2], vn[4 * x + 3]);
        }
      }
    }
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (*abort_flag) break;

    // ---- P[0:64] += Aqk v_new (rows 64..127 of the A operand are unused),
    //      kg^T v_new -> U
    if (tid == 0) {
      tc::tc_fence_after();
      const uint32_t vn0 = tc::smem_u32(sm + S_VN);
      if (MODE == CHAIN_FWD) {
        const uint32_t idb = tc::idesc_bf16_f32(128, 128, false, true);
        const uint32_t q0 = tc::smem_u32(buf + PK_AQK);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tP, tc::smem_desc_sw128(q0 + kk * 32, 16, 1024),
                       tc::smem_desc_sw128(vn0 + kk * 2048, 8192, 1024), idb, true);
      }
      const uint32_t idc = tc::idesc_bf16_f32(128, 128, true, true);
      const uint32_t g0 = tc::smem_u32(buf + PK_KG);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_bf16(tU, tc::smem_desc_sw128(g0 + kk * 2048, 8192, 1024),
                     tc::smem_desc_sw128(vn0 + kk * 2048, 8192, 1024), idc, kk > 0);
      tc::mma_commit(bar_mma);
      mma_pending = true;
    }
    __syncwarp();
    ok = wait_or_flag(bar_mma, mph, a.err);
    if (ok) { mma_pending = false; mph ^= 1; }
    else *abort_flag = 1;
    tc::tc_fence_after();
    __syncthreads();
    if (*abort_flag) break;

    // ---- h' = e^{G_C} h + kg^T v_new
    {
      const float gcv = reinterpret_cast<const float *>(buf + PK_GC)[kr];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float d[16];
        tc::tmem_ld16(tU + ((uint32_t)(32 * q4) << 16) + 64 * hf + 16 * cc, d);
        tc::tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 16; ++x) hr[16 * cc + x] = fmaf(gcv, hr[16 * cc + x], d[x]);
      }
      store_hb();
    }
    // ---- o = qg h + Aqk v_new (P rows 0..63)
    if (MODE == CHAIN_FWD && q4 < 2) {
      const int r = 32 * q4 + lane;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float d[16];
        __syncwarp();
        tc::tmem_ld16(tP + ((uint32_t)(32 * q4) << 16) + 64 * hf + 16 * cc, d);
        tc::tmem_ld_wait();
        if (r < len) {
          uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) +
                                                 ((tc0 + r) * H + h) * V + 64 * hf + 16 * cc);
          dst[0] = make_uint4(pack_bf16(d[0], d[1]), pack_bf16(d[2], d[3]), pack_bf16(d[4], d[5]),
                              pack_bf16(d[6], d[7]));
          dst[1] = make_uint4(pack_bf16(d[8], d[9]), pack_bf16(d[10], d[11]),
                              pack_bf16(d[12], d[13]), pack_bf16(d[14], d[15]));
        }
      }
    }
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (*abort_flag) break;
    if (tid == 0 && c + 2 < nch) {
      ++loads_issued;
      tc::mbar_arrive_expect_tx(full + b, PK_BYTES);
      bulk_load(buf, a.pkg + (size_t)((c0 + c + 2) * H + h) * PK_BYTES, PK_BYTES, full + b);
    }
  }

  if (*abort_flag == 0) {
    if (MODE == CHAIN_FWD) {
      if (a.final_state) {
        float4 *dst = reinterpret_cast<float4 *>(a.final_state + (unit * K + kr) * V + 64 * hf);
#pragma unroll
        for (int x = 0; x < 16; ++x) dst[x] = make_float4(hr[4 * x], hr[4 * x + 1], hr[4 * x + 2], hr[4 * x + 3]);
      }
    } else {
      float *base = part == 0 ? a.S_tilde + (unit * K + kr) * V : a.M + (unit * K + kr) * K;
      float4 *dst = reinterpret_cast<float4 *>(base + 64 * hf);
#pragma unroll
      for (int x = 0; x < 16; ++x) dst[x] = make_float4(hr[4 * x], hr[4 * x + 1], hr[4 * x + 2], hr[4 * x + 3]);
    }
  } else if (tid == 0) {
    // a wait gave up: let the copies and the MMA this CTA started finish
    // (each wait bounded) before its shared and tensor memory are released
    if (mma_pending) drain_wait(bar_mma, mph);
    for (int64_t c = loads_done; c < loads_issued; ++c) drain_wait(full + (c & 1), (uint32_t)((c >> 1) & 1));
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

}  // namespace

cudaError_t launch_tc_chain(ChainMode mode, const ChainArgs &a, const SeqInfo &s, int H,
                            cudaStream_t st) {
  const dim3 grid((unsigned)((int64_t)s.N * H), mode == CHAIN_SUMMARY ? 2 : 1);
  if (grid.x == 0) return cudaSuccess;
  if (mode == CHAIN_FWD) {
    cudaError_t e = cudaFuncSetAttribute(tc_chain_kernel<CHAIN_FWD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    tc_chain_kernel<CHAIN_FWD><<<grid, NT, SMEM_BYTES, st>>>(a, s, H);
  } else {
    cudaError_t e = cudaFuncSetAttribute(tc_chain_kernel<CHAIN_SUMMARY>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    tc_chain_kernel<CHAIN_SUMMARY><<<grid, NT, SMEM_BYTES, st>>>(a, s, H);
  }
  return cudaGetLastError();
}

}  // namespace tcp
}  // namespace kda
