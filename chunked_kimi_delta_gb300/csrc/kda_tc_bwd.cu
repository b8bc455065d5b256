// kda_tc_bwd.cu - reverse chain of the state gradient on the tensor cores
// (bf16 inputs, d_k = d_v = 128).
//
// "KDA Chunk Backward - TPU/Pallas Kernel Design" section 2.3 (the dhu part
// of the fused backward: the state gradient dh runs through the chunks in
// reverse, collecting the output path, the delta-update path and the chunk
// decay).  One CTA per (sequence, head) walks the chunks backwards with the
// gradient dh' of the state leaving the chunk:
//   kg dh' + Aqk^T dO          -> dv_new   (tcgen05, M=64,  N=128, K=128+64)
//   qg^T dO - w^T dv_new       -> D        (tcgen05, M=128, N=128, K=64+64)
//   dh = e^{G_C} . dh' + D                 (fp32, registers)
// The operands are the forward's per-chunk packages, read in place: the
// K-major [qg; w] tile is the MN-major A operand of [qg; w]^T, the MN-major
// kg tile is the K-major A operand of kg, the K-major Aqk tile the MN-major
// A operand of Aqk^T (same bytes, the other major).  dO comes in by TMA in
// the layout of the forward's v tiles.  Outputs: dh' of every chunk and
// dv_new (fp32, for the per-chunk backward kernels) and the initial-state
// gradient.  Without d_out (a zero output gradient) the dO terms and copies
// are left out.
#include <cuda_bf16.h>
#include <string.h>

#include "kda_tc.cuh"

namespace kda {
namespace tcp {
namespace {

constexpr int NT = 256;
// per buffer: WQ (32 KB), KG + AQK + GC (25,088 B, as in the package), dO
// (two 8 KB SW128 panels of 64 tokens x 64 value channels)
constexpr uint32_t B_WQ = 0;
constexpr uint32_t B_KG = 32768;
constexpr uint32_t B_AQK = B_KG + (PK_AQK - PK_KG);
constexpr uint32_t B_GC = B_KG + (PK_GC - PK_KG);
constexpr uint32_t B_DO = 58368;             // 1024-aligned
constexpr uint32_t BUF_STRIDE = 74752;
constexpr uint32_t S_HB = 2 * BUF_STRIDE;    // dh' bf16, MN-major (K = 128 channels)
constexpr uint32_t S_DV = S_HB + 32768;      // -dv_new bf16, MN-major (K = 64 tokens)
constexpr uint32_t S_BAR = S_DV + 16384;
constexpr uint32_t SMEM_BYTES = S_BAR + 128 + 1024;
constexpr uint32_t TMEM_COLS = 256;          // D1 (dv_new) and D2
constexpr uint32_t LOAD_BYTES = 32768 + (PK_BYTES - PK_KG) + 16384;
static_assert(B_GC + 512 <= B_DO && B_DO + 16384 <= BUF_STRIDE, "buffer layout");

__global__ void __launch_bounds__(NT, 1)
tc_bwd_dh_kernel(const __grid_constant__ CUtensorMap map_do, BwdChainArgs a, SeqInfo s, int H) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + S_BAR);  // [2]
  uint64_t *bar_d1 = full + 2;     // kg dh' + Aqk^T dO
  uint64_t *bar_d2 = full + 3;     // everything of the chunk
  uint64_t *dv_ready = full + 4;   // -dv_new in shared memory (8 warp arrivals)
  uint32_t *tslot = reinterpret_cast<uint32_t *>(full + 5);
  volatile uint32_t *abort_flag = tslot + 1;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q4 = warp & 3, hf = warp >> 2;
  const int kr = 32 * q4 + lane;  // key channel (state row) of this thread
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
  const bool has_do = a.d_out != nullptr;
  if (tid == 0) {
    tc::mbar_init(full, 1);
    tc::mbar_init(full + 1, 1);
    tc::mbar_init(bar_d1, 1);
    tc::mbar_init(bar_d2, 1);
    tc::mbar_init(dv_ready, 8);
    tc::mbar_fence_init();
    *abort_flag = 0;
    if (has_do) tc::tma_prefetch_desc(&map_do);
  }

  // the gradient of the state leaving the last chunk -> registers and bf16
  float dh[64];
  if (a.d_final) {
    const float4 *src = reinterpret_cast<const float4 *>(a.d_final + (unit * K + kr) * V + 64 * hf);
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      const float4 v = src[x];
      dh[4 * x] = v.x; dh[4 * x + 1] = v.y; dh[4 * x + 2] = v.z; dh[4 * x + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int x = 0; x < 64; ++x) dh[x] = 0.f;
  }
  // dh' (bf16) -> the MMA operand tile (with dh_img, the tile itself is
  // copied out as the byte image of the gradient of the state leaving the
  // chunk it serves)
  auto store_hb = [&]() {
#pragma unroll
    for (int x = 0; x < 64; x += 8) {
      const uint4 v = make_uint4(pack_bf16(dh[x], dh[x + 1]), pack_bf16(dh[x + 2], dh[x + 3]),
                                 pack_bf16(dh[x + 4], dh[x + 5]), pack_bf16(dh[x + 6], dh[x + 7]));
      *reinterpret_cast<uint4 *>(sm + S_HB + mnmaj_off(128, kr, 64 * hf + x)) = v;
    }
  };
  store_hb();
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tD1 = tmem, tD2 = tmem + 128;

  // thread 0 starts the copies and the MMAs and counts them, for the drain.
  // Step i handles chunk nch - 1 - i in buffer i & 1.
  int64_t issued = 0, done = 0;
  auto load = [&](int64_t i) {
    const int bb = (int)(i & 1);
    const int64_t c = nch - 1 - i;
    uint8_t *dst = sm + bb * BUF_STRIDE;
    const char *src = a.pkg + (size_t)((c0 + c) * H + h) * PK_BYTES;
    tc::mbar_arrive_expect_tx(full + bb, has_do ? LOAD_BYTES : LOAD_BYTES - 16384);
    bulk_load(dst + B_WQ, src + PK_WQ, 32768, full + bb);
    bulk_load(dst + B_KG, src + PK_KG, PK_BYTES - PK_KG, full + bb);
    if (has_do) {
      const int32_t tok = (int32_t)(t0 + c * BT);
      tma_load_3d(dst + B_DO, &map_do, full + bb, 0, h, tok);
      tma_load_3d(dst + B_DO + 8192, &map_do, full + bb, 64, h, tok);
    }
    ++issued;
  };
  // d2_open: MMAs into D2 issued but not yet covered by a commit
  bool d1_pending = false, d2_pending = false, d2_open = false;
  uint32_t d1_par = 0, d2_par = 0;
  if (tid == 0)
    for (int64_t i = 0; i < 2 && i < nch; ++i) load(i);

  for (int64_t i = 0; i < nch; ++i) {
    const int b = (int)(i & 1);
    const int64_t c = nch - 1 - i;
    uint8_t *buf = sm + b * BUF_STRIDE;
    const int64_t tc0 = t0 + c * BT;
    const int len = (int)((t1 - tc0) < BT ? (t1 - tc0) : BT);
    bool ok = wait_or_flag(full + b, (uint32_t)((i >> 1) & 1), a.err);
    if (!ok) *abort_flag = 1;
    else if (tid == 0) done = i + 1;
    // e^{G_C} of this chunk, read now: the buffer is refilled as soon as the
    // chunk's last MMA has finished
    const float gcv = ok ? reinterpret_cast<const float *>(buf + B_GC)[kr] : 0.f;
    if (a.dhn) {  // gradient of the state leaving chunk c
      float4 *dst = reinterpret_cast<float4 *>(a.dhn + (((c0 + c) * H + h) * K + kr) * V + 64 * hf);
#pragma unroll
      for (int x = 0; x < 16; ++x) dst[x] = make_float4(dh[4 * x], dh[4 * x + 1], dh[4 * x + 2], dh[4 * x + 3]);
    }
    __syncthreads();  // dh' (bf16) and the chunk's operands are in place
    if (*abort_flag) break;

    if (tid == 0) {
      if (a.dh_img || a.dv_img) {
        // the previous step's -dv_new image has been read out of S_DV before
        // this step's replaces it; the dh' tile goes out as its image
        bulk_wait_read();
        if (a.dh_img) {
          bulk_store(a.dh_img + (size_t)((c0 + c) * H + h) * 32768, sm + S_HB, 32768);
          bulk_commit();
        }
      }
      tc::tc_fence_after();
      // ---- D1 = kg dh' + Aqk^T dO   (M = 64 tokens)
      const uint32_t idk = tc::idesc_bf16_f32(64, 128, false, true);
      const uint32_t g0 = tc::smem_u32(buf + B_KG), hb = tc::smem_u32(sm + S_HB);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc::mma_bf16(tD1, tc::smem_desc_sw128(g0 + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                     tc::smem_desc_sw128(hb + kk * 2048, 16384, 1024), idk, kk > 0);
      const uint32_t idt = tc::idesc_bf16_f32(64, 128, true, true);
      const uint32_t q0 = tc::smem_u32(buf + B_AQK), o0 = tc::smem_u32(buf + B_DO);
      if (has_do)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tD1, tc::smem_desc_sw128(q0 + kk * 2048, 8192, 1024),
                       tc::smem_desc_sw128(o0 + kk * 2048, 8192, 1024), idt, true);
      tc::mma_commit(bar_d1);
      d1_pending = true;
      d1_par = (uint32_t)(i & 1);
      // ---- D2 = qg^T dO  (M = 128 channels; w^T (-dv_new) follows)
      if (has_do) {
        const uint32_t idq = tc::idesc_bf16_f32(128, 128, true, true);
        const uint32_t w0 = tc::smem_u32(buf + B_WQ);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tD2, tc::smem_desc_sw128(w0 + kk * 2048, 16384, 1024),
                       tc::smem_desc_sw128(o0 + kk * 2048, 8192, 1024), idq, kk > 0);
        d2_open = true;
      }
    }

    // ---- dv_new: D1 row r (M = 64 layout) in TMEM lane (r % 16) + 32 (r / 16)
    __syncwarp();
    ok = __all_sync(0xffffffffu, wait_or_flag(bar_d1, (uint32_t)(i & 1), a.err));
    if (tid == 0 && ok) d1_pending = false;
    if (!ok) *abort_flag = 1;
    tc::tc_fence_after();
    if (ok) {
      const int r = 16 * q4 + lane;  // valid for lane < 16
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float d[16];
        __syncwarp();
        tc::tmem_ld16(tD1 + ((uint32_t)(32 * q4) << 16) + 64 * hf + 16 * cc, d);
        tc::tmem_ld_wait();
        if (lane < 16) {
          const int col = 64 * hf + 16 * cc;
          if (a.dvn && r < len) {
            float4 *dst = reinterpret_cast<float4 *>(a.dvn + ((tc0 + r) * H + h) * V + col);
#pragma unroll
            for (int x = 0; x < 4; ++x) dst[x] = make_float4(d[4 * x], d[4 * x + 1], d[4 * x + 2], d[4 * x + 3]);
          }
          const uint4 v0 = make_uint4(pack_bf16(-d[0], -d[1]), pack_bf16(-d[2], -d[3]),
                                      pack_bf16(-d[4], -d[5]), pack_bf16(-d[6], -d[7]));
          const uint4 v1 = make_uint4(pack_bf16(-d[8], -d[9]), pack_bf16(-d[10], -d[11]),
                                      pack_bf16(-d[12], -d[13]), pack_bf16(-d[14], -d[15]));
          *reinterpret_cast<uint4 *>(sm + S_DV + mnmaj_off(64, r, col)) = v0;
          *reinterpret_cast<uint4 *>(sm + S_DV + mnmaj_off(64, r, col + 8)) = v1;
        }
      }
    }
    // publish -dv_new (generic writes read by the tensor cores) and the end
    // of this warp's TMEM reads of D1
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(dv_ready);

    // ---- D2 += w^T (-dv_new); then the buffer takes step i + 2
    bool go = false;
    if (tid == 0) {
      go = !*abort_flag && wait_or_flag(dv_ready, (uint32_t)(i & 1), a.err);
      if (go) {
        // the dh' image has been read out of S_HB before the update below rewrites it
        if (a.dh_img) bulk_wait_read();
        tc::tc_fence_after();
        const uint32_t idq = tc::idesc_bf16_f32(128, 128, true, true);
        const uint32_t w0 = tc::smem_u32(buf + B_WQ), v0 = tc::smem_u32(sm + S_DV);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tD2, tc::smem_desc_sw128(w0 + (kk + 4) * 2048, 16384, 1024),
                       tc::smem_desc_sw128(v0 + kk * 2048, 8192, 1024), idq, has_do || kk > 0);
        tc::mma_commit(bar_d2);
        d2_pending = true;
        d2_open = false;
        d2_par = (uint32_t)(i & 1);
        if (a.dv_img) {  // the -dv_new tile goes out as its image
          bulk_store(a.dv_img + (size_t)((c0 + c) * H + h) * 16384, sm + S_DV, 16384);
          bulk_commit();
        }
      } else {
        *abort_flag = 1;
        if (d2_open) {  // cover the qg^T dO MMAs already issued, for the drain
          tc::mma_commit(bar_d2);
          d2_pending = true;
          d2_open = false;
          d2_par = (uint32_t)(i & 1);
        }
      }
    }
    __syncwarp();
    ok = __all_sync(0xffffffffu, wait_or_flag(bar_d2, (uint32_t)(i & 1), a.err));
    if (!ok) {
      *abort_flag = 1;
    } else {
      if (tid == 0) {
        d2_pending = false;
        if (i + 2 < nch && !*abort_flag) load(i + 2);  // every read of this buffer is done
      }
      tc::tc_fence_after();
      // ---- dh = e^{G_C} . dh' + D2
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float d[16];
        tc::tmem_ld16(tD2 + ((uint32_t)(32 * q4) << 16) + 64 * hf + 16 * cc, d);
        tc::tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 16; ++x) dh[16 * cc + x] = fmaf(gcv, dh[16 * cc + x], d[x]);
      }
      store_hb();
    }
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();
  }
  __syncthreads();

  if (*abort_flag == 0) {
    if (a.d_initial) {
      float4 *dst = reinterpret_cast<float4 *>(a.d_initial + (unit * K + kr) * V + 64 * hf);
#pragma unroll
      for (int x = 0; x < 16; ++x) dst[x] = make_float4(dh[4 * x], dh[4 * x + 1], dh[4 * x + 2], dh[4 * x + 3]);
    }
  } else if (tid == 0) {
    // a wait gave up: let the MMAs and copies this CTA started finish (each
    // wait bounded) before its tensor and shared memory are released
    if (d1_pending) drain_wait(bar_d1, d1_par);
    if (d2_pending) drain_wait(bar_d2, d2_par);
    for (int64_t x = done; x < issued; ++x) drain_wait(full + (x & 1), (uint32_t)((x >> 1) & 1));
  }
  if (tid == 0) bulk_wait_all();  // the image copies are complete before the CTA ends
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// State-contraction terms per (chunk, head) ([TPU] section 2.3, the parts of
// the WY backward that involve the states): with h the state entering the
// chunk and dh' the gradient of the state leaving it,
//   d(qg) = dO h^T,   dw = -dv_new h^T,   dkg = v_new dh'^T   (tcgen05, M=64,
//   N=128, K=128 value channels), d(e^{G_C}) = sum_v dh' . h  (fp32).
// The operands are the chains' bf16 tile images: the MN-major h / dh' tiles
// (K = channels) serve as K-major B operands of h^T / dh'^T, the MN-major
// v_new / -dv_new tiles (K = tokens) and the TMA dO tile as K-major A.
// ---------------------------------------------------------------------------
constexpr uint32_t T_H = 0, T_DH = 32768, T_DV = 65536, T_VN = 81920, T_DO = 98304;
constexpr uint32_t T_TILES = 114688;
// Two CTAs per SM: 2 x (dynamic + 1 KB reserved) must fit the SM's 228 KB, so
// the dynamic size is the tiles plus the 1 KB alignment allowance only; the
// 64 bytes of barriers go below the 1024-aligned tiles when the alignment gap
// holds them, else above the tiles (then the gap is under 64 bytes).
constexpr uint32_t T_SMEM = T_TILES + 1024;
static_assert(2 * (T_SMEM + 1024) <= 233472, "two CTAs per SM");
constexpr uint32_t T_TMEM = 256;

__global__ void __launch_bounds__(NT, 2)
tc_bwd_state_kernel(const __grid_constant__ CUtensorMap map_do, BwdStateArgs a, SeqInfo s, int H) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(sm - smem_raw >= 64 ? sm - 64 : sm + T_TILES);
  uint64_t *bar1 = full + 1, *bar2 = full + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(full + 3);
  volatile uint32_t *abort_flag = tslot + 1;
  const int64_t c = (int64_t)blockIdx.x / H;  // head fastest: adjacent CTAs share tokens
  const int h = (int)(blockIdx.x % H);
  int n, len;
  int64_t t0;
  if (!chunk_lookup(s, c, n, t0, len)) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q4 = warp & 3, hf = warp >> 2;
  const bool has_do = a.d_out != nullptr;
  const size_t item = (size_t)(c * H + h);

  if (warp == 0) {
    tc::tmem_alloc(tslot, T_TMEM);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(full, 1);
    tc::mbar_init(bar1, 1);
    tc::mbar_init(bar2, 1);
    tc::mbar_fence_init();
    *abort_flag = 0;
    tc::mbar_arrive_expect_tx(full, has_do ? 114688u : 98304u);
    bulk_load(sm + T_H, a.h_img + item * 32768, 32768, full);
    bulk_load(sm + T_DH, a.dh_img + item * 32768, 32768, full);
    bulk_load(sm + T_DV, a.dv_img + item * 16384, 16384, full);
    bulk_load(sm + T_VN, a.vn_img + item * 16384, 16384, full);
    if (has_do) {
      tma_load_3d(sm + T_DO, &map_do, full, 0, h, (int32_t)t0);
      tma_load_3d(sm + T_DO + 8192, &map_do, full, 64, h, (int32_t)t0);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = wait_or_flag(full, 0, a.err);
  if (!ok) *abort_flag = 1;
  __syncthreads();
  bool issued1 = false, issued2 = false;
  if (!*abort_flag && tid == 0) {
    tc::tc_fence_after();
    const uint32_t id = tc::idesc_bf16_f32(64, 128, false, false);
    const uint32_t hb = tc::smem_u32(sm + T_H), db = tc::smem_u32(sm + T_DH);
    const uint32_t ob = tc::smem_u32(sm + T_DO), vb = tc::smem_u32(sm + T_VN);
    if (has_do)  // d(qg) = dO h^T -> columns 0..127
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc::mma_bf16(tmem, tc::smem_desc_sw128(ob + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                     tc::smem_desc_sw128(hb + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), id, kk > 0);
    // dkg = v_new dh'^T -> columns 128..255
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      tc::mma_bf16(tmem + 128, tc::smem_desc_sw128(vb + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                   tc::smem_desc_sw128(db + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), id, kk > 0);
    tc::mma_commit(bar1);
    issued1 = true;
  }
  // d(e^{G_C}) = sum_v dh' . h per key channel, while the MMAs run
  if (!*abort_flag && tid < K) {
    float acc = 0.f;
#pragma unroll 4
    for (int v8 = 0; v8 < V; v8 += 8) {
      const uint4 x = *reinterpret_cast<const uint4 *>(sm + T_H + mnmaj_off(128, tid, v8));
      const uint4 y = *reinterpret_cast<const uint4 *>(sm + T_DH + mnmaj_off(128, tid, v8));
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xs[e]));
        const float2 yf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ys[e]));
        acc = fmaf(xf.x, yf.x, fmaf(xf.y, yf.y, acc));
      }
    }
    a.dgc[item * K + tid] = acc;
  }
  // readout of a 64 x 128 product (M = 64 layout: row r in TMEM lane
  // (r % 16) + 32 (r / 16)) into fp32 [T_tot, H, K] rows below len
  auto readout = [&](uint32_t tcol, float *dst, bool zero) {
    const int r = 16 * q4 + lane;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      float d[16];
      __syncwarp();
      tc::tmem_ld16(tcol + ((uint32_t)(32 * q4) << 16) + 64 * hf + 16 * cc, d);
      tc::tmem_ld_wait();
      if (lane < 16 && r < len) {
        float4 *o = reinterpret_cast<float4 *>(dst + ((t0 + r) * H + h) * (int64_t)K + 64 * hf + 16 * cc);
#pragma unroll
        for (int x = 0; x < 4; ++x)
          o[x] = zero ? make_float4(0.f, 0.f, 0.f, 0.f)
                      : make_float4(d[4 * x], d[4 * x + 1], d[4 * x + 2], d[4 * x + 3]);
      }
    }
  };
  __syncwarp();
  ok = !*abort_flag && __all_sync(0xffffffffu, wait_or_flag(bar1, 0, a.err));
  if (!ok) *abort_flag = 1;
  else {
    tc::tc_fence_after();
    readout(tmem, a.dqg, !has_do);
    readout(tmem + 128, a.dkg, false);
  }
  tc::tc_fence_before();
  __syncthreads();  // columns 0..127 are free again
  if (!*abort_flag && tid == 0) {
    tc::tc_fence_after();
    // dw = (-dv_new) h^T -> columns 0..127
    const uint32_t id = tc::idesc_bf16_f32(64, 128, false, false);
    const uint32_t hb = tc::smem_u32(sm + T_H), vb = tc::smem_u32(sm + T_DV);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      tc::mma_bf16(tmem, tc::smem_desc_sw128(vb + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                   tc::smem_desc_sw128(hb + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), id, kk > 0);
    tc::mma_commit(bar2);
    issued2 = true;
  }
  __syncwarp();
  ok = !*abort_flag && __all_sync(0xffffffffu, wait_or_flag(bar2, 0, a.err));
  if (!ok) *abort_flag = 1;
  else if (a.dw_img) {  // dw as a bf16 tile image, every row (zeros past the chunk end)
    tc::tc_fence_after();
    uint8_t *img = a.dw_img + item * 16384;
    const int r = 16 * q4 + lane;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      float d[16];
      __syncwarp();
      tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + 64 * hf + 16 * cc, d);
      tc::tmem_ld_wait();
      if (lane < 16) {
        const int col = 64 * hf + 16 * cc;
        const bool in = r < len;
        *reinterpret_cast<uint4 *>(img + mnmaj_off(64, r, col)) =
            in ? make_uint4(pack_bf16(d[0], d[1]), pack_bf16(d[2], d[3]), pack_bf16(d[4], d[5]),
                            pack_bf16(d[6], d[7]))
               : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(img + mnmaj_off(64, r, col + 8)) =
            in ? make_uint4(pack_bf16(d[8], d[9]), pack_bf16(d[10], d[11]), pack_bf16(d[12], d[13]),
                            pack_bf16(d[14], d[15]))
               : make_uint4(0, 0, 0, 0);
      }
    }
  } else {
    tc::tc_fence_after();
    readout(tmem, a.dw, false);
  }
  if (*abort_flag && tid == 0) {  // bounded drain of what this CTA started
    drain_wait(full, 0);
    if (issued1) drain_wait(bar1, 0);
    if (issued2) drain_wait(bar2, 0);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, T_TMEM);
}

}  // namespace

cudaError_t launch_tc_bwd_state(const BwdStateArgs &a, const SeqInfo &s, int64_t nchunks, int H,
                                cudaStream_t st) {
  if (nchunks == 0 || H == 0) return cudaSuccess;
  CUtensorMap map_do;
  memset(&map_do, 0, sizeof(map_do));  // not read without d_out
  if (a.d_out && (s.T_tot <= 0 || !make_value_map(a.d_out, s.T_tot, H, map_do))) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)T_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(nchunks * H));
  tc_bwd_state_kernel<<<grid, NT, T_SMEM, st>>>(map_do, a, s, H);
  return cudaGetLastError();
}

cudaError_t launch_tc_bwd_dh(const BwdChainArgs &a, const SeqInfo &s, int H, int64_t T_tot,
                             cudaStream_t st) {
  const int64_t units = (int64_t)s.N * H;
  if (units == 0) return cudaSuccess;
  CUtensorMap map_do;
  memset(&map_do, 0, sizeof(map_do));  // not read without d_out
  if (a.d_out && (T_tot <= 0 || !make_value_map(a.d_out, T_tot, H, map_do))) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_dh_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  tc_bwd_dh_kernel<<<(unsigned)units, NT, SMEM_BYTES, st>>>(map_do, a, s, H);
  return cudaGetLastError();
}

}  // namespace tcp
}  // namespace kda
