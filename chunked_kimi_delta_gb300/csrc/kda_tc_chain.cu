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
// channels); a bf16 copy in shared memory is the MMA operand.  Only
// [qg; w] h -> v_new -> kg^T v_new -> h' is on the recurrence's critical path:
// warps of lane quarters 2 and 3 compute v_new and signal it through an
// mbarrier to the thread that issues the MMAs; kg^T v_new commits to its own
// barrier ahead of Aqk v_new; the output tile P alternates between two TMEM
// buffers, so the warps of lane quarters 0 and 1 read o of chunk c while the
// first MMA of chunk c + 1 runs.  Packages are double-buffered in two halves
// that are refilled as soon as their last reader is done: WQ and U of chunk
// c + 2 once v_new of chunk c is computed, KG, AQK and GC of chunk c + 1 once
// the MMAs of chunk c - 1 have finished.  o of a full chunk is staged in
// shared memory and written by TMA tensor stores; the backward's bf16 tile
// images of h and v_new are the shared-memory tiles themselves, copied out
// by one bulk copy each per chunk.
//
#include <cuda_bf16.h>
#include <string.h>

#include "kda_tc.cuh"

namespace kda {
namespace tcp {
namespace {

constexpr int NT = 256;
constexpr uint32_t S_BUF0 = 0;
constexpr uint32_t S_BAR = PK_BYTES;         // mbarriers in the gap before buffer 1
constexpr uint32_t S_BUF1 = 74752;           // 1024-aligned
constexpr uint32_t S_HB = 149504;            // h bf16, MN-major (K = 128 channels)
constexpr uint32_t S_VN = 182272;            // v_new bf16, MN-major (K = 64 tokens)
constexpr uint32_t S_OST = 198656;           // o of a full chunk, bf16, staged for the TMA store
constexpr uint32_t SMEM_BYTES = S_OST + 16384 + 1024;
static_assert(S_OST % 1024 == 0 && SMEM_BYTES <= 232448, "shared memory layout");
constexpr uint32_t BUF_STRIDE = S_BUF1 - S_BUF0;
constexpr uint32_t TMEM_COLS = 512;          // P (two buffers) and U

// 3-D TMA store of a staged tile (coordinates: channel, head, token), tracked
// by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int32_t x, int32_t y,
                                             int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
               :: "l"(reinterpret_cast<uint64_t>(map)), "r"(tc::smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Barrier over the 128 threads of the o warps (lane quarters 0 and 1), the
// AND of their flags returned to each.
__device__ __forceinline__ bool o_warps_and(bool v) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 128, p;\n\t"
               "selp.u32 %0, 1, 0, q;\n\t}"
               : "=r"(r) : "r"((uint32_t)v) : "memory");
  return r != 0;
}

// EXTRAS: the optional outputs (per-chunk states and v_new, the backward's
// tile images, the test-only wait); the instantiation without them keeps the
// per-chunk loops free of their branches.
template <bool EXTRAS>
__global__ void __launch_bounds__(NT, 1) tc_chain_kernel(const __grid_constant__ CUtensorMap map_o,
                                                         ChainArgs a, SeqInfo s, int H, bool o_tma) {
  if (!EXTRAS) {
    a.h_out = a.v_new_out = nullptr;
    a.h_img = a.vn_img = nullptr;
    a.test_wait_timeout = false;
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *fullA = reinterpret_cast<uint64_t *>(sm + S_BAR);  // [2] WQ, U of a buffer
  uint64_t *fullB = fullA + 2;   // [2] KG, AQK, GC of a buffer
  uint64_t *bar_ma = fullA + 4;  // [qg; w] h
  uint64_t *bar_mc = fullA + 5;  // kg^T v_new
  uint64_t *bar_mb = fullA + 6;  // Aqk v_new
  uint64_t *vn_ready = fullA + 7;  // v_new of the chunk is in shared memory (4 warp arrivals)
  uint32_t *tslot = reinterpret_cast<uint32_t *>(fullA + 8);
  volatile uint32_t *abort_flag = tslot + 1;
  uint64_t *bar_never = fullA + 16;  // test only: a barrier nothing completes

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q4 = warp & 3, hf = warp >> 2;
  const int kr = 32 * q4 + lane;  // key channel (state row) owned by this thread
  // the caller's state window: rows < dk, columns < dv (narrow heads: the rest
  // of the 128 x 128 state stays zero and is not stored)
  const int dk = a.dk, dv = a.dv;
  const bool sown = kr < dk && 64 * hf < dv;
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
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(fullA + x, 1);
      tc::mbar_init(fullB + x, 1);
    }
    tc::mbar_init(bar_ma, 1);
    tc::mbar_init(bar_mc, 1);
    tc::mbar_init(bar_mb, 1);
    tc::mbar_init(vn_ready, 4);
    tc::mbar_init(bar_never, 1);
    tc::mbar_fence_init();
    *abort_flag = 0;
  }

  // initial state -> registers and the bf16 operand
  float hr[64];
  if (a.initial_state && sown) {
    const float4 *src = reinterpret_cast<const float4 *>(a.initial_state + (unit * dk + kr) * dv + 64 * hf);
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      const float4 v = src[x];
      hr[4 * x] = v.x; hr[4 * x + 1] = v.y; hr[4 * x + 2] = v.z; hr[4 * x + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int x = 0; x < 64; ++x) hr[x] = 0.f;
  }
  // h (bf16) -> the MMA operand tile (with h_img, the tile itself is copied
  // out as the byte image of the state entering the chunk, for the backward)
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
  const uint32_t tU = tmem + 256;  // P buffers at columns 0 and 128

  // thread LEAD (lane 0 of the first v_new warp) starts the package copies
  // and the MMAs and keeps count of them, for the drain.  Buffer b holds
  // chunks b, b + 2, ...; its first half (WQ, U) is free once v_new of its
  // chunk is done, its second half (KG, AQK, GC) once the chunk's last MMA is.
  constexpr int LEAD = 64;
  int64_t a_issued = 0, a_done = 0, b_issued = 0, b_done = 0;
  auto load_a = [&](int64_t cc) {
    const int bb = (int)(cc & 1);
    tc::mbar_arrive_expect_tx(fullA + bb, PK_FIRST);
    bulk_load(sm + S_BUF0 + bb * BUF_STRIDE, a.pkg + (size_t)((c0 + cc) * H + h) * PK_BYTES, PK_FIRST,
              fullA + bb);
    ++a_issued;
  };
  auto load_b = [&](int64_t cc) {
    const int bb = (int)(cc & 1);
    tc::mbar_arrive_expect_tx(fullB + bb, PK_BYTES - PK_FIRST);
    bulk_load(sm + S_BUF0 + bb * BUF_STRIDE + PK_FIRST,
              a.pkg + (size_t)((c0 + cc) * H + h) * PK_BYTES + PK_FIRST, PK_BYTES - PK_FIRST, fullB + bb);
    ++b_issued;
  };
  bool ma_pending = false, mc_pending = false, mb_issued = false;
  uint32_t ma_par = 0, mc_par = 0, mb_par = 0;  // parity of the last completion
  if (tid == LEAD) {
    for (int64_t c = 0; c < 2 && c < nch; ++c) {
      load_a(c);
      load_b(c);
    }
  }

  // o of a finished chunk: P rows 0..63 of its buffer, by the warps of lane
  // quarters 0 and 1 once Aqk v_new has landed (Mb completion number cp).  A
  // full chunk goes out through the shared staging tile and one TMA store
  // per 64 columns (whole 128-byte lines); a shorter one (the end of a
  // sequence: the rows after it belong to the next) row by row.
  auto read_o = [&](int64_t cp, int lenp) {
    // tcgen05.ld needs the whole warp, the staging tile all four o warps: act
    // on a verdict shared by the four
    bool ok = __all_sync(0xffffffffu, wait_or_flag(bar_mb, (uint32_t)(cp & 1), a.err));
    const bool staged = o_tma && a.out && lenp == BT;
    if (staged) {
      if (tid == 0) bulk_wait_read();  // the previous tile's store has read the staging buffer
      ok = o_warps_and(ok);
    }
    if (!ok) { *abort_flag = 1; return; }
    tc::tc_fence_after();
    const uint32_t tPp = tmem + 128u * (uint32_t)(cp & 1);
    const int r = 32 * q4 + lane;
    const int64_t tcp = t0 + cp * BT;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      float d[16];
      __syncwarp();
      tc::tmem_ld16(tPp + ((uint32_t)(32 * q4) << 16) + 64 * hf + 16 * cc, d);
      tc::tmem_ld_wait();
      const uint4 o0 = make_uint4(pack_bf16(d[0], d[1]), pack_bf16(d[2], d[3]), pack_bf16(d[4], d[5]),
                                  pack_bf16(d[6], d[7]));
      const uint4 o1 = make_uint4(pack_bf16(d[8], d[9]), pack_bf16(d[10], d[11]), pack_bf16(d[12], d[13]),
                                  pack_bf16(d[14], d[15]));
      const int col = 64 * hf + 16 * cc;
      if (staged) {
        *reinterpret_cast<uint4 *>(sm + S_OST + mnmaj_off(64, r, col)) = o0;
        *reinterpret_cast<uint4 *>(sm + S_OST + mnmaj_off(64, r, col + 8)) = o1;
      } else if (a.out && r < lenp && 64 * hf < dv) {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + ((tcp + r) * H + h) * dv + col);
        dst[0] = o0;
        dst[1] = o1;
      }
    }
    if (staged) {
      tc::fence_proxy_async_smem();  // the tile's generic writes, before the TMA reads it
      o_warps_and(true);
      if (tid == 0) {
        tma_store_3d(&map_o, sm + S_OST, 0, h, (int32_t)tcp);
        if (dv == 128) tma_store_3d(&map_o, sm + S_OST + 8192, 64, h, (int32_t)tcp);
        bulk_commit();
      }
    }
  };

  for (int64_t c = 0; c < nch; ++c) {
    const int b = (int)(c & 1);
    uint8_t *buf = sm + S_BUF0 + b * BUF_STRIDE;
    const int64_t tc0 = t0 + c * BT;
    const int len = (int)((t1 - tc0) < BT ? (t1 - tc0) : BT);
    const uint32_t tP = tmem + 128u * (uint32_t)b;
    bool ok = wait_or_flag(fullA + b, (uint32_t)((c >> 1) & 1), a.err);
    if (!ok) *abort_flag = 1;
    else if (tid == LEAD) a_done = c + 1;
    // test only: give up on a wait with the next copies still in flight
    if (a.test_wait_timeout && c == 0 && tid == LEAD && !wait_or_flag(bar_never, 0, a.err, 1000000ull))
      *abort_flag = 1;
    if (a.h_out && sown) {
      float4 *dst = reinterpret_cast<float4 *>(a.h_out + (((c0 + c) * H + h) * dk + kr) * dv + 64 * hf);
#pragma unroll
      for (int x = 0; x < 16; ++x) dst[x] = make_float4(hr[4 * x], hr[4 * x + 1], hr[4 * x + 2], hr[4 * x + 3]);
    }
    __syncthreads();  // h (bf16) of this chunk and the package are in place
    if (*abort_flag) break;

    // ---- [qg; w] h -> P (this chunk's buffer)
    if (tid == LEAD) {
      if (a.h_img || a.vn_img) {
        // the previous chunk's v_new image has been read out of S_VN before
        // this chunk's v_new replaces it; the h tile goes out as its image
        bulk_wait_read();
        if (a.h_img) {
          bulk_store(a.h_img + (size_t)((c0 + c) * H + h) * 32768, sm + S_HB, 32768);
          bulk_commit();
        }
      }
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(128, 128, false, true);
      const uint32_t a0 = tc::smem_u32(buf + PK_WQ), b0 = tc::smem_u32(sm + S_HB);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc::mma_bf16(tP, tc::smem_desc_sw128(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                     tc::smem_desc_sw128(b0 + kk * 2048, 16384, 1024), idesc, kk > 0);
      tc::mma_commit(bar_ma);
      ma_pending = true;
      ma_par = (uint32_t)(c & 1);
    }
    // warps of lane quarters 0 and 1: o of the previous chunk, off the
    // recurrence's critical path
    if (q4 < 2 && c > 0) read_o(c - 1, BT);

    // ---- v_new = u - w h  (P rows 64..127 live in TMEM lanes 64..127), by
    //      the warps of lane quarters 2 and 3
    if (q4 >= 2) {
      __syncwarp();
      ok = __all_sync(0xffffffffu, wait_or_flag(bar_ma, (uint32_t)(c & 1), a.err));
      if (tid == LEAD && ok) {
        ma_pending = false;
        // every MMA of chunk c - 1 has finished: the second half of its
        // buffer takes chunk c + 1
        if (c > 0 && c + 1 < nch && !*abort_flag) load_b(c + 1);
      }
      if (!ok) *abort_flag = 1;
      tc::tc_fence_after();
    }
    if (ok && q4 >= 2) {
      const int r = 32 * (q4 - 2) + lane;
      constexpr int PER = 4;  // TMEM loads per wait (all four, then one wait)
#pragma unroll
      for (int cg = 0; cg < 4; cg += PER) {
      float dd[PER][16];
      uint4 uu[PER][2];
      __syncwarp();
#pragma unroll
      for (int x = 0; x < PER; ++x)
        tc::tmem_ld16(tP + ((uint32_t)(32 * q4) << 16) + 64 * hf + 16 * (cg + x), dd[x]);
#pragma unroll
      for (int x = 0; x < PER; ++x) {
        const int colx = 64 * hf + 16 * (cg + x);
        uu[x][0] = *reinterpret_cast<const uint4 *>(buf + PK_U + u_offset(r, colx));
        uu[x][1] = *reinterpret_cast<const uint4 *>(buf + PK_U + u_offset(r, colx + 8));
      }
      tc::tmem_ld_wait();
#pragma unroll
      for (int x = 0; x < PER; ++x) {
        const int cc = cg + x;
        const float *d = dd[x];
        const int col = 64 * hf + 16 * cc;
        float vn[16];
        {
          const uint4 ua = uu[x][0], ub = uu[x][1];
          const uint32_t uw[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
          for (int x2 = 0; x2 < 8; ++x2) {
            const float2 u2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&uw[x2]));
            vn[2 * x2] = u2.x - d[2 * x2];
            vn[2 * x2 + 1] = u2.y - d[2 * x2 + 1];
          }
        }
        const uint4 v0 = make_uint4(pack_bf16(vn[0], vn[1]), pack_bf16(vn[2], vn[3]),
                                    pack_bf16(vn[4], vn[5]), pack_bf16(vn[6], vn[7]));
        const uint4 v1 = make_uint4(pack_bf16(vn[8], vn[9]), pack_bf16(vn[10], vn[11]),
                                    pack_bf16(vn[12], vn[13]), pack_bf16(vn[14], vn[15]));
        *reinterpret_cast<uint4 *>(sm + S_VN + mnmaj_off(64, r, col)) = v0;
        *reinterpret_cast<uint4 *>(sm + S_VN + mnmaj_off(64, r, col + 8)) = v1;
        if (a.v_new_out && r < len && col < dv) {
          float4 *dst = reinterpret_cast<float4 *>(a.v_new_out + ((tc0 + r) * H + h) * dv + col);
#pragma unroll
          for (int x3 = 0; x3 < 4; ++x3) dst[x3] = make_float4(vn[4 * x3], vn[4 * x3 + 1], vn[4 * x3 + 2], vn[4 * x3 + 3]);
        }
      }
      }
    }
    if (q4 >= 2) {
      // publish v_new (generic writes, read by the tensor cores) and the end
      // of this warp's TMEM reads of P
      tc::tc_fence_before();
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(vn_ready);
    }

    // ---- kg^T v_new -> U (critical path, own barrier), then
    //      P[0:64] += Aqk v_new (rows 64..127 of the A operand are unused)
    bool go = false;
    if (tid == LEAD) {
      go = !*abort_flag && wait_or_flag(vn_ready, (uint32_t)(c & 1), a.err);
      if (go) {
        // WQ and U of this chunk are consumed: the first half takes chunk c + 2
        if (c + 2 < nch) load_a(c + 2);
        go = wait_or_flag(fullB + b, (uint32_t)((c >> 1) & 1), a.err);
        if (go) b_done = c + 1;
      }
      if (!go) *abort_flag = 1;
    }
    if (go) {
      // the h image has been read out of S_HB before the update below rewrites it
      if (a.h_img) bulk_wait_read();
      tc::tc_fence_after();
      const uint32_t vn0 = tc::smem_u32(sm + S_VN);
      const uint32_t idc = tc::idesc_bf16_f32(128, 128, true, true);
      const uint32_t g0 = tc::smem_u32(buf + PK_KG);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_bf16(tU, tc::smem_desc_sw128(g0 + kk * 2048, 8192, 1024),
                     tc::smem_desc_sw128(vn0 + kk * 2048, 8192, 1024), idc, kk > 0);
      tc::mma_commit(bar_mc);
      mc_pending = true;
      mc_par = (uint32_t)(c & 1);
      {
        const uint32_t idb = tc::idesc_bf16_f32(128, 128, false, true);
        const uint32_t q0 = tc::smem_u32(buf + PK_AQK);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tP, tc::smem_desc_sw128(q0 + kk * 32, 16, 1024),
                       tc::smem_desc_sw128(vn0 + kk * 2048, 8192, 1024), idb, true);
        tc::mma_commit(bar_mb);
        mb_issued = true;
        mb_par = (uint32_t)(c & 1);
      }
      if (a.vn_img) {  // the v_new tile goes out as its image, for the backward
        bulk_store(a.vn_img + (size_t)((c0 + c) * H + h) * 16384, sm + S_VN, 16384);
        bulk_commit();
      }
    }
    __syncwarp();
    ok = __all_sync(0xffffffffu, wait_or_flag(bar_mc, (uint32_t)(c & 1), a.err));
    if (tid == LEAD && ok) mc_pending = false;
    if (!ok) {
      *abort_flag = 1;
    } else {
      tc::tc_fence_after();
      wait_or_flag(fullB + b, (uint32_t)((c >> 1) & 1), a.err);  // complete: acquires GC
      // ---- h' = e^{G_C} h + kg^T v_new
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
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();
  }
  // o of the last chunk
  __syncthreads();
  if (nch > 0 && !*abort_flag && q4 < 2) read_o(nch - 1, (int)(t1 - (t0 + (nch - 1) * BT)));
  __syncthreads();

  if (*abort_flag == 0) {
    if (a.final_state && sown) {
      float4 *dst = reinterpret_cast<float4 *>(a.final_state + (unit * dk + kr) * dv + 64 * hf);
#pragma unroll
      for (int x = 0; x < 16; ++x) dst[x] = make_float4(hr[4 * x], hr[4 * x + 1], hr[4 * x + 2], hr[4 * x + 3]);
    }
  } else if (tid == LEAD) {
    // a wait gave up: let the MMAs and copies this CTA started finish (each
    // wait bounded) before its tensor and shared memory are released
    if (ma_pending) drain_wait(bar_ma, ma_par);
    if (mc_pending) drain_wait(bar_mc, mc_par);
    if (mb_issued) drain_wait(bar_mb, mb_par);
    for (int64_t c = a_done; c < a_issued; ++c) drain_wait(fullA + (c & 1), (uint32_t)((c >> 1) & 1));
    for (int64_t c = b_done; c < b_issued; ++c) drain_wait(fullB + (c & 1), (uint32_t)((c >> 1) & 1));
  }
  // the TMA stores of o (thread 0) and the image copies (LEAD) are complete
  // before the CTA ends
  if (tid == 0 || tid == LEAD) bulk_wait_all();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_tc_chain(const ChainArgs &a, const SeqInfo &s, int H, cudaStream_t st) {
  const int64_t units = (int64_t)s.N * H;
  if (units == 0) return cudaSuccess;
  const bool extras = a.h_out || a.v_new_out || a.h_img || a.vn_img || a.test_wait_timeout;
  auto kern = extras ? tc_chain_kernel<true> : tc_chain_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // o of full chunks by TMA: [T_tot, H, dv] bf16 with 16-byte aligned rows
  // (without a map the rows are stored one by one)
  CUtensorMap map_o;
  memset(&map_o, 0, sizeof(map_o));
  const bool o_tma = a.out && (reinterpret_cast<uintptr_t>(a.out) & 15u) == 0 &&
                     make_out_map(a.out, s.T_tot, H, a.dv, map_o);
  kern<<<(unsigned)units, NT, SMEM_BYTES, st>>>(map_o, a, s, H, o_tma);
  return cudaGetLastError();
}

}  // namespace tcp
}  // namespace kda
