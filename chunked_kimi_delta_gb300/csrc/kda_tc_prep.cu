// kda_tc_prep.cu - intra-chunk stage of the tensor-core KDA forward.
//
// Per (chunk, head), following "KDA Chunk Backward - TPU/Pallas Kernel
// Design" sections 1.2 (WY representation), 3.1 (base-2 gates) and 3.7
// (sub-block reference gates):
//   g     = gate(x) in log2 units; G = chunk-local inclusive cumsum
//   L_rj  = beta_r sum_c k^_rc k^_jc 2^{G_rc - G_jc}          (j < r)
//   Aqk_rj = scale sum_c q^_rc k^_jc 2^{G_rc - G_jc}         (j <= r)
//   A = (I + L)^-1, w = A (k^ . beta . 2^G), u = A (v . beta)
//   qg = scale q^ . 2^G, kg = k^ . 2^{G_C - G}, gC = 2^{G_C}
//
// Decay factorisation.  2^{G_r - G_j} is split around a reference gate b
// that sits between j and r, so that no factor exceeds 1 where it matters:
// the chunk is cut into four 16-token sub-blocks with b_R the cumulative gate
// at the end of sub-block R-1 (b_0 = 0).  Row r of sub-block R carries
// 2^{G_r - b_R} <= 1; column j is stored once per later sub-block R' as
// 2^{b_R' - G_j} <= 1 (off-diagonal blocks) and once with its own block's
// reference, 2^{b_R(j) - G_j} (diagonal blocks, bounded by 16 tokens of
// decay; clamped at 2^126, i.e. exact unless the gate falls below about
// -5.5 nats per token for 16 tokens in a row).  One M=128 x N=160 x K=128
// tcgen05 MMA then yields every needed block of both A_kk and A_qk:
//   A rows  0..63 : k^_r 2^{G_r - b_R}      A rows 64..127: q^_r 2^{G_r - b_R}
//   B rows  0..15 : k^_j 2^{b_1 - G_j}, j < 16
//   B rows 16..47 : k^_j 2^{b_2 - G_j}, j < 32
//   B rows 48..95 : k^_j 2^{b_3 - G_j}, j < 48
//   B rows 96..159: k^_j 2^{b_R(j) - G_j}, j < 64 (own block)
//
// One persistent CTA per SM loops over (chunk, head) items; TMA brings the
// next item's q, k, gate input and v while the current one computes.
#include <cuda_bf16.h>

#include "kda_tc.cuh"

namespace kda {
namespace tcp {
namespace {

constexpr int NT = 256;   // two CTAs (two items) per SM

// Shared memory (bytes from a 1024-aligned base), about 108 KB per CTA.
constexpr uint32_t S_V = 0;          // v, MN-major SW128 (K = tokens), TMA destination
constexpr uint32_t S_OPA = 16384;    // [k E ; q E] K-major, 128 rows (32768)
constexpr uint32_t S_B1 = 49152;     // 160 rows K-major (2 panels x 20480)
constexpr uint32_t S_B2A = 90112;    // k^ 2^G, MN-major (16384)
// after the first MMA the OPA/B1 region is reused:
constexpr int LFS = 68;              // row stride of L (16-byte aligned rows)
constexpr uint32_t S_LF = 16384;     // fp32 L [64][68]
constexpr uint32_t S_AF = 33792;     // fp32 A [64][65]
constexpr uint32_t S_TT = 50432;     // fp32 scratch [32][33]
constexpr uint32_t S_AINV = 55296;   // bf16 A.diag(beta), K-major 64 rows (8192)
// staging of package parts for bulk stores (regions free at that time):
constexpr uint32_t S_STG_AQK = 73728;  // Aqk image (8192), written after MMA 1 (B1 dead)
constexpr uint32_t S_STG_W = 16384;    // w rows of WQ, 2 panels x 8192, after MMA 2
constexpr uint32_t S_STG_U = 32768;    // U image (32768), after MMA 2
constexpr uint32_t S_MISC = 106496;
constexpr uint32_t M_RQ = S_MISC;           // fp32 [64] rstd q
constexpr uint32_t M_RK = S_MISC + 256;     // fp32 [64] rstd k
constexpr uint32_t M_BETA = S_MISC + 512;   // fp32 [64]
constexpr uint32_t M_TOT = S_MISC + 768;    // fp32 [4][128] sub-block gate totals
constexpr uint32_t M_BAR = S_MISC + 2816;   // bar_v, bar_mma
constexpr uint32_t M_TSLOT = S_MISC + 2832;
constexpr uint32_t M_ABORT = S_MISC + 2836;
constexpr uint32_t M_ITEM = S_MISC + 2848;  // 2 x ItemSlot
constexpr uint32_t SMEM_BYTES = S_MISC + 2912 + 1024;

constexpr uint32_t B1_PANEL = 160 * 128;
constexpr uint32_t TMEM_COLS = 256;

__device__ __forceinline__ int b1_off(int Rp) { return 8 * Rp * (Rp - 1); }  // 0, 16, 48

struct Item {
  int n, len, h;
  int64_t t0, gc;
  bool ok;
};

// What every thread needs of an item; written by thread 0, read by all.
struct ItemSlot {
  int64_t t0, gc;
  int32_t len, h, ok, pad;
};

__device__ __forceinline__ Item get_item(const SeqInfo &s, int H, int64_t w) {
  Item it;
  it.gc = w / H;
  it.h = (int)(w % H);
  it.ok = chunk_lookup(s, it.gc, it.n, it.t0, it.len);
  return it;
}

__device__ __forceinline__ void issue_v(const TcMaps &m, uint8_t *dst, uint64_t *bar,
                                        const Item &it) {
  tc::mbar_arrive_expect_tx(bar, 16384);
  tma_load_3d(dst, &m.v, bar, 0, it.h, (int32_t)it.t0);
  tma_load_3d(dst + 8192, &m.v, bar, 64, it.h, (int32_t)it.t0);
}

__device__ __forceinline__ void put_slot(ItemSlot &sl, const Item &it, bool ok) {
  sl.t0 = it.t0;
  sl.gc = it.gc;
  sl.len = it.len;
  sl.h = it.h;
  sl.ok = ok ? 1 : 0;
}

__device__ __forceinline__ void st_u32(uint8_t *base, uint32_t off, uint32_t v) {
  *reinterpret_cast<uint32_t *>(base + off) = v;
}

template <typename T>
__device__ __forceinline__ T ldg_stream(const T *p) {
  return __ldg(p);
}

__global__ void __launch_bounds__(NT, 2)
tc_prep_kernel(const __grid_constant__ TcMaps maps, const __nv_bfloat16 *__restrict__ qg_in,
               const __nv_bfloat16 *__restrict__ kg_in, const float *__restrict__ xg_in,
               const float *__restrict__ beta, GateParams gp, SeqInfo s, int64_t nitems, int H,
               char *__restrict__ pkg, uint32_t *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *rq = reinterpret_cast<float *>(sm + M_RQ);
  float *rk = reinterpret_cast<float *>(sm + M_RK);
  float *sbeta = reinterpret_cast<float *>(sm + M_BETA);
  float *tot = reinterpret_cast<float *>(sm + M_TOT);
  uint64_t *bar_v = reinterpret_cast<uint64_t *>(sm + M_BAR);
  uint64_t *bar_mma = bar_v + 1;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + M_TSLOT);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sm + M_ABORT);
  ItemSlot *slots = reinterpret_cast<ItemSlot *>(sm + M_ITEM);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;
  const bool l2n = (gp.flags & KDA_L2NORM_QK) != 0;
  const bool sig = (gp.flags & KDA_BETA_SIGMOID) != 0;
  constexpr float kLog2e = 1.4426950408889634f;
  const int64_t rowH = (int64_t)H * 128;  // elements between consecutive tokens

  if (warp == 0) {
    tc::tmem_alloc(tslot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar_v, 1);
    tc::mbar_init(bar_mma, 1);
    tc::mbar_fence_init();
    *abort_flag = 0;
    tc::tma_prefetch_desc(&maps.v);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;

  // elementwise roles: channel pair p (channels c0, c0 + 1), sub-block R
  // (rows 16 R .. 16 R + 15)
  const int p = tid & 63, R = tid >> 6;
  const int c0 = 2 * p;
  const uint32_t ch16 = (uint32_t)((c0 & 63) >> 3), cbyte = (uint32_t)(c0 & 7) * 2u;
  const uint32_t pan = (uint32_t)(c0 >> 6);

  const int64_t G = gridDim.x;
  // thread 0 keeps count of the loads and MMAs it started, for the drain
  int64_t v_issued = 0, v_done = 0;
  bool mma_pending = false;
  if (tid == 0) {
    Item it0 = get_item(s, H, blockIdx.x);
    const bool ok0 = blockIdx.x < nitems && it0.ok;
    put_slot(slots[0], it0, ok0);
    if (ok0) {
      issue_v(maps, sm + S_V, bar_v, it0);
      v_issued = 1;
    }
  }
  __syncthreads();

  uint32_t mma_phase = 0;
  int64_t i = 0;
  for (int64_t w = blockIdx.x; w < nitems; w += G, ++i) {
    const ItemSlot it = slots[i & 1];
    if (!it.ok) break;  // items past the last chunk are all invalid
    const int len = it.len, h = it.h;
    const int64_t t0 = it.t0;
    uint8_t *pk = reinterpret_cast<uint8_t *>(pkg + (size_t)(it.gc * H + h) * PK_BYTES);
    const int64_t base_h = t0 * rowH + (int64_t)h * 128;  // element offset of (t0, h, 0)
    Item nx;
    bool okn = false;
    if (tid == 0) {
      const int64_t wn = w + G;
      nx = get_item(s, H, wn < nitems ? wn : 0);
      okn = wn < nitems && nx.ok;
      put_slot(slots[(i + 1) & 1], nx, okn);
      if (okn) {
        tma_prefetch_l2_3d(&maps.q, 0, nx.h, (int32_t)nx.t0);
        tma_prefetch_l2_3d(&maps.k, 0, nx.h, (int32_t)nx.t0);
        tma_prefetch_l2_3d(&maps.x, 0, nx.h, (int32_t)nx.t0);
      }
    }

    // ---- pass A: row norms of q and k (8 rows per warp), beta; all loads
    //      are issued before any arithmetic
    {
      uint2 qa[8], ka[8];
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int r = warp * 8 + rr;
        qa[rr] = make_uint2(0, 0);
        ka[rr] = make_uint2(0, 0);
        if (r < len) {
          qa[rr] = ldg_stream(reinterpret_cast<const uint2 *>(qg_in + base_h + r * rowH) + lane);
          ka[rr] = ldg_stream(reinterpret_cast<const uint2 *>(kg_in + base_h + r * rowH) + lane);
        }
      }
      float sq[8], sk[8];
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qa[rr]);
        const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&ka[rr]);
        const float2 a0 = __bfloat1622float2(q2[0]), a1 = __bfloat1622float2(q2[1]);
        const float2 b0 = __bfloat1622float2(k2[0]), b1 = __bfloat1622float2(k2[1]);
        sq[rr] = a0.x * a0.x + a0.y * a0.y + a1.x * a1.x + a1.y * a1.y;
        sk[rr] = b0.x * b0.x + b0.y * b0.y + b1.x * b1.x + b1.y * b1.y;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          sq[rr] += __shfl_xor_sync(0xffffffffu, sq[rr], o);
          sk[rr] += __shfl_xor_sync(0xffffffffu, sk[rr], o);
        }
      if (lane < 8) {
        const int r = warp * 8 + lane;
        float vq = sq[0], vk = sk[0];
#pragma unroll
        for (int rr = 1; rr < 8; ++rr)
          if (lane == rr) { vq = sq[rr]; vk = sk[rr]; }
        const bool v = r < len;
        rq[r] = v ? (l2n ? rsqrtf(vq + gp.eps) : 1.f) : 0.f;
        rk[r] = v ? (l2n ? rsqrtf(vk + gp.eps) : 1.f) : 0.f;
      }
      if (tid < 64) {
        float b = 0.f;
        if (tid < len) {
          b = beta[(t0 + tid) * H + h];
          if (sig) b = 1.f / (1.f + tc::ex2(-b * kLog2e));
        }
        sbeta[tid] = b;
      }
    }

    // ---- phase 1: gate (log2 units) and the sub-block cumulative sums
    float Gl[16][2];
    {
      const float A_h = gate ? tc::ex2(gp.a_log[h] * kLog2e) : 0.f;
      const float db0 = (gate && gp.dt_bias) ? gp.dt_bias[h * 128 + c0] : 0.f;
      const float db1 = (gate && gp.dt_bias) ? gp.dt_bias[h * 128 + c0 + 1] : 0.f;
      float2 xs[16];
#pragma unroll
      for (int ii = 0; ii < 16; ++ii) {
        const int r = 16 * R + ii;
        xs[ii] = r < len ? ldg_stream(reinterpret_cast<const float2 *>(xg_in + base_h + r * rowH + c0))
                         : make_float2(0.f, 0.f);
      }
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int ii = 0; ii < 16; ++ii) {
        const int r = 16 * R + ii;
        float g0, g1;
        if (gate) {
          // softplus(z) log2 e = max(z, 0) log2 e + log2(1 + 2^{-|z| log2 e})
          const float z0 = (xs[ii].x + db0) * kLog2e, z1 = (xs[ii].y + db1) * kLog2e;
          g0 = -A_h * (fmaxf(z0, 0.f) + tc::lg2(1.f + tc::ex2(-fabsf(z0))));
          g1 = -A_h * (fmaxf(z1, 0.f) + tc::lg2(1.f + tc::ex2(-fabsf(z1))));
        } else {
          g0 = xs[ii].x * kLog2e;
          g1 = xs[ii].y * kLog2e;
        }
        if (r >= len) g0 = g1 = 0.f;
        acc0 += g0;
        acc1 += g1;
        Gl[ii][0] = acc0;
        Gl[ii][1] = acc1;
      }
      *reinterpret_cast<float2 *>(tot + R * 128 + c0) = make_float2(acc0, acc1);
    }
    // the staging buffers of the previous item must be read out before this
    // item's operand tiles overwrite them
    if (tid == 0) bulk_wait_read();
    __syncthreads();  // sub-block totals, rstd and beta published

    // ---- phase 2: operand tiles and the elementwise package parts
    {
      float bAll[4][2], GC[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float a = 0.f;
#pragma unroll
        for (int RR = 0; RR < 4; ++RR) {
          bAll[RR][j] = a;
          a += tot[RR * 128 + c0 + j];
        }
        GC[j] = a;
      }
      float bR[2], eb[2], egc[2], cR[4][2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        bR[j] = bAll[0][j];
#pragma unroll
        for (int RR = 1; RR < 4; ++RR)
          if (RR == R) bR[j] = bAll[RR][j];
        eb[j] = tc::ex2(bR[j]);
        egc[j] = tc::ex2(GC[j] - bR[j]);
#pragma unroll
        for (int RR = 0; RR < 4; ++RR) cR[RR][j] = tc::ex2(fminf(bAll[RR][j] - bR[j], 0.f));
      }
      if (R == 0)
        *reinterpret_cast<float2 *>(pk + PK_GC + c0 * 4) = make_float2(tc::ex2(GC[0]), tc::ex2(GC[1]));
      const float sc0 = gp.scale * eb[0], sc1 = gp.scale * eb[1];
      const uint32_t kp128 = pan * 128u * 128u, kp160 = pan * B1_PANEL, kp64 = pan * 64u * 128u;
      uint32_t qraw8[8], kraw8[8];
#pragma unroll
      for (int ii = 0; ii < 16; ++ii) {
        const int r = 16 * R + ii;
        if ((ii & 7) == 0) {
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int rj = r + jj;
            qraw8[jj] = 0;
            kraw8[jj] = 0;
            if (rj < len) {
              qraw8[jj] = ldg_stream(reinterpret_cast<const uint32_t *>(qg_in + base_h + rj * rowH + c0));
              kraw8[jj] = ldg_stream(reinterpret_cast<const uint32_t *>(kg_in + base_h + rj * rowH + c0));
            }
          }
        }
        const uint32_t qraw = qraw8[ii & 7], kraw = kraw8[ii & 7];
        const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qraw));
        const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kraw));
        const uint32_t xo = ((ch16 ^ (uint32_t)(ii & 7)) << 4) | cbyte;
        const float sq = rq[r], sk = rk[r];
        const float e0 = tc::ex2(Gl[ii][0]), e1 = tc::ex2(Gl[ii][1]);
        const float f0 = tc::ex2(fminf(-Gl[ii][0], 126.f)), f1 = tc::ex2(fminf(-Gl[ii][1], 126.f));
        const float kn0 = kf.x * sk, kn1 = kf.y * sk;
        const float qn0 = qf.x * sq, qn1 = qf.y * sq;
        const float ke0 = kn0 * e0, ke1 = kn1 * e1;
        const float kf0 = kn0 * f0, kf1 = kn1 * f1;
        const float qe0 = qn0 * e0, qe1 = qn1 * e1;
        const uint32_t rowb = (uint32_t)r * 128u + xo;
        st_u32(sm + S_OPA, kp128 + rowb, pack_bf16(ke0, ke1));
        st_u32(sm + S_OPA, kp128 + 64u * 128u + rowb, pack_bf16(qe0, qe1));
        st_u32(sm + S_B1, kp160 + 96u * 128u + rowb, pack_bf16(kf0, kf1));
#pragma unroll
        for (int Rp = 1; Rp < 4; ++Rp)
          if (Rp > R)
            st_u32(sm + S_B1, kp160 + (uint32_t)b1_off(Rp) * 128u + rowb,
                   pack_bf16(kf0 * cR[Rp][0], kf1 * cR[Rp][1]));
        st_u32(sm + S_B2A, kp64 + rowb, pack_bf16(ke0 * eb[0], ke1 * eb[1]));
        // package: qg = scale q^ 2^G (WQ rows 0..63), kg = k^ 2^{G_C - G} (KG)
        st_u32(pk, PK_WQ + kp128 + rowb, pack_bf16(qe0 * sc0, qe1 * sc1));
        st_u32(pk, PK_KG + kp64 + rowb, pack_bf16(kf0 * egc[0], kf1 * egc[1]));
      }
    }
    tc::fence_proxy_async_smem();
    __syncthreads();

    // ---- MMA 1: [kE; qE] x B1^T -> D1 (128 x 160)
    if (tid == 0) {
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(128, 160, false, false);
      const uint32_t a0 = tc::smem_u32(sm + S_OPA), b0 = tc::smem_u32(sm + S_B1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t ad = tc::smem_desc_sw128(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = tc::smem_desc_sw128(b0 + (kk >> 2) * B1_PANEL + (kk & 3) * 32, 16, 1024);
        tc::mma_bf16(tmem, ad, bd, idesc, kk > 0);
      }
      tc::mma_commit(bar_mma);
      mma_pending = true;
    }
    __syncwarp();
    bool ok = wait_or_flag(bar_mma, mma_phase, err);
    if (ok) { mma_pending = false; mma_phase ^= 1; }
    else *abort_flag = 1;
    tc::tc_fence_after();
    __syncthreads();
    if (*abort_flag) break;

    // ---- read D1: L (k rows) to shared fp32, Aqk (q rows) to the package;
    //      zero the inverse buffer
    {
      float *AF = reinterpret_cast<float *>(sm + S_AF);
      for (int x = tid; x < 64 * 65; x += NT) AF[x] = 0.f;
      const int q4 = warp & 3, cq = warp >> 2;
      const int m = 32 * q4 + lane;          // D1 row = TMEM lane
      const bool krow = m < 64;
      const int r = krow ? m : m - 64;
      const int Rr = r >> 4;
      float *LF = reinterpret_cast<float *>(sm + S_LF);
      const float br = sbeta[r];
      uint8_t *saqk = sm + S_STG_AQK;
      if (!krow && cq == 0) {
        // Aqk groups above the diagonal block are zero
        for (int gi = Rr + 1; gi < 4; ++gi) {
          const uint4 z = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(saqk + kmaj_off(64, r, 16 * gi)) = z;
          *reinterpret_cast<uint4 *>(saqk + kmaj_off(64, r, 16 * gi + 8)) = z;
        }
      }
      // column blocks of D1 this warp reads: rows 0..31 (sub-blocks 0, 1)
      // need blocks 0, 6, 7; rows 32..63 (sub-blocks 2, 3) need 1..5, 8, 9
      int chs[4] = {-1, -1, -1, -1};
      if ((q4 & 1) == 0) {
        if (cq == 0) { chs[0] = 0; chs[1] = 7; } else { chs[0] = 6; }
      } else {
        if (cq == 0) { chs[0] = 1; chs[1] = 2; chs[2] = 3; chs[3] = 8; }
        else { chs[0] = 4; chs[1] = 5; chs[2] = 9; }
      }
#pragma unroll
      for (int bt = 0; bt < 2; ++bt) {
      float d[2][16];
      __syncwarp();
#pragma unroll
      for (int cx = 0; cx < 2; ++cx)
        if (chs[2 * bt + cx] >= 0)
          tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + 16 * chs[2 * bt + cx], d[cx]);
      tc::tmem_ld_wait();
#pragma unroll
      for (int cx = 0; cx < 2; ++cx) {
        const int cix = cx;
        const int ch = chs[2 * bt + cx];
        // which 16 tokens j0.. this column block holds for a row of block Rr
        int j0 = -1;
        bool diag = false;
        if (ch == 0 && Rr == 1) j0 = 0;
        else if ((ch == 1 || ch == 2) && Rr == 2) j0 = 16 * (ch - 1);
        else if (ch >= 3 && ch <= 5 && Rr == 3) j0 = 16 * (ch - 3);
        else if (ch >= 6 && ch - 6 == Rr) { j0 = 16 * Rr; diag = true; }
        if (j0 < 0) continue;
        if (krow) {
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const int j = j0 + x;
            if (!diag || j < r) LF[r * LFS + j] = br * d[cix][x];
          }
        } else {
          uint32_t pkd[8];
#pragma unroll
          for (int x = 0; x < 16; x += 2) {
            const int j = j0 + x;
            const float a0 = (!diag || j <= r) ? gp.scale * d[cix][x] : 0.f;
            const float a1 = (!diag || j + 1 <= r) ? gp.scale * d[cix][x + 1] : 0.f;
            pkd[x / 2] = pack_bf16(a0, a1);
          }
          *reinterpret_cast<uint4 *>(saqk + kmaj_off(64, r, j0)) =
              make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
          *reinterpret_cast<uint4 *>(saqk + kmaj_off(64, r, j0 + 8)) =
              make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
        }
      }
      }
    }
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store(pk + PK_AQK, sm + S_STG_AQK, 8192);
      bulk_commit();
    }

    // ---- (I + L)^-1 in fp32
    {
      const float *LF = reinterpret_cast<const float *>(sm + S_LF);
      float *AF = reinterpret_cast<float *>(sm + S_AF);
      float *TT = reinterpret_cast<float *>(sm + S_TT);
      // (1) the four 16 x 16 diagonal blocks X_I = (I + L_II)^-1 by forward
      //     substitution: four lanes per column, lane `part` owns rows
      //     part, part + 4, part + 8, part + 12 and the finished entry of
      //     each step is broadcast inside the 4-lane group.
      {
        const int col = tid >> 2, part = tid & 3;
        const int base = 16 * (col >> 4), jj = col & 15;
        float x[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) x[a] = (part + 4 * a == jj) ? 1.f : 0.f;
#pragma unroll
        for (int mm = 0; mm < 15; ++mm) {
          const float xm = __shfl_sync(0xffffffffu, x[mm >> 2], (tid & ~3) | (mm & 3));
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const int ii = part + 4 * a;
            if (ii > mm) x[a] = fmaf(-LF[(base + ii) * LFS + base + mm], xm, x[a]);
          }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) AF[(base + part + 4 * a) * 65 + base + jj] = x[a];
      }
      __syncthreads();
      // (2) 32 x 32 diagonal halves: X_10 = -X_1 L_10 X_0, X_32 = -X_3 L_32 X_2
      //     (two outputs per thread: both halves)
      {
        const int ii = tid >> 4, jj = tid & 15;
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const int rI = 32 * pr + 16, cJ = 32 * pr;
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int m = 0; m < 16; m += 2) {
            a0 = fmaf(LF[(rI + ii) * LFS + cJ + m], AF[(cJ + m) * 65 + cJ + jj], a0);
            a1 = fmaf(LF[(rI + ii) * LFS + cJ + m + 1], AF[(cJ + m + 1) * 65 + cJ + jj], a1);
          }
          TT[(16 * pr + ii) * 33 + jj] = a0 + a1;
        }
        __syncthreads();
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const int rI = 32 * pr + 16, cJ = 32 * pr;
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int m = 0; m < 16; m += 2) {
            a0 = fmaf(AF[(rI + ii) * 65 + rI + m], TT[(16 * pr + m) * 33 + jj], a0);
            a1 = fmaf(AF[(rI + ii) * 65 + rI + m + 1], TT[(16 * pr + m + 1) * 33 + jj], a1);
          }
          AF[(rI + ii) * 65 + cJ + jj] = -(a0 + a1);
        }
      }
      __syncthreads();
      // (3) lower-left 32 x 32 block: A_21 = -A_2 (L_21 A_1)  (4 outputs per thread)
      {
        const int ii = tid >> 3, jj = tid & 7;  // rows 0..31, columns jj + 8 c
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          const float l = LF[(32 + ii) * LFS + m];
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[c] = fmaf(l, AF[m * 65 + jj + 8 * c], acc[c]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) TT[ii * 33 + jj + 8 * c] = acc[c];
        __syncthreads();
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = 0.f;
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          const float xv = AF[(32 + ii) * 65 + 32 + m];
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[c] = fmaf(xv, TT[m * 33 + jj + 8 * c], acc[c]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) AF[(32 + ii) * 65 + jj + 8 * c] = -acc[c];
      }
      __syncthreads();
      // A . diag(beta) -> bf16 K-major tile (two 8-column groups per thread)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = (tid >> 3) + 32 * hh, g = tid & 7;
        uint32_t pkd[4];
#pragma unroll
        for (int x = 0; x < 8; x += 2) {
          const int jj = 8 * g + x;
          const float a0 = (jj <= r) ? AF[r * 65 + jj] * sbeta[jj] : 0.f;
          const float a1 = (jj + 1 <= r) ? AF[r * 65 + jj + 1] * sbeta[jj + 1] : 0.f;
          pkd[x / 2] = pack_bf16(a0, a1);
        }
        *reinterpret_cast<uint4 *>(sm + S_AINV + kmaj_off(64, r, 8 * g)) =
            make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
      }
    }
    tc::fence_proxy_async_smem();
    // v of this item must have landed before the second MMA reads it
    ok = wait_or_flag(bar_v, (uint32_t)(i & 1), err);
    if (ok) v_done = i + 1;
    else *abort_flag = 1;
    __syncthreads();
    if (*abort_flag) break;

    // ---- MMA 2: w = A' (k^ 2^G) -> cols 0..127, u = A' v -> cols 128..255 (M = 64)
    if (tid == 0) {
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(64, 128, false, true);
      const uint32_t a0 = tc::smem_u32(sm + S_AINV);
      const uint32_t bw = tc::smem_u32(sm + S_B2A), bu = tc::smem_u32(sm + S_V);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = tc::smem_desc_sw128(a0 + kk * 32, 16, 1024);
        tc::mma_bf16(tmem, ad, tc::smem_desc_sw128(bw + kk * 2048, 8192, 1024), idesc, kk > 0);
        tc::mma_bf16(tmem + 128, ad, tc::smem_desc_sw128(bu + kk * 2048, 8192, 1024), idesc, kk > 0);
      }
      tc::mma_commit(bar_mma);
      mma_pending = true;
    }
    __syncwarp();
    ok = wait_or_flag(bar_mma, mma_phase, err);
    if (ok) { mma_pending = false; mma_phase ^= 1; }
    else *abort_flag = 1;
    tc::tc_fence_after();
    __syncthreads();
    if (*abort_flag) break;

    // v is free: fetch the next item's v
    if (tid == 0 && okn) {
      issue_v(maps, sm + S_V, bar_v, nx);
      ++v_issued;
    }

    // ---- read D2 (M = 64 layout: row r in lane (r % 16) + 32 (r / 16)):
    //      w -> package WQ rows 64..127, u -> package U
    {
      const int q4 = warp & 3;
      const bool is_u = warp >= 4;
      const int r = 16 * q4 + lane;  // valid for lane < 16
#pragma unroll
      for (int half = 0; half < 4; ++half) {
        float d[2][16];
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
          tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (is_u ? 128 : 0) + 32 * half + 16 * cc,
                        d[cc]);
        tc::tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int col = 32 * half + 16 * cc;  // column inside w or u
            if (!is_u) {
              uint32_t pkd[8];
#pragma unroll
              for (int x = 0; x < 16; x += 2) pkd[x / 2] = pack_bf16(d[cc][x], d[cc][x + 1]);
              // rows 64.. of WQ, panel by panel: same swizzle phase (row % 8)
              *reinterpret_cast<uint4 *>(sm + S_STG_W + kmaj_off(64, r, col)) =
                  make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
              *reinterpret_cast<uint4 *>(sm + S_STG_W + kmaj_off(64, r, col + 8)) =
                  make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
            } else {
#pragma unroll
              for (int x = 0; x < 16; x += 4)
                *reinterpret_cast<float4 *>(sm + S_STG_U + u_offset(r, col + x)) =
                    make_float4(d[cc][x], d[cc][x + 1], d[cc][x + 2], d[cc][x + 3]);
            }
          }
        }
      }
    }
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store(pk + PK_WQ + 64 * 128, sm + S_STG_W, 8192);
      bulk_store(pk + PK_WQ + 16384 + 64 * 128, sm + S_STG_W + 8192, 8192);
      bulk_store(pk + PK_U, sm + S_STG_U, 32768);
      bulk_commit();
    }
  }

  // Drain after a timeout: wait (bounded) for the load and the MMA this CTA
  // started, so that nothing lands in memory it no longer owns.  On the
  // normal path every issued load has been consumed.
  __syncthreads();
  if (tid == 0) {
    bulk_wait_all();  // package stores complete before the CTA exits
    if (*abort_flag) {
      if (mma_pending) drain_wait(bar_mma, mma_phase);
      for (int64_t x = v_done; x < v_issued; ++x) drain_wait(bar_v, (uint32_t)(x & 1));
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_tc_prep(const TcMaps &maps, const void *q, const void *k, const float *x,
                           const float *beta, const GateParams &gp, const SeqInfo &s,
                           int64_t nchunks, int H, char *pkg, uint32_t *err, cudaStream_t st) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  cudaError_t e = cudaFuncSetAttribute(tc_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t nitems = nchunks * H;
  if (nitems == 0) return cudaSuccess;
  const int64_t slots = 2 * (int64_t)sms;
  const int grid = (int)(nitems < slots ? nitems : slots);
  tc_prep_kernel<<<grid, NT, SMEM_BYTES, st>>>(maps, static_cast<const __nv_bfloat16 *>(q),
                                              static_cast<const __nv_bfloat16 *>(k), x, beta, gp, s,
                                              nitems, H, pkg, err);
  return cudaGetLastError();
}

}  // namespace tcp
}  // namespace kda
