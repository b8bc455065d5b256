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
// reference, 2^{b_R(j) - G_j} (diagonal blocks, bounded by the decay of the
// block's own 16 tokens).  Where some channel's gate moves by more than
// STRONG_DECAY_LOG2 inside one sub-block, the affected threads rewrite their
// off-diagonal column factors and kg from exact exponents, and the four
// diagonal 16 x 16 blocks of L and A_qk are recomputed from exact gate
// differences on the CUDA cores (every off-diagonal product has both factors
// <= 1, so it stays exact up to terms below 2^-126); the item is listed for
// the backward, which does the same for its own factored products.  For every
// other item all factors lie inside [2^-96, 2^96].  One M=128 x N=160 x K=128
// tcgen05 MMA then yields every needed block of both A_kk and A_qk:
//   A rows  0..63 : k^_r 2^{G_r - b_R}      A rows 64..127: q^_r 2^{G_r - b_R}
//   B rows  0..15 : k^_j 2^{b_1 - G_j}, j < 16
//   B rows 16..47 : k^_j 2^{b_2 - G_j}, j < 32
//   B rows 48..95 : k^_j 2^{b_3 - G_j}, j < 48
//   B rows 96..159: k^_j 2^{b_R(j) - G_j}, j < 64 (own block)
//
// Two persistent CTAs per SM loop over (chunk, head) items.  Once an item's
// second MMA has finished, cp.async brings the next item's q, k and gate input
// into shared memory while the current one reads out w and u; the item's v
// arrives by TMA during its own operand build.
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
constexpr int LFS = 68;              // row stride of L and A (16-byte aligned rows)
constexpr int TTS = 36;              // row stride of the product scratch
constexpr uint32_t S_AF = 16384;     // fp32 A [64][68]
constexpr uint32_t S_LF = 33792;     // fp32 L [64][68]
constexpr uint32_t S_TT = 51200;     // fp32 scratch [32][36]
// A' = A.diag(beta) stacked twice, [A'; A'] (K-major, 128 rows, 16384): the
// A operand of both second-stage MMAs; written after the inverse, over L
constexpr uint32_t S_AINV = 33792;
// staging of package parts for bulk stores (regions free at that time):
constexpr uint32_t S_STG_AQK = 73728;  // Aqk image (8192), written after MMA 1 (B1 dead)
// strong decay, between the D1 readout and the inverse: one sub-block's raw
// q, k (bf16) and chunk-local gate (fp32), 16 rows x 128 channels (B1 dead)
constexpr uint32_t S_FIX = 56320;      // G [16][128] fp32, then q, k [16][128] bf16 (ends at 72704)
constexpr uint32_t S_STG_W = 90112;    // w rows of WQ, 2 panels x 8192, after MMA 2 (B2A dead)
constexpr uint32_t S_STG_U = 49152;    // U image (16384), after MMA 2 (B1 dead)
// OPA holds nothing between items: the next item's raw q and k rows land there,
// at the positions phase 2 overwrites with the scaled operands.
constexpr uint32_t S_MISC = 106496;
constexpr uint32_t M_RQ = S_MISC;           // fp32 [64] scale x rstd q
constexpr uint32_t M_RK = S_MISC + 256;     // fp32 [64] rstd k
constexpr uint32_t M_BETA = S_MISC + 512;   // fp32 [64]
constexpr uint32_t M_TOT = S_MISC + 768;    // fp32 [8][128] row-group gate totals
constexpr uint32_t M_BAR = S_MISC + 4864;   // bar_v, bar_mma
constexpr uint32_t M_TSLOT = S_MISC + 4880;
constexpr uint32_t M_ABORT = S_MISC + 4884;
constexpr uint32_t M_STRONG = S_MISC + 4888;  // some warp saw strong decay in this item
constexpr uint32_t M_ITEM = S_MISC + 4896;  // 2 x ItemSlot
constexpr uint32_t SMEM_BYTES = S_MISC + 4960 + 1024;

constexpr uint32_t B1_PANEL = 160 * 128;
constexpr uint32_t TMEM_COLS = 256;

__device__ __forceinline__ int b1_off(int Rp) { return 8 * Rp * (Rp - 1); }  // 0, 16, 48

// Rows of the first MMA's A operand (= TMEM lanes of D1) hold the 16-token
// blocks in the order 0, 3, 1, 2, so that each 32-lane quarter holds one
// block with few and one with many D1 column blocks to read.
__device__ __forceinline__ int lane_block(int Rt) { return (0x1320 >> (4 * Rt)) & 3; }   // 0,2,3,1
__device__ __forceinline__ int token_block(int Lb) { return (0x2130 >> (4 * Lb)) & 3; }  // 0,3,1,2

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

__device__ __forceinline__ void put_slot(ItemSlot &sl, const Item &it, bool ok) {
  sl.t0 = it.t0;
  sl.gc = it.gc;
  sl.len = it.len;
  sl.h = it.h;
  sl.ok = ok ? 1 : 0;
}

__device__ __forceinline__ void st_u64(uint8_t *base, uint32_t off, uint2 v) {
  *reinterpret_cast<uint2 *>(base + off) = v;
}

__device__ __forceinline__ uint2 pack4(float a, float b, float c, float d) {
  return make_uint2(pack_bf16(a, b), pack_bf16(c, d));
}
__device__ __forceinline__ uint2 pack4(float2 a, float2 b) {
  return make_uint2(pack_bf16(a.x, a.y), pack_bf16(b.x, b.y));
}

// fp32 x rounded to tf32 (to nearest), as the bits an MMA operand takes.
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// d += a b for one m16n8k8 tf32 tile (warp-level MMA, fp32 accumulate).
__device__ __forceinline__ void mma_m16n8k8_tf32(float (&d)[4], const uint32_t (&a)[4],
                                                 const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc += X[0:16, 0:KK] Y[0:KK, 0:8] for one warp (X, Y fp32 in shared
// memory, row strides ldx, ldy; g = lane / 4, t = lane % 4), as m16n8k8
// tf32 MMAs with fp32 accumulation; acc holds rows g, g + 8 and columns
// 2 t, 2 t + 1 of the 16 x 8 result.  The operands are rounded to tf32
// (relative 2^-11), finer than the bf16 (2^-9) in which the inverse leaves
// for the second MMA.
template <int KK>
__device__ __forceinline__ void warp_mm_tf32(const float *X, int ldx, const float *Y, int ldy, int g,
                                             int t, float (&acc)[4]) {
#pragma unroll
  for (int k0 = 0; k0 < KK; k0 += 8) {
    uint32_t a[4], b[2];
    a[0] = to_tf32(X[g * ldx + k0 + t]);
    a[1] = to_tf32(X[(g + 8) * ldx + k0 + t]);
    a[2] = to_tf32(X[g * ldx + k0 + t + 4]);
    a[3] = to_tf32(X[(g + 8) * ldx + k0 + t + 4]);
    b[0] = to_tf32(Y[(k0 + t) * ldy + g]);
    b[1] = to_tf32(Y[(k0 + t + 4) * ldy + g]);
    mma_m16n8k8_tf32(acc, a, b);
  }
}

// Barrier over the 128 threads of one half of the CTA (ids 1, 2).
__device__ __forceinline__ void half_sync(int half) {
  asm volatile("bar.sync %0, 128;" :: "r"(1 + half) : "memory");
}

// L2 policy for data touched once - the inputs after their one read, the
// package (read back only after the whole pass): evicted first, so that it
// does not push the next items' prefetched inputs out of L2.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint2 ldg_u2_hint(const void *p, uint64_t pol) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
               : "=r"(v.x), "=r"(v.y) : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ float4 ldg_f4_hint(const void *p, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ void stg_hint(uint8_t *base, uint32_t off, uint2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.b32 [%0], {%1, %2}, %3;"
               :: "l"(base + off), "r"(v.x), "r"(v.y), "l"(pol) : "memory");
}
__device__ __forceinline__ void bulk_store_hint(void *dst, const void *src, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
               :: "l"(reinterpret_cast<uint64_t>(dst)), "r"(tc::smem_u32(src)), "r"(bytes), "l"(pol)
               : "memory");
}

// Asynchronous global -> shared copies of 8 and 16 bytes (no registers held
// while they are in flight); a row that is not valid copies nothing and reads
// as zero (src-size 0; the source address is then not dereferenced, and a
// valid one is passed anyway).
__device__ __forceinline__ void cp_async8(uint8_t *dst, const void *src, bool valid, uint64_t pol) {
  asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 8, %2, %3;"
               :: "r"(tc::smem_u32(dst)), "l"(src), "r"(valid ? 8 : 0), "l"(pol) : "memory");
}
__device__ __forceinline__ void cp_async16(uint8_t *dst, const void *src, bool valid, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;"
               :: "r"(tc::smem_u32(dst)), "l"(src), "r"(valid ? 16 : 0), "l"(pol) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Where a thread's gate-input row rr (16 bytes, fp32 channels c0 .. c0 + 3)
// waits for phase 1: rows 0..5 in the B1 region from S_XIN (dead from the
// second MMA of the item before until the operand build), rows 6, 7 in the
// first v panel (the item's v is requested only after phase 1).  Consecutive
// threads take consecutive 16-byte slots.
constexpr uint32_t S_XIN = 65536;
__device__ __forceinline__ uint32_t x_slot(int rr, int tid) {
  return rr < 6 ? S_XIN + (uint32_t)(rr * NT + tid) * 16u : S_V + (uint32_t)((rr - 6) * NT + tid) * 16u;
}

// Strong decay, per thread: its channels decay past the factored range
// inside their sub-block, so the column factor k^ 2^{b_R - G} may be clamped;
// its off-diagonal copies k^ 2^{b_R' - G} (B1) and kg = k^ 2^{G_C - G} (the
// package), both <= 1, are rewritten from exact exponents.  k and the gate
// input come again from global memory (OPA holds the scaled operand by now).
// Out of line, so that the common path's registers do not carry it.
__device__ __noinline__ void strong_factors_exact(uint8_t *sm, uint8_t *pk, const __nv_bfloat16 *kg_in,
                                                  const float *xg_in, const GateParams &gp, int h, int len,
                                                  int64_t base_h, int64_t base_k, int64_t rowH, int64_t rowHk,
                                                  uint32_t kp160, uint32_t kp64, uint64_t pol_once,
                                                  uint64_t pol_qk) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float *tot = reinterpret_cast<const float *>(sm + M_TOT);
  const float *rk = reinterpret_cast<const float *>(sm + M_RK);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c0 = 4 * lane, R = warp >> 1;
  const uint32_t ch16 = (uint32_t)((lane & 15) >> 1), cbyte = (uint32_t)(lane & 1) * 8u;
  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;
  float dl[4][4], dg[4], acc[4];
  {
    float a[4] = {0.f, 0.f, 0.f, 0.f}, bA[4][4];
#pragma unroll
    for (int gg = 0; gg < 8; ++gg) {
      const float4 t = *reinterpret_cast<const float4 *>(tot + gg * 128 + c0);
      const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if ((gg & 1) == 0) bA[gg >> 1][j] = a[j];
        if (gg == (warp | 1) - 1) acc[j] = (warp & 1) ? tv[j] : 0.f;  // gate before this group
        a[j] += tv[j];
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float bl = bA[0][j];
#pragma unroll
      for (int RR = 1; RR < 4; ++RR)
        if (RR == R) bl = bA[RR][j];
#pragma unroll
      for (int RR = 1; RR < 4; ++RR) dl[RR][j] = bA[RR][j] - bl;
      dg[j] = a[j] - bl;
    }
  }
  const float A_h = gate ? tc::ex2(gp.a_log[h] * kLog2e) : 0.f;
  float dbl[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    dbl[j] = (gate && gp.dt_bias) ? gp.dt_bias[h * gp.dk + c0 + j] * kLog2e : 0.f;  // c0 < dk here
#pragma unroll 1
  for (int rr = 0; rr < 8; ++rr) {
    const int r = 8 * warp + rr;
    const uint32_t rowb = (uint32_t)r * 128u + (((ch16 ^ (uint32_t)rr) << 4) | cbyte);
    float kn[4] = {0.f, 0.f, 0.f, 0.f}, xv[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < len) {
      const uint2 kraw = ldg_u2_hint(kg_in + base_k + r * rowHk + c0, pol_qk);
      const float4 x4 = ldg_f4_hint(xg_in + base_h + r * rowH + c0, pol_once);
      const float2 ka = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kraw.x));
      const float2 kb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kraw.y));
      const float sk = rk[r];
      kn[0] = ka.x * sk; kn[1] = ka.y * sk; kn[2] = kb.x * sk; kn[3] = kb.y * sk;
      xv[0] = x4.x; xv[1] = x4.y; xv[2] = x4.z; xv[3] = x4.w;
    }
    float G[4], x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // the gate as in phase 1, chunk-local from the sub-block start
      float g;
      if (gate) {
        const float z = fmaf(xv[j], kLog2e, dbl[j]);
        g = -A_h * (fmaxf(z, 0.f) + tc::lg2(1.f + tc::ex2(-fabsf(z))));
      } else {
        g = xv[j] * kLog2e;
      }
      acc[j] += r < len ? g : 0.f;
      G[j] = acc[j];
    }
#pragma unroll
    for (int Rp = 1; Rp < 4; ++Rp)
      if (Rp > R) {
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = kn[j] * tc::ex2(dl[Rp][j] - G[j]);
        st_u64(sm + S_B1, kp160 + (uint32_t)b1_off(Rp) * 128u + rowb, pack4(x[0], x[1], x[2], x[3]));
      }
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = kn[j] * tc::ex2(dg[j] - G[j]);
    stg_hint(pk, PK_KG + kp64 + rowb, pack4(x[0], x[1], x[2], x[3]), pol_once);
  }
}

// Strong decay: the four 16 x 16 diagonal blocks of L and A_qk of the item
// again, from exponentials of exact gate differences (every factor <= 1):
//   L_rj = beta_r sum_c k^_rc k^_jc 2^{G_rc - G_jc} (j < r),
//   Aqk_rj = scale sum_c q^_rc k^_jc 2^{G_rc - G_jc} (j <= r),
// over the item's fp32 L (LFS-strided) and its bf16 A_qk image.  Per
// sub-block the 256 threads load its 16 rows (raw q, k and the gate, the
// gate summed from the sub-block start); warp w then takes rows 2w, 2w + 1,
// a lane four channels, and a reduce-scatter over the warp's lanes leaves the
// 32 sums of a row (16 of L, 16 of A_qk) one per lane.
__device__ __noinline__ void diagonal_blocks_exact(uint8_t *sm, const __nv_bfloat16 *qg_in,
                                                   const __nv_bfloat16 *kg_in, const float *xg_in,
                                                   const GateParams &gp, int h, int len, int64_t base_h,
                                                   int64_t base_k, int64_t rowH, int64_t rowHk) {
  constexpr float kLog2e = 1.4426950408889634f;
  float *FG = reinterpret_cast<float *>(sm + S_FIX);
  __nv_bfloat16 *FQ = reinterpret_cast<__nv_bfloat16 *>(sm + S_FIX + 8192);
  __nv_bfloat16 *FK = FQ + 16 * 128;
  float *LF = reinterpret_cast<float *>(sm + S_LF);
  const float *rq = reinterpret_cast<const float *>(sm + M_RQ);
  const float *rk = reinterpret_cast<const float *>(sm + M_RK);
  const float *sbeta = reinterpret_cast<const float *>(sm + M_BETA);
  uint8_t *saqk = sm + S_STG_AQK;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;
#pragma unroll 1
  for (int Rb = 0; Rb < 4; ++Rb) {
    if (tid < 128) {  // thread = channel; the sub-block's 16 rows in order
      const int c = tid;
      const float A_h = gate ? tc::ex2(gp.a_log[h] * kLog2e) : 0.f;
      const bool cin = c < gp.dk;  // channels past a narrow head: zero q, k and gate
      const float dbc = (gate && gp.dt_bias && cin) ? gp.dt_bias[h * gp.dk + c] * kLog2e : 0.f;
      float acc = 0.f;
#pragma unroll 1
      for (int rl = 0; rl < 16; ++rl) {
        const int r = 16 * Rb + rl;
        __nv_bfloat16 qv = __float2bfloat16_rn(0.f), kv = qv;
        float g = 0.f;
        if (r < len && cin) {
          qv = qg_in[base_k + r * rowHk + c];
          kv = kg_in[base_k + r * rowHk + c];
          const float x = xg_in[base_h + r * rowH + c];
          if (gate) {
            const float z = fmaf(x, kLog2e, dbc);
            g = -A_h * (fmaxf(z, 0.f) + tc::lg2(1.f + tc::ex2(-fabsf(z))));
          } else {
            g = x * kLog2e;
          }
        }
        acc += g;
        FG[rl * 128 + c] = acc;
        FQ[rl * 128 + c] = qv;
        FK[rl * 128 + c] = kv;
      }
    }
    __syncthreads();
#pragma unroll 1
    for (int sub = 0; sub < 2; ++sub) {
      const int rl = 2 * warp + sub, r = 16 * Rb + rl;
      const int c4 = 4 * lane;
      float qh[4], kh[4], Gr[4];
      {
        const float qs = rq[r], ks = rk[r];
        const uint2 qq = *reinterpret_cast<const uint2 *>(FQ + rl * 128 + c4);
        const uint2 kk = *reinterpret_cast<const uint2 *>(FK + rl * 128 + c4);
        const float2 q0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qq.x));
        const float2 q1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qq.y));
        const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kk.x));
        const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kk.y));
        qh[0] = q0.x * qs; qh[1] = q0.y * qs; qh[2] = q1.x * qs; qh[3] = q1.y * qs;
        kh[0] = k0.x * ks; kh[1] = k0.y * ks; kh[2] = k1.x * ks; kh[3] = k1.y * ks;
        const float4 g4 = *reinterpret_cast<const float4 *>(FG + rl * 128 + c4);
        Gr[0] = g4.x; Gr[1] = g4.y; Gr[2] = g4.z; Gr[3] = g4.w;
      }
      float v[32];  // v[j]: L sum with token j, v[16 + j]: A_qk sum
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        v[j] = 0.f;
        v[16 + j] = 0.f;
        if (j <= rl) {  // uniform over the warp
          const float kjs = rk[16 * Rb + j];
          const uint2 kk = *reinterpret_cast<const uint2 *>(FK + j * 128 + c4);
          const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kk.x));
          const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kk.y));
          const float4 g4 = *reinterpret_cast<const float4 *>(FG + j * 128 + c4);
          const float kj[4] = {k0.x * kjs, k0.y * kjs, k1.x * kjs, k1.y * kjs};
          const float Gj[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const float t = kj[x] * tc::ex2(Gr[x] - Gj[x]);
            v[j] = fmaf(kh[x], t, v[j]);
            v[16 + j] = fmaf(qh[x], t, v[16 + j]);
          }
        }
      }
      // reduce-scatter: after step s the lane keeps the half of its values
      // selected by lane bit 4 - s; lane l ends with the total of value l
#pragma unroll
      for (int st = 0; st < 5; ++st) {
        const int half = 16 >> st;
        const bool up = (lane & half) != 0;
#pragma unroll
        for (int i2 = 0; i2 < half; ++i2) {
          const float send = up ? v[i2] : v[i2 + half];
          const float keep = up ? v[i2 + half] : v[i2];
          v[i2] = keep + __shfl_xor_sync(0xffffffffu, send, half);
        }
      }
      const int j = lane & 15;
      if (lane < 16) {
        LF[r * LFS + 16 * Rb + j] = j < rl ? sbeta[r] * v[0] : 0.f;
      } else {
        *reinterpret_cast<__nv_bfloat16 *>(saqk + kmaj_off(64, r, 16 * Rb + j)) =
            __float2bfloat16_rn(j <= rl ? v[0] : 0.f);
      }
    }
    __syncthreads();
  }
}

// Phase-1 inputs of one item, copied asynchronously into shared memory: this
// thread's 8 rows x 4 channels of q and k go straight to the positions of
// the operand tile that phase 2 reads them from (raw bf16), the gate input
// to the thread's x slots.  Rows past the item's end and channels past a
// narrow head read as zero.  Only the issuing thread reads these copies
// back, after its own wait.
template <bool GROUPED>
__device__ __forceinline__ void stage_rows(uint8_t *sm, const ItemSlot &it, const __nv_bfloat16 *qg_in,
                                           const __nv_bfloat16 *kg_in, const float *xg_in, int dk,
                                           int64_t rowH, int64_t rowHk, int grp, int warp, int c0, bool cin,
                                           int tid, uint32_t kp128, int prow0, uint32_t ch16, uint32_t cbyte,
                                           uint64_t pol_qk, uint64_t pol_once) {
  const int len = it.len, h = it.h;
  const int64_t base_h = it.t0 * rowH + (int64_t)h * dk;
  const int64_t base_k = it.t0 * rowHk + (int64_t)(GROUPED ? h / grp : h) * dk;
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int r = 8 * warp + rr;
    const bool ok = r < len && cin;
    const int64_t off = ok ? base_h + r * rowH + c0 : 0;
    const int64_t offk = GROUPED ? (ok ? base_k + r * rowHk + c0 : 0) : off;
    const uint32_t orow = (uint32_t)(prow0 + rr) * 128u + (((ch16 ^ (uint32_t)rr) << 4) | cbyte);
    cp_async8(sm + S_OPA + kp128 + orow, kg_in + offk, ok, pol_qk);
    cp_async8(sm + S_OPA + kp128 + 64u * 128u + orow, qg_in + offk, ok, pol_qk);
    cp_async16(sm + x_slot(rr, tid), xg_in + off, ok, pol_once);
  }
  cp_async_commit();
}

// GROUPED: q, k have Hk < H heads (value head h reads key head h / (H / Hk));
// the ungrouped instantiation shares the gate input's addressing, which keeps
// its per-row address arithmetic out of the issue-bound load phase.
// NARROW: d_k or d_v is 64 (gp.dk, gp.dv); the 128-wide instantiation keeps
// the widths constant, and the masks out of its issue-bound phases.
template <bool GROUPED, bool NARROW>
__global__ void __launch_bounds__(NT, 2)
tc_prep_kernel(const __grid_constant__ TcMaps maps, const __nv_bfloat16 *__restrict__ qg_in,
               const __nv_bfloat16 *__restrict__ kg_in, const float *__restrict__ xg_in,
               const float *__restrict__ beta, GateParams gp, SeqInfo s, int64_t nitems, int H,
               int Hk, char *__restrict__ pkg, float *__restrict__ a_out, uint32_t *err,
               uint32_t *__restrict__ flag_count, uint32_t *__restrict__ flag_list) {
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
  uint32_t *strong_flag = reinterpret_cast<uint32_t *>(sm + M_STRONG);
  ItemSlot *slots = reinterpret_cast<ItemSlot *>(sm + M_ITEM);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;
  const bool l2n = (gp.flags & KDA_L2NORM_QK) != 0;
  const bool sig = (gp.flags & KDA_BETA_SIGMOID) != 0;
  constexpr float kLog2e = 1.4426950408889634f;
  const int dk = NARROW ? gp.dk : 128, dv = NARROW ? gp.dv : 128;  // narrow heads are read with the
                                              // channels from dk on held at zero
  const int64_t rowH = (int64_t)H * dk;       // elements between tokens of the gate input
  const int64_t rowHk = GROUPED ? (int64_t)Hk * dk : rowH;  // and of q, k
  const int grp = GROUPED ? H / Hk : 1;                       // value heads per key head

  if (warp == 0) {
    tc::tmem_alloc(tslot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar_v, 1);
    tc::mbar_init(bar_mma, 1);
    tc::mbar_fence_init();
    *abort_flag = 0;
    *strong_flag = 0;
    tc::tma_prefetch_desc(&maps.v);
  }
  if (dv < 128) {  // the v tile's second panel is never loaded: zero, for every item
    reinterpret_cast<uint4 *>(sm + S_V + 8192)[tid] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4 *>(sm + S_V + 8192)[tid + NT] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;

  // elementwise roles: lane = channel quad (channels c0 .. c0 + 3), warp =
  // row group (rows 8 warp .. 8 warp + 7) inside sub-block R = warp / 2
  const int c0 = 4 * lane, R = warp >> 1;
  const bool cin = !NARROW || c0 < dk;  // this thread's channels exist (d_k = 64: lanes 16..31 do not)
  const uint32_t ch16 = (uint32_t)((lane & 15) >> 1), cbyte = (uint32_t)(lane & 1) * 8u;
  const uint32_t pan = (uint32_t)(lane >> 4);

  const int64_t G = gridDim.x;
  const uint64_t pol_once = policy_evict_first();
  // q, k rows shared by a group of value heads are read once per head
  const uint64_t pol_qk = GROUPED ? policy_evict_normal() : pol_once;
  // thread 0 keeps count of the loads and MMAs it started, for the drain
  int64_t v_issued = 0, v_done = 0;
  bool mma_pending = false;
  const uint32_t kp128 = pan * 128u * 128u, kp160 = pan * B1_PANEL, kp64 = pan * 64u * 128u;
  const int prow0 = 16 * lane_block(R) + 8 * (warp & 1);  // OPA row of this thread's first row
  if (tid == 0) {
    Item it0 = get_item(s, H, blockIdx.x);
    const bool ok0 = blockIdx.x < nitems && it0.ok;
    put_slot(slots[0], it0, ok0);
  }
  __syncthreads();
  // the first item's rows; every later item's are requested during the item
  // before it, once that item's second MMA has finished, so that they arrive
  // while it reads out w and u
  float bnext = 0.f;
  if (slots[0].ok) {
    stage_rows<GROUPED>(sm, slots[0], qg_in, kg_in, xg_in, dk, rowH, rowHk, grp, warp, c0, cin, tid, kp128,
                        prow0, ch16, cbyte, pol_qk, pol_once);
    if (tid < 64 && tid < slots[0].len) bnext = beta[(slots[0].t0 + tid) * H + slots[0].h];
  }

  uint32_t mma_phase = 0;
  int64_t i = 0;
  for (int64_t w = blockIdx.x; w < nitems; w += G, ++i) {
    const ItemSlot it = slots[i & 1];
    if (!it.ok) break;  // items past the last chunk are all invalid
    const int len = it.len, h = it.h;
    const int64_t t0 = it.t0;
    uint8_t *pk = reinterpret_cast<uint8_t *>(pkg + (size_t)(it.gc * H + h) * PK_BYTES);
    const int64_t base_h = t0 * rowH + (int64_t)h * dk;            // (t0, h, 0) of the gate input
    const int64_t base_k = t0 * rowHk + (int64_t)(GROUPED ? h / grp : h) * dk;  // (t0, h / grp, 0) of q, k
    Item nx;
    bool okn = false;
    if (tid == 0) {
      const int64_t wn = w + G;
      nx = get_item(s, H, wn < nitems ? wn : 0);
      okn = wn < nitems && nx.ok;
      put_slot(slots[(i + 1) & 1], nx, okn);
      if (okn) {
        tma_prefetch_l2_3d(&maps.q, 0, nx.h / grp, (int32_t)nx.t0);
        tma_prefetch_l2_3d(&maps.k, 0, nx.h / grp, (int32_t)nx.t0);
        tma_prefetch_l2_3d(&maps.x, 0, nx.h, (int32_t)nx.t0);
      }
    }

    // ---- phase 1: the item's loads (q, k, gate input: 8 rows x 4 channels
    //      per thread; beta), row norms (warp butterfly over the 16 partial
    //      sums of its 8 rows), gate in log2 units and the cumulative sums
    //      of each 8-row group
    float Gl[8][4];
    {
      uint2 qv[8], kv[8];
      float4 xs[8];
      cp_async_wait_all();  // this thread's own copies: no barrier needed
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const uint32_t orow = (uint32_t)(prow0 + rr) * 128u + (((ch16 ^ (uint32_t)rr) << 4) | cbyte);
        kv[rr] = *reinterpret_cast<const uint2 *>(sm + S_OPA + kp128 + orow);
        qv[rr] = *reinterpret_cast<const uint2 *>(sm + S_OPA + kp128 + 64u * 128u + orow);
        xs[rr] = *reinterpret_cast<const float4 *>(sm + x_slot(rr, tid));
      }
      const float bload = bnext;
      const float A_h = gate ? tc::ex2(gp.a_log[h] * kLog2e) : 0.f;
      float dbl[4];  // dt_bias in log2 units
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dbl[j] = (gate && gp.dt_bias && cin) ? gp.dt_bias[h * dk + c0 + j] * kLog2e : 0.f;

      float v[16];
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qv[rr]);
        const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kv[rr]);
        const float2 a0 = __bfloat1622float2(q2[0]), a1 = __bfloat1622float2(q2[1]);
        const float2 b0 = __bfloat1622float2(k2[0]), b1 = __bfloat1622float2(k2[1]);
        v[rr] = a0.x * a0.x + a0.y * a0.y + a1.x * a1.x + a1.y * a1.y;
        v[8 + rr] = b0.x * b0.x + b0.y * b0.y + b1.x * b1.x + b1.y * b1.y;
      }
      // butterfly: each step halves the values a lane holds; afterwards lane
      // l holds the warp sum of value ((l>>4)&1)*8 + ((l>>3)&1)*4 + ((l>>2)&1)*2 + ((l>>1)&1)
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const int half = 8 >> st, msk = 16 >> st;
        const bool up = (lane & msk) != 0;
#pragma unroll
        for (int i2 = 0; i2 < half; ++i2) {
          const float send = up ? v[i2] : v[i2 + half];
          const float keep = up ? v[i2 + half] : v[i2];
          v[i2] = keep + __shfl_xor_sync(0xffffffffu, send, msk);
        }
      }
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
      if ((lane & 1) == 0) {
        const int idx = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 +
                        ((lane >> 1) & 1);
        const int r = 8 * warp + (idx & 7);
        const float nv = r < len ? (l2n ? rsqrtf(v[0] + gp.eps) : 1.f) : 0.f;
        if (idx < 8) rq[r] = nv * gp.scale;  // q rows carry the attention scale
        else rk[r] = nv;
      }
      if (tid < 64) sbeta[tid] = (sig && tid < len) ? 1.f / (1.f + tc::ex2(-bload * kLog2e)) : bload;

      float2 acc[2] = {splat2(0.f), splat2(0.f)};
      const float2 dbl2[2] = {make_float2(dbl[0], dbl[1]), make_float2(dbl[2], dbl[3])};
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int r = 8 * warp + rr;
        const float2 xv[2] = {make_float2(xs[rr].x, xs[rr].y), make_float2(xs[rr].z, xs[rr].w)};
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          float2 g;
          if (gate) {
            // softplus(z) log2 e = max(z, 0) log2 e + log2(1 + 2^{-|z| log2 e})
            const float2 z = fma2(xv[p], splat2(kLog2e), dbl2[p]);
            const float2 t = add2(splat2(1.f), make_float2(tc::ex2(-fabsf(z.x)), tc::ex2(-fabsf(z.y))));
            g = mul2(splat2(-A_h), add2(make_float2(fmaxf(z.x, 0.f), fmaxf(z.y, 0.f)),
                                        make_float2(tc::lg2(t.x), tc::lg2(t.y))));
          } else {
            g = mul2(xv[p], splat2(kLog2e));
          }
          if (r >= len || !cin) g = splat2(0.f);
          acc[p] = add2(acc[p], g);
          Gl[rr][2 * p] = acc[p].x;
          Gl[rr][2 * p + 1] = acc[p].y;
        }
      }
      *reinterpret_cast<float4 *>(tot + warp * 128 + c0) = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
    }
    // the staging buffers of the previous item must be read out before this
    // item's operand tiles overwrite them
    if (tid == 0) bulk_wait_read();
    __syncthreads();  // group totals, rstd and beta published; x slots read
    // every thread has read its x slots: the item's v may land in the first panel
    if (tid == 0) {
      tc::fence_proxy_async_smem();
      tc::mbar_arrive_expect_tx(bar_v, dv == 128 ? 16384u : 8192u);
      tma_load_3d(sm + S_V, &maps.v, bar_v, 0, h, (int32_t)t0);
      if (dv == 128) tma_load_3d(sm + S_V + 8192, &maps.v, bar_v, 64, h, (int32_t)t0);
      ++v_issued;
    }

    // ---- phase 2: operand tiles and the elementwise package parts
    bool strong = false;
    {
      // b_RR = gate sum before sub-block RR, G_C = sum over the chunk
      float bAll[4][4], GC[4], prev[4];
      {
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int gg = 0; gg < 8; ++gg) {
          const float4 t = *reinterpret_cast<const float4 *>(tot + gg * 128 + c0);
          const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if ((gg & 1) == 0) bAll[gg >> 1][j] = a[j];
            if (gg == (warp | 1) - 1) prev[j] = tv[j];
            a[j] += tv[j];
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) GC[j] = a[j];
      }
      // rows of the second group of a sub-block: relative to its start
      if (warp & 1) {
#pragma unroll
        for (int rr = 0; rr < 8; ++rr)
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const float2 gs = add2(make_float2(Gl[rr][2 * p], Gl[rr][2 * p + 1]),
                                   make_float2(prev[2 * p], prev[2 * p + 1]));
            Gl[rr][2 * p] = gs.x;
            Gl[rr][2 * p + 1] = gs.y;
          }
      }
      // strong decay: the gate decays (g <= 0), so inside a sub-block it
      // has moved furthest at the last row - of this thread's 8-row group,
      // and of the sub-block at the second group's last row
#pragma unroll
      for (int j = 0; j < 4; ++j) strong |= -Gl[7][j] > STRONG_DECAY_LOG2;
      float ebs[4], egcs[4], cRs[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float bR = bAll[0][j];
#pragma unroll
        for (int RR = 1; RR < 4; ++RR)
          if (RR == R) bR = bAll[RR][j];
        ebs[j] = tc::ex2(bR);
        egcs[j] = tc::ex2(GC[j] - bR);
#pragma unroll
        for (int RR = 1; RR < 4; ++RR) cRs[RR][j] = tc::ex2(fminf(bAll[RR][j] - bR, 0.f));
      }
      float2 eb[2], egc[2], cR[4][2];
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        eb[p] = make_float2(ebs[2 * p], ebs[2 * p + 1]);
        egc[p] = make_float2(egcs[2 * p], egcs[2 * p + 1]);
#pragma unroll
        for (int RR = 1; RR < 4; ++RR) cR[RR][p] = make_float2(cRs[RR][2 * p], cRs[RR][2 * p + 1]);
      }
      if (warp == 0)
        *reinterpret_cast<float4 *>(pk + PK_GC + c0 * 4) =
            make_float4(tc::ex2(GC[0]), tc::ex2(GC[1]), tc::ex2(GC[2]), tc::ex2(GC[3]));
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int r = 8 * warp + rr;
        const uint32_t xo = ((ch16 ^ (uint32_t)rr) << 4) | cbyte;
        const uint32_t rowb = (uint32_t)r * 128u + xo;
        const uint32_t orow = (uint32_t)(prow0 + rr) * 128u + xo;
        const float sq = rq[r], sk = rk[r];
        // raw rows this thread copied in (cp.async) and read in phase 1
        const uint2 qraw = *reinterpret_cast<const uint2 *>(sm + S_OPA + kp128 + 64u * 128u + orow);
        const uint2 kraw = *reinterpret_cast<const uint2 *>(sm + S_OPA + kp128 + orow);
        const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qraw);
        const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kraw);
        const float2 qa = __bfloat1622float2(q2[0]), qb = __bfloat1622float2(q2[1]);
        const float2 ka = __bfloat1622float2(k2[0]), kb = __bfloat1622float2(k2[1]);
        const float2 qn[2] = {mul2(qa, splat2(sq)), mul2(qb, splat2(sq))};
        const float2 kn[2] = {mul2(ka, splat2(sk)), mul2(kb, splat2(sk))};
        float2 ke[2], kf[2], qe[2], kd[2], qg[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const float g0 = Gl[rr][2 * p], g1 = Gl[rr][2 * p + 1];
          const float2 e = make_float2(tc::ex2(g0), tc::ex2(g1));
          const float2 f = make_float2(tc::ex2(fminf(-g0, 126.f)), tc::ex2(fminf(-g1, 126.f)));
          ke[p] = mul2(kn[p], e);
          kf[p] = mul2(kn[p], f);
          qe[p] = mul2(qn[p], e);
          kd[p] = mul2(ke[p], eb[p]);  // k^ 2^G, G from the chunk start
          qg[p] = mul2(qe[p], eb[p]);  // scale q^ 2^G
        }
        st_u64(sm + S_OPA, kp128 + orow, pack4(ke[0], ke[1]));
        st_u64(sm + S_OPA, kp128 + 64u * 128u + orow, pack4(qe[0], qe[1]));
        st_u64(sm + S_B1, kp160 + 96u * 128u + rowb, pack4(kf[0], kf[1]));
#pragma unroll
        for (int Rp = 1; Rp < 4; ++Rp)
          if (Rp > R)
            st_u64(sm + S_B1, kp160 + (uint32_t)b1_off(Rp) * 128u + rowb,
                   pack4(mul2(kf[0], cR[Rp][0]), mul2(kf[1], cR[Rp][1])));
        st_u64(sm + S_B2A, kp64 + rowb, pack4(kd[0], kd[1]));
        // package: qg = scale q^ 2^G (WQ rows 0..63), kg = k^ 2^{G_C - G} (KG)
        stg_hint(pk, PK_WQ + kp128 + rowb, pack4(qg[0], qg[1]), pol_once);
        stg_hint(pk, PK_KG + kp64 + rowb, pack4(mul2(kf[0], egc[0]), mul2(kf[1], egc[1])), pol_once);
      }
    }
    if (strong)
      strong_factors_exact(sm, pk, kg_in, xg_in, gp, h, len, base_h, base_k, rowH, rowHk, kp160, kp64, pol_once,
                           pol_qk);
    tc::fence_proxy_async_smem();
    // an item under strong decay: the warps that see it mark it; after the
    // first MMA its diagonal blocks are recomputed and thread 0 lists it for
    // the backward
    if (__any_sync(0xffffffffu, strong) && lane == 0) atomicOr(strong_flag, 1u);
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
    if (tid == 0 && *strong_flag)  // the backward recomputes these items exactly too
      flag_list[atomicAdd(flag_count, 1u)] = (uint32_t)w;

    // ---- read D1: L (k rows) to shared fp32, Aqk (q rows) to the package;
    //      zero the inverse buffer
    {
      const int q4 = warp & 3, cq = warp >> 2;
      const int m = 32 * q4 + lane;          // D1 row = TMEM lane
      const bool krow = m < 64;
      const int Rr = token_block((m & 63) >> 4);
      const int r = 16 * Rr + (m & 15);
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
      // column blocks of D1 this warp reads: lanes of token blocks 0 and 3
      // need blocks 6 and 3, 4, 5, 9; those of blocks 1 and 2 need 0, 7 and
      // 1, 2, 8
      int chs[4] = {-1, -1, -1, -1};
      if ((q4 & 1) == 0) {
        if (cq == 0) { chs[0] = 3; chs[1] = 4; chs[2] = 9; } else { chs[0] = 5; chs[1] = 6; }
      } else {
        if (cq == 0) { chs[0] = 0; chs[1] = 1; chs[2] = 7; } else { chs[0] = 2; chs[1] = 8; }
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
          for (int x = 0; x < 16; x += 4) {
            const int j = j0 + x;
            const float2 p0 = mul2(splat2(br), make_float2(d[cix][x], d[cix][x + 1]));
            const float2 p1 = mul2(splat2(br), make_float2(d[cix][x + 2], d[cix][x + 3]));
            float4 l4;
            l4.x = (!diag || j < r) ? p0.x : 0.f;
            l4.y = (!diag || j + 1 < r) ? p0.y : 0.f;
            l4.z = (!diag || j + 2 < r) ? p1.x : 0.f;
            l4.w = (!diag || j + 3 < r) ? p1.y : 0.f;
            *reinterpret_cast<float4 *>(LF + r * LFS + j) = l4;
          }
        } else {
          uint32_t pkd[8];
#pragma unroll
          for (int x = 0; x < 16; x += 2) {
            const int j = j0 + x;
            const float a0 = (!diag || j <= r) ? d[cix][x] : 0.f;
            const float a1 = (!diag || j + 1 <= r) ? d[cix][x + 1] : 0.f;
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
    if (*reinterpret_cast<volatile uint32_t *>(strong_flag)) {
      diagonal_blocks_exact(sm, qg_in, kg_in, xg_in, gp, h, len, base_h, base_k, rowH, rowHk);
      tc::fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) *strong_flag = 0;  // every thread has read it; the next item marks after barriers
    }
    if (tid == 0) {
      bulk_store_hint(pk + PK_AQK, sm + S_STG_AQK, 8192, pol_once);
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
      //     each step is broadcast inside the 4-lane group.  The threads of
      //     blocks 0 and 2 also clear the block to their right, the zero
      //     upper corner of each 32 x 32 diagonal half.
      {
        const int col = tid >> 2, part = tid & 3;
        const int blk = col >> 4, base = 16 * blk, jj = col & 15;
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
        for (int a = 0; a < 4; ++a) {
          AF[(base + part + 4 * a) * LFS + base + jj] = x[a];
          if ((blk & 1) == 0) AF[(base + part + 4 * a) * LFS + base + 16 + jj] = 0.f;
        }
      }
      // step (2) of a half reads only that half's diagonal blocks
      half_sync(warp >> 2);
      // (2) 32 x 32 diagonal halves: X_10 = -X_1 (L_10 X_0), X_32 = -X_3 (L_32 X_2),
      //     16 x 16 x 16 products as warp-level MMAs: in half pr, warps 0 and 1
      //     of the half own the 8-column tiles of the 16 x 16 result
      {
        const int pr = warp >> 2, wl = warp & 3;
        const int rI = 32 * pr + 16, cJ = 32 * pr;
        const int g = lane >> 2, t = lane & 3;
        float *T2 = TT + pr * 16 * TTS;
        if (wl < 2) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          warp_mm_tf32<16>(LF + rI * LFS + cJ, LFS, AF + cJ * LFS + cJ + 8 * wl, LFS, g, t, acc);
          *reinterpret_cast<float2 *>(T2 + g * TTS + 8 * wl + 2 * t) = make_float2(acc[0], acc[1]);
          *reinterpret_cast<float2 *>(T2 + (g + 8) * TTS + 8 * wl + 2 * t) = make_float2(acc[2], acc[3]);
        }
        half_sync(pr);
        if (wl < 2) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          warp_mm_tf32<16>(AF + rI * LFS + rI, LFS, T2 + 8 * wl, TTS, g, t, acc);
          *reinterpret_cast<float2 *>(AF + (rI + g) * LFS + cJ + 8 * wl + 2 * t) = make_float2(-acc[0], -acc[1]);
          *reinterpret_cast<float2 *>(AF + (rI + g + 8) * LFS + cJ + 8 * wl + 2 * t) =
              make_float2(-acc[2], -acc[3]);
        }
      }
      __syncthreads();
      // (3) lower-left 32 x 32 block: A_21 = -A_2 (L_21 A_1), both 32 x 32 x 32
      //     products on the tensor cores with warp-level MMAs (operands and
      //     results stay in registers, no tensor-memory round trip); warp w
      //     owns the 16 x 8 output tile (rows 16 (w >> 2), columns 8 (w & 3))
      {
        const int rt = 16 * (warp >> 2), ct = 8 * (warp & 3);
        const int g = lane >> 2, t = lane & 3;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        warp_mm_tf32<32>(LF + (32 + rt) * LFS, LFS, AF + ct, LFS, g, t, acc);
        *reinterpret_cast<float2 *>(TT + (rt + g) * TTS + ct + 2 * t) = make_float2(acc[0], acc[1]);
        *reinterpret_cast<float2 *>(TT + (rt + g + 8) * TTS + ct + 2 * t) = make_float2(acc[2], acc[3]);
        __syncthreads();
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        warp_mm_tf32<32>(AF + (32 + rt) * LFS + 32, LFS, TT + ct, TTS, g, t, acc);
        *reinterpret_cast<float2 *>(AF + (32 + rt + g) * LFS + ct + 2 * t) = make_float2(-acc[0], -acc[1]);
        *reinterpret_cast<float2 *>(AF + (32 + rt + g + 8) * LFS + ct + 2 * t) = make_float2(-acc[2], -acc[3]);
      }
      __syncthreads();
      if (a_out) {  // A = (I + L)^-1 of the item in fp32, for a backward (rows past the end: 0)
        float4 *dst = reinterpret_cast<float4 *>(a_out + (size_t)(it.gc * H + h) * (BT * BT));
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int e = 4 * (tid + 256 * x), r = e >> 6, j = e & 63;
          float v4[4];
#pragma unroll
          for (int y = 0; y < 4; ++y) v4[y] = (r < len && j + y <= r) ? AF[r * LFS + j + y] : 0.f;
          dst[tid + 256 * x] = make_float4(v4[0], v4[1], v4[2], v4[3]);
        }
      }
      // A . diag(beta) -> bf16, rows r and 64 + r of [A'; A']
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = (tid >> 3) + 32 * hh, g = tid & 7;
        uint32_t pkd[4];
#pragma unroll
        for (int x = 0; x < 8; x += 2) {
          const int jj = 8 * g + x;
          const float2 ab = mul2(*reinterpret_cast<const float2 *>(AF + r * LFS + jj),
                                 *reinterpret_cast<const float2 *>(sbeta + jj));
          pkd[x / 2] = pack_bf16((jj <= r) ? ab.x : 0.f, (jj + 1 <= r) ? ab.y : 0.f);
        }
        const uint4 av = make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
        *reinterpret_cast<uint4 *>(sm + S_AINV + kmaj_off(128, r, 8 * g)) = av;
        *reinterpret_cast<uint4 *>(sm + S_AINV + kmaj_off(128, 64 + r, 8 * g)) = av;
      }
    }
    tc::fence_proxy_async_smem();
    // v of this item must have landed before the second MMA reads it
    ok = wait_or_flag(bar_v, (uint32_t)(i & 1), err);
    if (ok) v_done = i + 1;
    else *abort_flag = 1;
    __syncthreads();
    if (*abort_flag) break;

    // ---- MMA 2: [A'; A'] x k^ 2^G -> D2 columns 0..127 (w in rows 0..63),
    //      [A'; A'] x v -> columns 128..255 (u in rows 64..127)
    if (tid == 0) {
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(128, 128, false, true);
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
    // the Aqk image must be read out before the U staging overwrites it
    if (tid == 0) bulk_wait_read();
    tc::tc_fence_after();
    __syncthreads();
    if (*abort_flag) break;

    // the second MMA and the read of the Aqk image are done: request the next
    // item's rows
    {
      const ItemSlot itn = slots[(i + 1) & 1];
      if (itn.ok) {
        stage_rows<GROUPED>(sm, itn, qg_in, kg_in, xg_in, dk, rowH, rowHk, grp, warp, c0, cin, tid, kp128,
                            prow0, ch16, cbyte, pol_qk, pol_once);
        if (tid < 64 && tid < itn.len) bnext = beta[(itn.t0 + tid) * H + itn.h];
      }
    }

    // ---- read D2: w (lanes 0..63 of columns 0..127) -> package WQ rows
    //      64..127, u (lanes 64..127 of columns 128..255) -> package U;
    //      warp = (lane quarter, 64-column half)
    {
      const int q4 = warp & 3, hf = warp >> 2;
      const bool is_u = q4 >= 2;
      const int r = 32 * (q4 & 1) + lane;
#pragma unroll
      for (int cp = 0; cp < 2; ++cp) {
        float d[2][16];
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
          tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (is_u ? 128 : 0) + 64 * hf + 32 * cp + 16 * cc,
                        d[cc]);
        tc::tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int col = 64 * hf + 32 * cp + 16 * cc;  // column inside w or u
          if (!is_u) {
            uint32_t pkd[8];
#pragma unroll
            for (int x = 0; x < 16; x += 2) pkd[x / 2] = pack_bf16(d[cc][x], d[cc][x + 1]);
            *reinterpret_cast<uint4 *>(sm + S_STG_W + kmaj_off(64, r, col)) =
                make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
            *reinterpret_cast<uint4 *>(sm + S_STG_W + kmaj_off(64, r, col + 8)) =
                make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
          } else {
            uint32_t pku[8];
#pragma unroll
            for (int x = 0; x < 16; x += 2) pku[x / 2] = pack_bf16(d[cc][x], d[cc][x + 1]);
            *reinterpret_cast<uint4 *>(sm + S_STG_U + u_offset(r, col)) =
                make_uint4(pku[0], pku[1], pku[2], pku[3]);
            *reinterpret_cast<uint4 *>(sm + S_STG_U + u_offset(r, col + 8)) =
                make_uint4(pku[4], pku[5], pku[6], pku[7]);
          }
        }
      }
    }
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store_hint(pk + PK_WQ + 64 * 128, sm + S_STG_W, 8192, pol_once);
      bulk_store_hint(pk + PK_WQ + 16384 + 64 * 128, sm + S_STG_W + 8192, 8192, pol_once);
      bulk_store_hint(pk + PK_U, sm + S_STG_U, 16384, pol_once);
      bulk_commit();
    }
  }

  // Drain after a timeout: wait (bounded) for the load and the MMA this CTA
  // started, so that nothing lands in memory it no longer owns.  On the
  // normal path every issued load has been consumed.
  cp_async_wait_all();
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

cudaError_t launch_tc_prep(const TcMaps &maps, const void *q, const void *k, const void *v,
                           const float *x, const float *beta, const GateParams &gp,
                           const SeqInfo &s, int64_t nchunks, int H, int Hk, char *pkg,
                           uint32_t *err, uint32_t *flag_count, uint32_t *flag_list,
                           cudaStream_t st, float *a_out) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  const bool narrow = gp.dk != 128 || gp.dv != 128;
  auto kern = Hk != H ? (narrow ? tc_prep_kernel<true, true> : tc_prep_kernel<true, false>)
                      : (narrow ? tc_prep_kernel<false, true> : tc_prep_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t nitems = nchunks * H;
  if (nitems == 0) return cudaSuccess;
  if (nitems > (int64_t)UINT32_MAX) return cudaErrorInvalidValue;  // list entries are 32-bit
  if ((e = cudaMemsetAsync(flag_count, 0, sizeof(uint32_t), st)) != cudaSuccess) return e;
  const int64_t slots = 2 * (int64_t)sms;
  const int grid = (int)(nitems < slots ? nitems : slots);
  kern<<<grid, NT, SMEM_BYTES, st>>>(maps, static_cast<const __nv_bfloat16 *>(q),
                                     static_cast<const __nv_bfloat16 *>(k), x, beta, gp, s, nitems,
                                     H, Hk, pkg, a_out, err, flag_count, flag_list);
  return cudaGetLastError();
}

}  // namespace tcp
}  // namespace kda
