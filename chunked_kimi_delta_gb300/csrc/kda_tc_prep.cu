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

constexpr int NT = 256;

// Shared memory (bytes from a 1024-aligned base).
constexpr uint32_t S_INQ = 0;        // bf16 [64][128] (plain rows)
constexpr uint32_t S_INK = 16384;    // bf16 [64][128]
constexpr uint32_t S_INX = 32768;    // fp32 [64][128]
constexpr uint32_t S_INV = 65536;    // 2 x 16384: v, MN-major SW128 (K = tokens)
constexpr uint32_t S_OPA = 98304;    // [k E ; q E] K-major, 128 rows (32768)
constexpr uint32_t S_B1 = 131072;    // 160 rows K-major (2 panels x 20480)
constexpr uint32_t S_B2A = 172032;   // k^ 2^G, MN-major (16384)
// after the first MMA the OPA/B1 region is reused:
constexpr uint32_t S_LF = 98304;     // fp32 L [64][65]
constexpr uint32_t S_AF = 114944;    // fp32 A [64][65]
constexpr uint32_t S_TT = 131584;    // fp32 scratch [16][48]
constexpr uint32_t S_AINV = 135168;  // bf16 A.diag(beta), K-major 64 rows (8192)
constexpr uint32_t S_MISC = 188416;
constexpr uint32_t M_RQ = S_MISC;          // fp32 [64] rstd q
constexpr uint32_t M_RK = S_MISC + 256;    // fp32 [64] rstd k
constexpr uint32_t M_BETA = S_MISC + 512;  // fp32 [64]
constexpr uint32_t M_TOT = S_MISC + 768;   // fp32 [4][128] sub-block gate totals
constexpr uint32_t M_BAR = S_MISC + 2816;  // bar_in, bar_v0, bar_v1, bar_mma
constexpr uint32_t M_TSLOT = S_MISC + 2848;
constexpr uint32_t M_ABORT = S_MISC + 2852;
constexpr uint32_t SMEM_BYTES = S_MISC + 2880 + 1024;

constexpr uint32_t B1_PANEL = 160 * 128;
constexpr uint32_t TMEM_COLS = 256;

__device__ __forceinline__ int b1_off(int Rp) { return 8 * Rp * (Rp - 1); }  // 0, 16, 48

struct Item {
  int n, len, h;
  int64_t t0, gc;
  bool ok;
};

__device__ __forceinline__ Item get_item(const SeqInfo &s, int H, int64_t w) {
  Item it;
  it.gc = w / H;
  it.h = (int)(w % H);
  it.ok = chunk_lookup(s, it.gc, it.n, it.t0, it.len);
  return it;
}

__device__ __forceinline__ void issue_qkx(const TcMaps &m, uint8_t *sm, uint64_t *bar,
                                          const Item &it) {
  tc::mbar_arrive_expect_tx(bar, 65536);
  tma_load_3d(sm + S_INQ, &m.q, bar, 0, it.h, (int32_t)it.t0);
  tma_load_3d(sm + S_INK, &m.k, bar, 0, it.h, (int32_t)it.t0);
  tma_load_3d(sm + S_INX, &m.x, bar, 0, it.h, (int32_t)it.t0);
}

__device__ __forceinline__ void issue_v(const TcMaps &m, uint8_t *dst, uint64_t *bar,
                                        const Item &it) {
  tc::mbar_arrive_expect_tx(bar, 16384);
  tma_load_3d(dst, &m.v, bar, 0, it.h, (int32_t)it.t0);
  tma_load_3d(dst + 8192, &m.v, bar, 64, it.h, (int32_t)it.t0);
}

__device__ __forceinline__ void st_u32(uint8_t *base, uint32_t off, uint32_t v) {
  *reinterpret_cast<uint32_t *>(base + off) = v;
}

__global__ void __launch_bounds__(NT, 1)
tc_prep_kernel(const __grid_constant__ TcMaps maps, const float *__restrict__ beta, GateParams gp,
               SeqInfo s, int64_t nitems, int H, char *__restrict__ pkg, uint32_t *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *rq = reinterpret_cast<float *>(sm + M_RQ);
  float *rk = reinterpret_cast<float *>(sm + M_RK);
  float *sbeta = reinterpret_cast<float *>(sm + M_BETA);
  float *tot = reinterpret_cast<float *>(sm + M_TOT);
  uint64_t *bar_in = reinterpret_cast<uint64_t *>(sm + M_BAR);
  uint64_t *bar_v = bar_in + 1;  // [2]
  uint64_t *bar_mma = bar_in + 3;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + M_TSLOT);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sm + M_ABORT);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;
  const bool l2n = (gp.flags & KDA_L2NORM_QK) != 0;
  const bool sig = (gp.flags & KDA_BETA_SIGMOID) != 0;
  constexpr float kLog2e = 1.4426950408889634f;

  if (warp == 0) {
    tc::tmem_alloc(tslot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar_in, 1);
    tc::mbar_init(bar_v, 1);
    tc::mbar_init(bar_v + 1, 1);
    tc::mbar_init(bar_mma, 1);
    tc::mbar_fence_init();
    *abort_flag = 0;
    tc::tma_prefetch_desc(&maps.q);
    tc::tma_prefetch_desc(&maps.k);
    tc::tma_prefetch_desc(&maps.v);
    tc::tma_prefetch_desc(&maps.x);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;

  const int64_t G = gridDim.x;
  // thread 0 keeps count of the loads and MMAs it started, for the drain
  int64_t qkx_issued = 0, qkx_done = 0, v_issued[2] = {0, 0}, v_done[2] = {0, 0};
  bool mma_pending = false;
  {
    Item it0 = get_item(s, H, blockIdx.x);
    if (tid == 0 && blockIdx.x < nitems && it0.ok) {
      issue_qkx(maps, sm, bar_in, it0);
      issue_v(maps, sm + S_INV, bar_v, it0);
      qkx_issued = 1;
      v_issued[0] = 1;
      Item it1 = get_item(s, H, blockIdx.x + G);
      if (blockIdx.x + G < nitems && it1.ok) {
        issue_v(maps, sm + S_INV + 16384, bar_v + 1, it1);
        v_issued[1] = 1;
      }
    }
  }

  uint32_t mma_phase = 0;
  int64_t i = 0;
  for (int64_t w = blockIdx.x; w < nitems; w += G, ++i) {
    const Item it = get_item(s, H, w);
    if (!it.ok) break;  // items past the last chunk are all invalid
    const int vb = (int)(i & 1);
    uint8_t *inv = sm + S_INV + vb * 16384;
    const int len = it.len, h = it.h;
    const int64_t t0 = it.t0;

    // ---- wait for this item's inputs
    bool ok = wait_or_flag(bar_in, (uint32_t)(i & 1), err);
    if (ok) qkx_done = i + 1;
    ok = ok && wait_or_flag(bar_v + vb, (uint32_t)((i >> 1) & 1), err);
    if (ok) v_done[vb] = (i >> 1) + 1;
    if (!ok) *abort_flag = 1;
    __syncthreads();
    if (*abort_flag) break;

    // ---- pass A: row norms, beta
    {
      const __nv_bfloat16 *Q = reinterpret_cast<const __nv_bfloat16 *>(sm + S_INQ);
      const __nv_bfloat16 *Kk = reinterpret_cast<const __nv_bfloat16 *>(sm + S_INK);
      for (int rr = 0; rr < 8; ++rr) {
        const int r = warp * 8 + rr;
        const uint2 qa = *reinterpret_cast<const uint2 *>(Q + r * 128 + lane * 4);
        const uint2 ka = *reinterpret_cast<const uint2 *>(Kk + r * 128 + lane * 4);
        const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qa);
        const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&ka);
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float2 a = __bfloat1622float2(q2[e]), b = __bfloat1622float2(k2[e]);
          sq += a.x * a.x + a.y * a.y;
          sk += b.x * b.x + b.y * b.y;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          sq += __shfl_xor_sync(0xffffffffu, sq, o);
          sk += __shfl_xor_sync(0xffffffffu, sk, o);
        }
        if (lane == 0) {
          const bool v = r < len;
          rq[r] = v ? (l2n ? rsqrtf(sq + gp.eps) : 1.f) : 0.f;
          rk[r] = v ? (l2n ? rsqrtf(sk + gp.eps) : 1.f) : 0.f;
        }
      }
      if (tid < 64) {
        float b = 0.f;
        if (tid < len) {
          b = beta[(t0 + tid) * H + h];
          if (sig) b = 1.f / (1.f + expf(-b));
        }
        sbeta[tid] = b;
      }
    }

    // ---- pass B phase 1: gate and sub-block cumulative sums in registers.
    // thread: channel pair p (channels 2p, 2p+1), sub-block R (rows 16R..16R+15)
    const int p = tid & 63, R = tid >> 6;
    const int c0 = 2 * p;
    float Gl[16][2], qv[16][2], kv[16][2];
    {
      const float A_h = gate ? expf(gp.a_log[h]) : 0.f;
      const float db0 = (gate && gp.dt_bias) ? gp.dt_bias[h * 128 + c0] : 0.f;
      const float db1 = (gate && gp.dt_bias) ? gp.dt_bias[h * 128 + c0 + 1] : 0.f;
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int ii = 0; ii < 16; ++ii) {
        const int r = 16 * R + ii;
        const float2 x = *reinterpret_cast<const float2 *>(sm + S_INX + (r * 128 + c0) * 4);
        const __nv_bfloat162 q2 = *reinterpret_cast<const __nv_bfloat162 *>(sm + S_INQ + (r * 128 + c0) * 2);
        const __nv_bfloat162 k2 = *reinterpret_cast<const __nv_bfloat162 *>(sm + S_INK + (r * 128 + c0) * 2);
        float g0, g1;
        if (gate) {
          const float z0 = x.x + db0, z1 = x.y + db1;
          // softplus in log2 units: max(z,0) log2 e + log2(1 + 2^{-|z| log2 e})
          const float s0 = fmaxf(z0, 0.f) * kLog2e + log2f(1.f + exp2f(-fabsf(z0) * kLog2e));
          const float s1 = fmaxf(z1, 0.f) * kLog2e + log2f(1.f + exp2f(-fabsf(z1) * kLog2e));
          g0 = -A_h * s0;
          g1 = -A_h * s1;
        } else {
          g0 = x.x * kLog2e;
          g1 = x.y * kLog2e;
        }
        if (r >= len) g0 = g1 = 0.f;
        acc0 += g0;
        acc1 += g1;
        Gl[ii][0] = acc0;
        Gl[ii][1] = acc1;
        const float2 qf = __bfloat1622float2(q2), kf = __bfloat1622float2(k2);
        qv[ii][0] = qf.x; qv[ii][1] = qf.y;
        kv[ii][0] = kf.x; kv[ii][1] = kf.y;
      }
      tot[R * 128 + c0] = acc0;
      tot[R * 128 + c0 + 1] = acc1;
    }
    __syncthreads();  // inputs q, k, x consumed; sub-block totals published

    // prefetch the next item's q, k, x into the freed buffers
    if (tid == 0) {
      const int64_t wn = w + G;
      if (wn < nitems) {
        Item nx = get_item(s, H, wn);
        if (nx.ok) {
          issue_qkx(maps, sm, bar_in, nx);
          ++qkx_issued;
        }
      }
    }

    // ---- pass B phase 2: operand tiles and the elementwise package parts
    {
      float bR[2], bAll[4][2], GC[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float a = 0.f;
#pragma unroll
        for (int RR = 0; RR < 4; ++RR) {
          bAll[RR][j] = a;
          a += tot[RR * 128 + c0 + j];
        }
        GC[j] = a;
        bR[j] = bAll[R][j];
      }
      float eb[2], egc[2], cR[4][2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        eb[j] = exp2f(bR[j]);
        egc[j] = exp2f(GC[j] - bR[j]);
#pragma unroll
        for (int RR = 0; RR < 4; ++RR) cR[RR][j] = exp2f(fminf(bAll[RR][j] - bR[j], 0.f));
      }
      char *pk = pkg + (size_t)(it.gc * H + h) * PK_BYTES;
      if (R == 0) {
        float2 gcv = make_float2(exp2f(GC[0]), exp2f(GC[1]));
        *reinterpret_cast<float2 *>(pk + PK_GC + c0 * 4) = gcv;
      }
#pragma unroll
      for (int ii = 0; ii < 16; ++ii) {
        const int r = 16 * R + ii;
        const float sq = rq[r], sk = rk[r];
        float kn[2], qn[2], e[2], f[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          kn[j] = kv[ii][j] * sk;
          qn[j] = qv[ii][j] * sq;
          e[j] = exp2f(Gl[ii][j]);
          f[j] = exp2f(fminf(-Gl[ii][j], 126.f));
        }
        st_u32(sm + S_OPA, kmaj_off(128, r, c0), pack_bf16(kn[0] * e[0], kn[1] * e[1]));
        st_u32(sm + S_OPA, kmaj_off(128, 64 + r, c0), pack_bf16(qn[0] * e[0], qn[1] * e[1]));
        const float kf0 = kn[0] * f[0], kf1 = kn[1] * f[1];
        st_u32(sm + S_B1, (c0 >> 6) * B1_PANEL + tc::sw128_offset(96 + r, (c0 & 63) * 2),
               pack_bf16(kf0, kf1));
#pragma unroll
        for (int Rp = 1; Rp < 4; ++Rp) {
          if (Rp > R) {
            const int row = b1_off(Rp) + r;
            st_u32(sm + S_B1, (c0 >> 6) * B1_PANEL + tc::sw128_offset(row, (c0 & 63) * 2),
                   pack_bf16(kf0 * cR[Rp][0], kf1 * cR[Rp][1]));
          }
        }
        st_u32(sm + S_B2A, mnmaj_off(64, r, c0),
               pack_bf16(kn[0] * e[0] * eb[0], kn[1] * e[1] * eb[1]));
        // package: qg (WQ rows 0..63), kg (KG)
        st_u32(reinterpret_cast<uint8_t *>(pk), PK_WQ + kmaj_off(128, r, c0),
               pack_bf16(gp.scale * qn[0] * e[0] * eb[0], gp.scale * qn[1] * e[1] * eb[1]));
        st_u32(reinterpret_cast<uint8_t *>(pk), PK_KG + mnmaj_off(64, r, c0),
               pack_bf16(kf0 * egc[0], kf1 * egc[1]));
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
    ok = wait_or_flag(bar_mma, mma_phase, err);
    if (ok) { mma_pending = false; mma_phase ^= 1; }
    else *abort_flag = 1;
    tc::tc_fence_after();
    __syncthreads();
    if (*abort_flag) break;

    // ---- read D1: L (k rows) to shared fp32, Aqk (q rows) to the package
    {
      const int q4 = warp & 3;
      const int m = 32 * q4 + lane;          // D1 row = TMEM lane
      const bool krow = m < 64;
      const int r = krow ? m : m - 64;
      const int Rr = r >> 4;
      float *LF = reinterpret_cast<float *>(sm + S_LF);
      char *pk = pkg + (size_t)(it.gc * H + h) * PK_BYTES;
      const float br = sbeta[r];
      const int ch_lo = (warp < 4) ? 0 : 5, ch_hi = (warp < 4) ? 5 : 10;
      if (!krow && warp < 4) {
        // Aqk groups above the diagonal block are zero
        for (int gi = Rr + 1; gi < 4; ++gi) {
          uint4 z = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(pk + PK_AQK + kmaj_off(64, r, 16 * gi)) = z;
          *reinterpret_cast<uint4 *>(pk + PK_AQK + kmaj_off(64, r, 16 * gi + 8)) = z;
        }
      }
      for (int ch = ch_lo; ch < ch_hi; ++ch) {
        float d[16];
        __syncwarp();
        tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + 16 * ch, d);
        tc::tmem_ld_wait();
        // which token block j0.. this chunk holds for a row of block Rr
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
            if (!diag || j < r) LF[r * 65 + j] = br * d[x];
          }
        } else {
          uint32_t pkd[8];
#pragma unroll
          for (int x = 0; x < 16; x += 2) {
            const int j = j0 + x;
            const float a0 = (!diag || j <= r) ? gp.scale * d[x] : 0.f;
            const float a1 = (!diag || j + 1 <= r) ? gp.scale * d[x + 1] : 0.f;
            pkd[x / 2] = pack_bf16(a0, a1);
          }
          *reinterpret_cast<uint4 *>(pk + PK_AQK + kmaj_off(64, r, j0)) =
              make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
          *reinterpret_cast<uint4 *>(pk + PK_AQK + kmaj_off(64, r, j0 + 8)) =
              make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
        }
      }
    }
    tc::tc_fence_before();
    __syncthreads();

    // ---- (I + L)^-1 in fp32, 16 x 16 blocks
    {
      const float *LF = reinterpret_cast<const float *>(sm + S_LF);
      float *AF = reinterpret_cast<float *>(sm + S_AF);
      float *TT = reinterpret_cast<float *>(sm + S_TT);
      // diagonal blocks: one thread per (block, column)
      if (tid < 64) {
        const int I = tid >> 4, jj = tid & 15, base = 16 * I;
        float x[16];
#pragma unroll
        for (int ii = 0; ii < 16; ++ii) {
          float a = (ii == jj) ? 1.f : 0.f;
#pragma unroll
          for (int mm = 0; mm < ii; ++mm) {
            if (mm >= jj) a = fmaf(-LF[(base + ii) * 65 + base + mm], x[mm], a);
          }
          x[ii] = (ii < jj) ? 0.f : a;
          AF[(base + ii) * 65 + base + jj] = x[ii];
        }
      }
      __syncthreads();
      // block rows I = 1..3:  T = L[I, 0:16I] A[0:16I, 0:16I];  A[I, 0:16I] = -X_II T
      for (int I = 1; I < 4; ++I) {
        const int ncol = 16 * I;
        for (int o = tid; o < 16 * ncol; o += NT) {
          const int ii = o / ncol, j = o % ncol;
          const int row = 16 * I + ii;
          float a = 0.f;
          for (int mm = j; mm < ncol; ++mm) a = fmaf(LF[row * 65 + mm], AF[mm * 65 + j], a);
          TT[ii * 48 + j] = a;
        }
        __syncthreads();
        for (int o = tid; o < 16 * ncol; o += NT) {
          const int ii = o / ncol, j = o % ncol;
          const int base = 16 * I;
          float a = 0.f;
          for (int mm = 0; mm <= ii; ++mm) a = fmaf(AF[(base + ii) * 65 + base + mm], TT[mm * 48 + j], a);
          AF[(base + ii) * 65 + j] = -a;
        }
        __syncthreads();
      }
      // A . diag(beta) -> bf16 K-major tile
      {
        const int r = tid >> 2, g4 = tid & 3;
        uint32_t pkd[8];
#pragma unroll
        for (int x = 0; x < 16; x += 2) {
          const int j = 16 * g4 + x;
          const float a0 = (j <= r) ? AF[r * 65 + j] * sbeta[j] : 0.f;
          const float a1 = (j + 1 <= r) ? AF[r * 65 + j + 1] * sbeta[j + 1] : 0.f;
          pkd[x / 2] = pack_bf16(a0, a1);
        }
        *reinterpret_cast<uint4 *>(sm + S_AINV + kmaj_off(64, r, 16 * g4)) =
            make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
        *reinterpret_cast<uint4 *>(sm + S_AINV + kmaj_off(64, r, 16 * g4 + 8)) =
            make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
      }
    }
    tc::fence_proxy_async_smem();
    __syncthreads();

    // ---- MMA 2: w = A' (k^ 2^G) -> cols 0..127, u = A' v -> cols 128..255 (M = 64)
    if (tid == 0) {
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(64, 128, false, true);
      const uint32_t a0 = tc::smem_u32(sm + S_AINV);
      const uint32_t bw = tc::smem_u32(sm + S_B2A), bu = tc::smem_u32(inv);
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

    // ---- read D2 (M = 64 layout: row r in lane (r % 16) + 32 (r / 16)):
    //      w -> package WQ rows 64..127, u -> package U
    {
      const int q4 = warp & 3;
      const int r = 16 * q4 + lane;  // valid for lane < 16
      const bool is_u = warp >= 4;
      char *pk = pkg + (size_t)(it.gc * H + h) * PK_BYTES;
      for (int cc = 0; cc < 8; ++cc) {
        float d[16];
        __syncwarp();
        tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (is_u ? 128 : 0) + 16 * cc, d);
        tc::tmem_ld_wait();
        if (lane < 16) {
          if (!is_u) {
            uint32_t pkd[8];
#pragma unroll
            for (int x = 0; x < 16; x += 2) pkd[x / 2] = pack_bf16(d[x], d[x + 1]);
            *reinterpret_cast<uint4 *>(pk + PK_WQ + kmaj_off(128, 64 + r, 16 * cc)) =
                make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
            *reinterpret_cast<uint4 *>(pk + PK_WQ + kmaj_off(128, 64 + r, 16 * cc + 8)) =
                make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
          } else {
#pragma unroll
            for (int x = 0; x < 16; x += 4)
              *reinterpret_cast<float4 *>(pk + PK_U + u_offset(r, 16 * cc + x)) =
                  make_float4(d[x], d[x + 1], d[x + 2], d[x + 3]);
          }
        }
      }
    }
    tc::tc_fence_before();
    __syncthreads();
    // v buffer vb is free again: fetch v of the item two steps ahead
    if (tid == 0) {
      const int64_t w2 = w + 2 * G;
      if (w2 < nitems) {
        Item n2 = get_item(s, H, w2);
        if (n2.ok) {
          issue_v(maps, inv, bar_v + vb, n2);
          ++v_issued[vb];
        }
      }
    }
  }

  // Drain after a timeout: wait (bounded) for the loads and the MMA this CTA
  // started, so that nothing lands in memory it no longer owns.  On the
  // normal path every issued load has been consumed.
  __syncthreads();
  if (tid == 0 && *abort_flag) {
    if (mma_pending) drain_wait(bar_mma, mma_phase);
    for (int64_t x = qkx_done; x < qkx_issued; ++x) drain_wait(bar_in, (uint32_t)(x & 1));
    for (int b2 = 0; b2 < 2; ++b2)
      for (int64_t x = v_done[b2]; x < v_issued[b2]; ++x) drain_wait(bar_v + b2, (uint32_t)(x & 1));
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_tc_prep(const TcMaps &maps, const float *beta, const GateParams &gp,
                           const SeqInfo &s, int64_t nchunks, int H, char *pkg, uint32_t *err,
                           cudaStream_t st) {
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
  const int grid = (int)(nitems < sms ? nitems : sms);
  tc_prep_kernel<<<grid, NT, SMEM_BYTES, st>>>(maps, beta, gp, s, nitems, H, pkg, err);
  return cudaGetLastError();
}

}  // namespace tcp
}  // namespace kda
