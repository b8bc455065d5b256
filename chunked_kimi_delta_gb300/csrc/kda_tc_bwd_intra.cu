// kda_tc_bwd_intra.cu - intra-chunk backward on the tensor cores (bf16
// inputs, d_k = d_v = 128).
//
// "KDA Chunk Backward - TPU/Pallas Kernel Design" section 2.3: the WY backward
// (from v_new = u - w h, u = A (v.beta), w = A (k^.beta.e^G) to q, k, v, beta,
// g and A), the intra-chunk attention backward (A_qk and the L of
// A = (I + L)^-1) and the reverse cumulative sum over the chunk, then the
// gate, L2-norm and sigmoid backward.  One CTA per (chunk, head).  Every
// contraction is a tcgen05 MMA on bf16 operands with fp32 accumulation in
// TMEM; the CUDA cores build operands and do the elementwise chain rule:
//   M1  dA    = [dv_new | dw] [v.beta | k^.beta.e^G]^T         (64 x 64, K = 256)
//   M2  [dvb | dkb] = A^T [dv_new | dw]                        (64 x 256, K = 64)
//   M4  dA_qk = dO v_new^T                                     (64 x 64, K = 128)
//   M3  T = A^T dA,  dL = -T A^T                               (64 x 64, K = 64)
//   M5  row side of the pairwise terms: for row i in 16-token block I,
//       sum_j Q_ij k^_jc e^{G_ic - G_jc} and sum_j dL_ij (...), with
//       e^{G_i - G_j} = e^{G_i - G_rI} e^{G_rI - G_j} (rI = 16 I) and the
//       blocks' right operands stacked along K (16 + 32 + 48 + 64 = 160)
//   M6  column side: for row j in block J, sum_i (beta_i dL_ij k^_ic + Q_ij q^_ic)
//       e^{G_ic - G_jc}, references at the blocks' last tokens, segments of
//       64 + 48 + 32 + 16 = 160 rows, the dL and Q parts accumulated
// (Q = scale dA_qk on j <= i, dL on j < i.)  Every pair (i, j) enters dG_i
// from the row side and -dG_j from the column side; after the reverse cumsum
// the two cancel in dg_r for r <= j, so both sides must round a pair alike:
// the left operands (Q, dL) are the same bf16 values on both sides, the
// right operands (k^ and q^ with their decay factors) are split into
// bf16 hi + lo parts (two accumulating MMAs), and the diagonal of Q, whose
// two terms cancel exactly in dG, stays out of M5 / M6 and enters dq^ and
// dk^ in fp32 ("dg ... where cumulative contributions nearly cancel",
// section 3.2 of the same design).  The sub-block reference decays
// are those of the forward's A_kk / A_qk (the same section's 3.7): every
// factor off the diagonal blocks is <= 1, inside a block at most 16 tokens of
// decay.
#include <cuda_bf16.h>
#include <string.h>

#include "kda_tc.cuh"

namespace kda {
namespace tcp {
namespace {

constexpr int NT = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// shared memory (bytes from a 1024-aligned base)
// Row strides: fp32 rows of 132 floats (528 bytes, 16-byte aligned) are read
// eight columns at a time by lanes that run over rows, which puts the eight
// lanes of each 128-bit access phase in different banks; the bf16 rows of
// 132 elements (264 bytes) are read as 8-byte vectors.
constexpr int GS = 132;                // floats per row of G and of the final fp32 arrays
constexpr int QS = 132;                // bf16 per row of the raw q / k copies (264 bytes)
constexpr int FS = 66;                 // floats per row of Q and dL (two rows = one GS row)
constexpr uint32_t S_G = 0;            // fp32 G [64][GS], log2 units (chunk-local cumsum)
constexpr uint32_t S_QR = 33792;       // bf16 raw q rows [64][QS]
constexpr uint32_t S_KR = 50688;       // bf16 raw k rows [64][QS]
constexpr uint32_t S_QF = 67584;       // fp32 Q [64][FS]
constexpr uint32_t S_DF = 84480;       // fp32 dL [64][FS]
constexpr uint32_t S_MISC = 101376;
constexpr uint32_t M_BETA = S_MISC;          // fp32 [64]
constexpr uint32_t M_RQ = S_MISC + 256;      // fp32 [64] rstd of q
constexpr uint32_t M_RK = S_MISC + 512;      // fp32 [64] rstd of k
constexpr uint32_t M_DB = S_MISC + 768;      // fp32 [64][4] dbeta parts
constexpr uint32_t M_QD = S_MISC + 1792;     // fp32 [64] diagonal of Q
constexpr uint32_t M_SRED = S_MISC + 2816;   // fp32 [8]
constexpr uint32_t M_BAR = S_MISC + 2880;    // 10 mbarriers
constexpr uint32_t M_TSLOT = S_MISC + 3008;
constexpr int NBAR = 10;
constexpr uint32_t S_R = 104448;       // reused region (120 KB)
// phase A / B tiles (offsets from S_R)
constexpr uint32_t R_DVN = 0, R_DW = 16384, R_VB = 32768, R_KB = 49152, R_AT = 65536;
constexpr uint32_t R_DO = 73728, R_VN = 90112, R_DA = 106496, R_TT = 114688;
// phase C / D tiles
constexpr uint32_t R_AQ = 0, R_AD = 24576, R_BB = 49152;  // M5: A rows (Q, dL), stacked B
constexpr uint32_t R_BLO = 90112;  // M5: lo part of stacked B rows 0..127 (128-row MN-major tile)
constexpr uint32_t R_AP = 0, R_BP = 24576, R_BPL = 65536;  // M6: A, stacked B hi, lo (one part at a time)
// final phase (fp32 [64][GS] each)
constexpr uint32_t R_FG = 0, R_FQ = 33792, R_FK = 67584;
constexpr uint32_t SMEM_BYTES = S_R + 122880 + 1024;
static_assert(S_G + 64 * GS * 4 <= S_QR && S_QR + 64 * QS * 2 <= S_KR && S_KR + 64 * QS * 2 <= S_QF &&
                  S_QF + 64 * FS * 4 == S_DF && S_DF + 64 * FS * 4 <= S_MISC && 2 * FS == GS &&
                  S_MISC + 3072 <= S_R && S_R % 1024 == 0 && R_FQ >= 64 * GS * 4 &&
                  R_FK >= R_FQ + 64 * GS * 4 && R_FK + 64 * GS * 4 + 2048 <= 122880 &&
                  R_BB + 160 * 256 <= R_BLO && R_BLO + 128 * 256 <= 122880,
              "shared memory layout");
static_assert(SMEM_BYTES <= 232448, "dynamic shared memory of one CTA");
constexpr uint32_t TMEM_COLS = 512;
// TMEM columns
constexpr uint32_t C_D2 = 0;      // [-dvb | dkb] (256); later D6Q in 0..127
constexpr uint32_t C_D1 = 256;    // dA, then T, then D6D (128 from 256)
constexpr uint32_t C_D5 = 320;    // dA_qk, then dL
constexpr uint32_t C_D7 = 384;    // column side (128)
constexpr uint32_t KB_BIG = 160;  // stacked segments

__device__ __forceinline__ int seg_off_row(int I) { return 8 * I * (I + 1); }        // 0, 16, 48, 96
__device__ __forceinline__ int seg_off_col(int J) { return 64 * J - 8 * J * (J - 1); } // 0, 64, 112, 144

// Bulk prefetch into L2 (16-byte aligned address, size a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

// Eight consecutive fp32 (16-byte aligned) / bf16 (8-byte aligned) values
// from shared memory.
__device__ __forceinline__ void lds_f8(const float *p, float (&x)[8]) {
  const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void lds_bf8(const __nv_bfloat16 *p, float (&x)[8]) {
  const uint2 a = reinterpret_cast<const uint2 *>(p)[0], b = reinterpret_cast<const uint2 *>(p)[1];
  const uint32_t w[4] = {a.x, a.y, b.x, b.y};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}

// Four consecutive outputs (16-byte aligned fp32 / 8-byte aligned bf16).
__device__ __forceinline__ void st4(float *p, const float (&x)[4]) {
  *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ void st4(__nv_bfloat16 *p, const float (&x)[4]) {
  *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]));
}

// bf16 K-major / MN-major SW128 element stores
__device__ __forceinline__ void st_bf16x8(uint8_t *tile, uint32_t off, const float (&x)[8]) {
  *reinterpret_cast<uint4 *>(tile + off) =
      make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}

template <typename Tdq>
__global__ void __launch_bounds__(NT, 1)
tc_bwd_intra_kernel(const __grid_constant__ CUtensorMap map_do, TcIntraArgs a, SeqInfo s, int H, int Hk,
                    GateParams gp, int64_t nitems) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *sG = reinterpret_cast<float *>(sm + S_G);
  const __nv_bfloat16 *sQR = reinterpret_cast<const __nv_bfloat16 *>(sm + S_QR);
  const __nv_bfloat16 *sKR = reinterpret_cast<const __nv_bfloat16 *>(sm + S_KR);
  float *sQF = reinterpret_cast<float *>(sm + S_QF);
  float *sDF = reinterpret_cast<float *>(sm + S_DF);
  float *sB = reinterpret_cast<float *>(sm + M_BETA);
  float *sRq = reinterpret_cast<float *>(sm + M_RQ);
  float *sRk = reinterpret_cast<float *>(sm + M_RK);
  float *sDB = reinterpret_cast<float *>(sm + M_DB);
  float *sSRed = reinterpret_cast<float *>(sm + M_SRED);
  float *sQD = reinterpret_cast<float *>(sm + M_QD);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + M_BAR);  // [0] loads, [1..9] MMA groups
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + M_TSLOT);
  volatile uint32_t *abort_flag = tslot + 1;
  uint8_t *R = sm + S_R;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q4 = warp & 3, hf = warp >> 2;
  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;
  const bool sig = (gp.flags & KDA_BETA_SIGMOID) != 0;
  const bool l2n = (gp.flags & KDA_L2NORM_QK) != 0;
  const bool has_do = a.d_out != nullptr;
  const float scale = gp.scale;
  const __nv_bfloat16 *qin = static_cast<const __nv_bfloat16 *>(a.q);
  const __nv_bfloat16 *kin = static_cast<const __nv_bfloat16 *>(a.k);
  const __nv_bfloat16 *vin = static_cast<const __nv_bfloat16 *>(a.v);

  if (warp == 0) {
    tc::tmem_alloc(tslot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int x = 0; x < NBAR; ++x) tc::mbar_init(bar + x, 1);
    tc::mbar_fence_init();
    *abort_flag = 0;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  int issued = 0;    // MMA groups of the current item started (thread 0), for the drain
  uint32_t par = 0;  // every barrier completes once per item: the item's parity

  // One persistent CTA per SM walks the (chunk, head) items, head fastest
  // (neighbouring CTAs share tokens); while it works on one item, the next
  // one's inputs and tile images are fetched into L2.
  for (int64_t w = blockIdx.x; w < nitems; w += gridDim.x, par ^= 1u) {
  const int64_t c = w / H;
  const int h = (int)(w % H);
  int n, len;
  int64_t t0;
  if (!chunk_lookup(s, c, n, t0, len)) break;  // items past the last chunk are all invalid
  const int hk = h / (H / Hk);
  const float A_h = gate ? tc::ex2(gp.a_log[h] * kLog2e) : 0.f;
  const size_t item = (size_t)w;
  auto tok = [&](int r, int heads, int head, int D) { return ((t0 + r) * heads + head) * (int64_t)D; };
  issued = 0;

  if (tid == 0) {
    // the previous item's accesses to the tile region precede these copies
    tc::fence_proxy_async_smem();
    // images of -dv_new, dw, v_new and the dO tile
    tc::mbar_arrive_expect_tx(bar, has_do ? 65536u : 49152u);
    bulk_load(R + R_DVN, a.dv_img + item * 16384, 16384, bar);
    bulk_load(R + R_DW, a.dw_img + item * 16384, 16384, bar);
    bulk_load(R + R_VN, a.vn_img + item * 16384, 16384, bar);
    if (has_do) {
      tma_load_3d(R + R_DO, &map_do, bar, 0, h, (int32_t)t0);
      tma_load_3d(R + R_DO + 8192, &map_do, bar, 64, h, (int32_t)t0);
    }
  }
  {  // the next item's q, k, v and gate rows (a thread each), A and images, into L2
    const int64_t wn = w + gridDim.x;
    int nn, lenn;
    int64_t t0n;
    if (wn < nitems && chunk_lookup(s, wn / H, nn, t0n, lenn)) {
      const int hn = (int)(wn % H), hkn = hn / (H / Hk), r = tid & 63, which = tid >> 6;
      if (r < lenn) {
        const int64_t t = t0n + r;
        if (which == 0) prefetch_l2(qin + (t * Hk + hkn) * K, K * 2);
        else if (which == 1) prefetch_l2(kin + (t * Hk + hkn) * K, K * 2);
        else if (which == 2) prefetch_l2(vin + (t * H + hn) * V, V * 2);
        else prefetch_l2(a.g + (t * H + hn) * K, K * 4);
      }
      if (tid == 0) {
        prefetch_l2(a.dv_img + (size_t)wn * 16384, 16384);
        prefetch_l2(a.dw_img + (size_t)wn * 16384, 16384);
        prefetch_l2(a.vn_img + (size_t)wn * 16384, 16384);
        prefetch_l2(a.a_in + (size_t)wn * (BT * BT), BT * BT * 4);
        if (has_do) {
          tma_prefetch_l2_3d(&map_do, 0, hn, (int32_t)t0n);
          tma_prefetch_l2_3d(&map_do, 64, hn, (int32_t)t0n);
        }
      }
    }
  }

  // ---- 0. every global load of the phase first (q, k, v rows; the gate
  //      input; A; beta), then the raw q, k rows to shared memory with their
  //      norms, and the gate in log2 units with its chunk-local inclusive
  //      cumsum (8-row groups in registers, then the groups' prefix)
  const int gc4 = 4 * lane;  // gate layout: rows 8 warp .. 8 warp + 7, channels gc4 .. gc4 + 3
  uint4 qv[4], kv[4], vv[4];
  float4 gx[8], av[4];
  float bload = 0.f;
#pragma unroll
  for (int it = 0; it < 4; ++it) {  // 16-byte groups of 8 channels: row (tid + 256 it) / 16
    const int i = tid + NT * it, r = i >> 4, c8 = (i & 15) * 8;
    qv[it] = kv[it] = vv[it] = make_uint4(0, 0, 0, 0);
    if (r < len) {
      qv[it] = *reinterpret_cast<const uint4 *>(qin + tok(r, Hk, hk, K) + c8);
      kv[it] = *reinterpret_cast<const uint4 *>(kin + tok(r, Hk, hk, K) + c8);
      vv[it] = *reinterpret_cast<const uint4 *>(vin + tok(r, H, h, V) + c8);
    }
  }
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    const int r = 8 * warp + x;
    gx[x] = r < len ? *reinterpret_cast<const float4 *>(a.g + tok(r, H, h, K) + gc4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int it = 0; it < 2; ++it) {  // A rows: 8 consecutive entries per thread and step
    const int i = tid + NT * it, r = i >> 3, j8 = (i & 7) * 8;
    av[2 * it] = av[2 * it + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < len) {
      const float4 *p = reinterpret_cast<const float4 *>(a.a_in + item * (BT * BT) + r * BT + j8);
      av[2 * it] = p[0];
      av[2 * it + 1] = p[1];
    }
  }
  if (tid < BT && tid < len) bload = a.beta[(t0 + tid) * H + h];

#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int i = tid + NT * it, r = i >> 4, c8 = (i & 15) * 8;
    uint2 *dq2 = reinterpret_cast<uint2 *>(sm + S_QR + r * (QS * 2) + c8 * 2);
    uint2 *dk2 = reinterpret_cast<uint2 *>(sm + S_KR + r * (QS * 2) + c8 * 2);
    dq2[0] = make_uint2(qv[it].x, qv[it].y);
    dq2[1] = make_uint2(qv[it].z, qv[it].w);
    dk2[0] = make_uint2(kv[it].x, kv[it].y);
    dk2[1] = make_uint2(kv[it].z, kv[it].w);
    // sums of squares over the row's 16 groups, held by 16 adjacent lanes
    const uint32_t qw[4] = {qv[it].x, qv[it].y, qv[it].z, qv[it].w};
    const uint32_t kw[4] = {kv[it].x, kv[it].y, kv[it].z, kv[it].w};
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fq = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qw[e]));
      const float2 fk = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kw[e]));
      sq = fmaf(fq.x, fq.x, fmaf(fq.y, fq.y, sq));
      sk = fmaf(fk.x, fk.x, fmaf(fk.y, fk.y, sk));
    }
#pragma unroll
    for (int o = 8; o; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if ((i & 15) == 0) {
      sRq[r] = l2n ? rsqrtf(sq + gp.eps) : 1.f;
      sRk[r] = l2n ? rsqrtf(sk + gp.eps) : 1.f;
    }
  }
  float Gl[8][4];
  {
    float dbl[4];  // dt_bias in log2 units
#pragma unroll
    for (int e = 0; e < 4; ++e) dbl[e] = (gate && gp.dt_bias) ? gp.dt_bias[h * K + gc4 + e] * kLog2e : 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const int r = 8 * warp + x;
      const float xs[4] = {gx[x].x, gx[x].y, gx[x].z, gx[x].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float g = xs[e] * kLog2e;
        if (gate) {
          // -exp(a_log) softplus(x + dt_bias), in log2 units
          const float z = fmaf(xs[e], kLog2e, dbl[e]);
          g = -A_h * (fmaxf(z, 0.f) + tc::lg2(1.f + tc::ex2(-fabsf(z))));
        }
        if (r >= len) g = 0.f;
        acc[e] += g;
        Gl[x][e] = acc[e];
      }
    }
    *reinterpret_cast<float4 *>(R + R_DA + (warp * 128 + gc4) * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  }
  if (tid < BT) {
    float b = bload;
    if (sig && tid < len) b = 1.f / (1.f + expf(-b));
    sB[tid] = b;
  }
  __syncthreads();
  {  // add the totals of the earlier 8-row groups
    const float *tot = reinterpret_cast<const float *>(R + R_DA);
    float pre[4] = {0.f, 0.f, 0.f, 0.f};
    for (int w2 = 0; w2 < warp; ++w2) {
      const float4 t = *reinterpret_cast<const float4 *>(tot + w2 * 128 + gc4);
      pre[0] += t.x; pre[1] += t.y; pre[2] += t.z; pre[3] += t.w;
    }
#pragma unroll
    for (int x = 0; x < 8; ++x)
      *reinterpret_cast<float4 *>(sG + (8 * warp + x) * GS + gc4) =
          make_float4(Gl[x][0] + pre[0], Gl[x][1] + pre[1], Gl[x][2] + pre[2], Gl[x][3] + pre[3]);
  }
  __syncthreads();
  auto qhat = [&](int r, int cc) { return __bfloat162float(sQR[r * QS + cc]) * sRq[r]; };
  auto khat = [&](int r, int cc) { return __bfloat162float(sKR[r * QS + cc]) * sRk[r]; };

  // ---- operands of M1 / M2: -v.beta, k^.beta.e^G (K-major [token][channel]),
  //      A (bf16, K-major [i][j])
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int i = tid + NT * it, r = i >> 4, c8 = (i & 15) * 8;
    float vb[8], kb[8];
    const uint32_t vw[4] = {vv[it].x, vv[it].y, vv[it].z, vv[it].w};
    const float br = sB[r];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vw[e]));
      vb[2 * e] = -br * f.x;
      vb[2 * e + 1] = -br * f.y;
    }
    float kr8[8], g8v[8];
    lds_bf8(sKR + r * QS + c8, kr8);
    lds_f8(sG + r * GS + c8, g8v);
    const float rk = sRk[r];
#pragma unroll
    for (int e = 0; e < 8; ++e) kb[e] = r < len ? kr8[e] * rk * br * tc::ex2(g8v[e]) : 0.f;
    st_bf16x8(R + R_VB, kmaj_off(64, r, c8), vb);
    st_bf16x8(R + R_KB, kmaj_off(64, r, c8), kb);
  }
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int i = tid + NT * it, r = i >> 3, j8 = (i & 7) * 8;
    const float x[8] = {av[2 * it].x, av[2 * it].y, av[2 * it].z, av[2 * it].w,
                        av[2 * it + 1].x, av[2 * it + 1].y, av[2 * it + 1].z, av[2 * it + 1].w};
    st_bf16x8(R + R_AT, kmaj_off(64, r, j8), x);
  }
  tc::fence_proxy_async_smem();
  bool ok = wait_or_flag(bar, par, a.err);
  if (!ok) *abort_flag = 1;
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();

  // ---- phase A: M1, M2, M4
  if (!*abort_flag && tid == 0) {
    const uint32_t dvn = tc::smem_u32(R + R_DVN), dw = tc::smem_u32(R + R_DW);
    const uint32_t vb = tc::smem_u32(R + R_VB), kb = tc::smem_u32(R + R_KB);
    const uint32_t at = tc::smem_u32(R + R_AT);
    const uint32_t i64 = tc::idesc_bf16_f32(64, 64, false, false);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {  // M1: dA (both products negated in the V half)
      const uint32_t ab = kk < 8 ? dvn : dw, bb = kk < 8 ? vb : kb, k8 = kk & 7;
      tc::mma_bf16(tmem + C_D1, tc::smem_desc_sw128(ab + (k8 >> 2) * 8192 + (k8 & 3) * 32, 16, 1024),
                   tc::smem_desc_sw128(bb + (k8 >> 2) * 8192 + (k8 & 3) * 32, 16, 1024), i64, kk > 0);
    }
    const uint32_t i256 = tc::idesc_bf16_f32(64, 256, true, true);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)  // M2: A^T [-dv_new | dw]
      tc::mma_bf16(tmem + C_D2, tc::smem_desc_sw128(at + kk * 2048, 8192, 1024),
                   tc::smem_desc_sw128(dvn + kk * 2048, 8192, 1024), i256, kk > 0);
    if (has_do) {
      const uint32_t o0 = tc::smem_u32(R + R_DO), v0 = tc::smem_u32(R + R_VN);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // M4: dO v_new^T
        tc::mma_bf16(tmem + C_D5, tc::smem_desc_sw128(o0 + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                     tc::smem_desc_sw128(v0 + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), i64, kk > 0);
    }
    tc::mma_commit(bar + 1);
    issued = 1;
  }
  // M=64 readout: row r = 16 q4 + lane (lanes < 16), columns in 16-column loads
  const int rr = 16 * q4 + lane;
  const bool rv = lane < 16;
  auto wait_mma = [&](int k) -> bool {
    __syncwarp();
    const bool ok = !*abort_flag && __all_sync(0xffffffffu, wait_or_flag(bar + k, par, a.err));
    if (!ok) *abort_flag = 1;
    tc::tc_fence_after();
    return ok;
  };
  if (wait_mma(1)) {
    // dA (j < i) -> bf16 MN-major B tile of M3a [i][j]; Q -> sQF; -dvb -> dv, dbeta part
    {
      float d[16];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int j0 = 32 * hf + 16 * cc;
        __syncwarp();
        tc::tmem_ld16(tmem + C_D1 + ((uint32_t)(32 * q4) << 16) + j0, d);
        tc::tmem_ld_wait();
        if (rv) {
          float x[8], y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            x[e] = (j0 + e < rr && rr < len) ? d[e] : 0.f;
            y[e] = (j0 + 8 + e < rr && rr < len) ? d[8 + e] : 0.f;
          }
          st_bf16x8(R + R_DA, mnmaj_off(64, rr, j0), x);
          st_bf16x8(R + R_DA, mnmaj_off(64, rr, j0 + 8), y);
        }
        __syncwarp();
        if (has_do) {
          tc::tmem_ld16(tmem + C_D5 + ((uint32_t)(32 * q4) << 16) + j0, d);
          tc::tmem_ld_wait();
        }
        if (rv)
#pragma unroll
          for (int e = 0; e < 16; e += 2)  // rows of FS floats are 8-byte aligned
            *reinterpret_cast<float2 *>(sQF + rr * FS + j0 + e) =
                make_float2((has_do && j0 + e <= rr && rr < len) ? scale * d[e] : 0.f,
                            (has_do && j0 + e + 1 <= rr && rr < len) ? scale * d[e + 1] : 0.f);
      }
      // -dv_new.beta: every lane works (lane l + 16 takes columns 8..15 of each
      // 16-column load of row 16 q4 + l); v rows loaded before the TMEM reads
      {
        const int row = 16 * q4 + (lane & 15), up = lane >> 4, s8 = 8 * up;
        const bool live = row < len;
        uint4 vraw[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          vraw[cc] = live ? *reinterpret_cast<const uint4 *>(vin + tok(row, H, h, V) + 64 * hf + 16 * cc + s8)
                          : make_uint4(0, 0, 0, 0);
        const float br = sB[row];
        float pb = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int v0 = 64 * hf + 16 * cc;
          __syncwarp();
          tc::tmem_ld16(tmem + C_D2 + ((uint32_t)(32 * q4) << 16) + v0, d);
          tc::tmem_ld_wait();
          float m[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float t = __shfl_sync(0xffffffffu, d[8 + e], lane & 15);
            m[e] = up ? t : d[e];
          }
          if (live) {
            const uint32_t vw[4] = {vraw[cc].x, vraw[cc].y, vraw[cc].z, vraw[cc].w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float dvb0 = -m[2 * e], dvb1 = -m[2 * e + 1];
              const float2 vf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vw[e]));
              pb = fmaf(dvb0, vf.x, fmaf(dvb1, vf.y, pb));
              const __nv_bfloat162 ob = __floats2bfloat162_rn(br * dvb0, br * dvb1);
              o[e] = *reinterpret_cast<const uint32_t *>(&ob);
            }
            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.dv) + tok(row, H, h, V) + v0 + s8) =
                make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        pb += __shfl_xor_sync(0xffffffffu, pb, 16);
        if (!up) sDB[row * 4 + hf] = pb;
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (tid < BT) sQD[tid] = sQF[tid * FS + tid];

  // ---- phase B: T = A^T dA, then dL = -T A^T
  if (!*abort_flag && tid == 0) {
    tc::tc_fence_after();
    const uint32_t at = tc::smem_u32(R + R_AT), da = tc::smem_u32(R + R_DA);
    const uint32_t id = tc::idesc_bf16_f32(64, 64, true, true);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      tc::mma_bf16(tmem + C_D1, tc::smem_desc_sw128(at + kk * 2048, 8192, 1024),
                   tc::smem_desc_sw128(da + kk * 2048, 8192, 1024), id, kk > 0);
    tc::mma_commit(bar + 2);
    issued = 2;
  }
  if (wait_mma(2)) {
    float d[16];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int q0 = 32 * hf + 16 * cc;
      __syncwarp();
      tc::tmem_ld16(tmem + C_D1 + ((uint32_t)(32 * q4) << 16) + q0, d);
      tc::tmem_ld_wait();
      if (rv) {
        float x[8], y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) { x[e] = d[e]; y[e] = d[8 + e]; }
        st_bf16x8(R + R_TT, kmaj_off(64, rr, q0), x);
        st_bf16x8(R + R_TT, kmaj_off(64, rr, q0 + 8), y);
      }
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  if (!*abort_flag && tid == 0) {
    tc::tc_fence_after();
    const uint32_t tt = tc::smem_u32(R + R_TT), at = tc::smem_u32(R + R_AT);
    const uint32_t id = tc::idesc_bf16_f32(64, 64, false, false);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      tc::mma_bf16(tmem + C_D5, tc::smem_desc_sw128(tt + kk * 32, 16, 1024),
                   tc::smem_desc_sw128(at + kk * 32, 16, 1024), id, kk > 0);
    tc::mma_commit(bar + 3);
    issued = 3;
  }
  if (wait_mma(3)) {
    float d[16];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int j0 = 32 * hf + 16 * cc;
      __syncwarp();
      tc::tmem_ld16(tmem + C_D5 + ((uint32_t)(32 * q4) << 16) + j0, d);
      tc::tmem_ld_wait();
      if (rv)
#pragma unroll
        for (int e = 0; e < 16; e += 2)
          *reinterpret_cast<float2 *>(sDF + rr * FS + j0 + e) =
              make_float2((j0 + e < rr && rr < len) ? -d[e] : 0.f, (j0 + e + 1 < rr && rr < len) ? -d[e + 1] : 0.f);
    }
  }
  tc::tc_fence_before();
  __syncthreads();

  // ---- phase C: row side.  A rows (K-major, K = 160 stacked segments) and
  //      the stacked right operand k^_j e^{G_rI - G_j} (MN-major, N = channels),
  //      its bf16 hi part then its lo part
  auto split = [](float x, bool lo) {
    const float hi = __bfloat162float(__float2bfloat16_rn(x));
    return lo ? x - hi : x;
  };
  for (int sub = 0; sub < 2; ++sub) {
    if (!*abort_flag) {
      if (sub == 0)
        for (int i = tid; i < BT * (KB_BIG / 8); i += NT) {  // [row][160 / 8] 16-byte groups, Q and dL rows
          // lanes run over rows: their reads of one column fall in different banks
          const int r = (i & 31) + 32 * ((i >> 5) & 1), g8 = (i >> 6) * 8, I = r >> 4, o = seg_off_row(I);
          float xq[8], xd[8];
          // tokens g8 - o .. g8 - o + 7 of row r's segment: the whole group lies
          // inside the segment or outside it (o and the segment length are
          // multiples of 8)
          const int jb = g8 - o;
          if (jb >= 0 && jb < 16 * (I + 1)) {
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const float2 qv2 = *reinterpret_cast<const float2 *>(sQF + r * FS + jb + e);
              const float2 dv2 = *reinterpret_cast<const float2 *>(sDF + r * FS + jb + e);
              xq[e] = jb + e < r ? qv2.x : 0.f;  // strictly below the diagonal
              xq[e + 1] = jb + e + 1 < r ? qv2.y : 0.f;
              xd[e] = dv2.x;
              xd[e + 1] = dv2.y;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) xq[e] = xd[e] = 0.f;
          }
          st_bf16x8(R + R_AQ, kmaj_off(64, r, g8), xq);
          st_bf16x8(R + R_AD, kmaj_off(64, r, g8), xd);
        }
      // stacked right operand: the first pass stores the hi part of all 160
      // rows and the lo part of rows 0..127 (to R_BLO); the second pass only
      // writes the lo part of rows 128..159 over the hi tile
      auto build_b = [&](int kr, int c8) {
        const int I = kr < 16 ? 0 : (kr < 48 ? 1 : (kr < 96 ? 2 : 3));
        const int j = kr - seg_off_row(I), ref = 16 * I;
        float x[8], lo[8], kr8[8], gr[8], gj[8];
        lds_bf8(sKR + j * QS + c8, kr8);
        lds_f8(sG + ref * GS + c8, gr);
        lds_f8(sG + j * GS + c8, gj);
        const float rk = sRk[j];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float2 dg = sub2(make_float2(gr[e], gr[e + 1]), make_float2(gj[e], gj[e + 1]));
          const float2 f = make_float2(tc::ex2(fminf(dg.x, 126.f)), tc::ex2(fminf(dg.y, 126.f)));
          float2 v = mul2(mul2(make_float2(kr8[e], kr8[e + 1]), splat2(rk)), f);
          if (j >= len) v = splat2(0.f);
          const float2 l = sub2(v, __bfloat1622float2(__float22bfloat162_rn(v)));  // v - bf16(v)
          lo[e] = l.x;
          lo[e + 1] = l.y;
          x[e] = sub ? l.x : v.x;
          x[e + 1] = sub ? l.y : v.y;
        }
        st_bf16x8(R + R_BB, mnmaj_off(KB_BIG, kr, c8), x);
        if (sub == 0 && kr < 128) st_bf16x8(R + R_BLO, mnmaj_off(128, kr, c8), lo);
      };
      if (sub == 0) {
        for (int i = tid; i < KB_BIG * 16; i += NT)  // [160 rows][128 / 8], lanes over rows
          build_b((i & 31) + 32 * ((i >> 5) % 5), ((i >> 5) / 5) * 8);
      } else {
        for (int i = tid; i < 32 * 16; i += NT) build_b(128 + (i & 31), (i >> 5) * 8);
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (!*abort_flag && tid == 0) {
      tc::tc_fence_after();
      const uint32_t aq = tc::smem_u32(R + R_AQ), ad = tc::smem_u32(R + R_AD), bb = tc::smem_u32(R + R_BB);
      const uint32_t id = tc::idesc_bf16_f32(64, 128, false, true);
      const uint32_t blo = tc::smem_u32(R + R_BLO);
#pragma unroll
      for (int kk = 0; kk < 10; ++kk) {
        const uint64_t bd = (sub == 1 && kk < 8) ? tc::smem_desc_sw128(blo + kk * 2048, 128 * 128, 1024)
                                                 : tc::smem_desc_sw128(bb + kk * 2048, KB_BIG * 128, 1024);
        tc::mma_bf16(tmem + C_D2, tc::smem_desc_sw128(aq + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), bd, id,
                     sub > 0 || kk > 0);
        tc::mma_bf16(tmem + C_D1, tc::smem_desc_sw128(ad + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), bd, id,
                     sub > 0 || kk > 0);
      }
      tc::mma_commit(bar + 4 + sub);
      issued = 4 + sub;
    }
    wait_mma(4 + sub);  // the operand region is rewritten next
    tc::tc_fence_before();
    __syncthreads();
  }

  // the fp32 rows the final readout reads (dq_g, dk_g), and the gate input
  // the gate backward reads again: fetched into L2 one phase ahead
  if (tid < len) {
    prefetch_l2(a.dqg + tok(tid, H, h, K), K * 4);
    prefetch_l2(a.dkg + tok(tid, H, h, K), K * 4);
    if (gate) prefetch_l2(a.g + tok(tid, H, h, K), K * 4);
  }

  // ---- phase D: column side, the dL part then the Q part; the right
  //      operand's hi and lo parts are built together
  for (int part = 0; part < 2; ++part) {
    if (!*abort_flag) {
      // A, MN-major [K slot][row j]: slot ks of rows j8 .. j8 + 7 (one 16-row
      // block J) holds token ii = ks - o + 16 J of their segment, i.e. eight
      // consecutive entries of row ii of dL (or Q); lanes run over K slots
      for (int i = tid; i < KB_BIG * 8; i += NT) {
        const int ks = i % KB_BIG, j8 = (i / KB_BIG) * 8, J = j8 >> 4, o = seg_off_col(J);
        const int ii = ks - o + 16 * J;
        float x[8];
        if (ks >= o && ks < o + 64 - 16 * J && ii < len) {
          const float *src = (part == 0 ? sDF : sQF) + ii * FS + j8;
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 v = *reinterpret_cast<const float2 *>(src + e);
            x[e] = ii > j8 + e ? v.x : 0.f;  // strictly below the diagonal
            x[e + 1] = ii > j8 + e + 1 ? v.y : 0.f;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
        st_bf16x8(R + R_AP, mnmaj_off(KB_BIG, ks, j8), x);
      }
      for (int i = tid; i < KB_BIG * 16; i += NT) {  // B hi and lo: [160 rows][128 / 8], lanes over rows
        const int kr = (i & 31) + 32 * ((i >> 5) % 5), c8 = ((i >> 5) / 5) * 8;
        const int J = kr < 64 ? 0 : (kr < 112 ? 1 : (kr < 144 ? 2 : 3));
        const int ii = kr - seg_off_col(J) + 16 * J, ref = 16 * J + 15;
        float xh[8], xl[8], raw[8], gi[8], gr[8];
        lds_bf8((part == 0 ? sKR : sQR) + ii * QS + c8, raw);
        lds_f8(sG + ii * GS + c8, gi);
        lds_f8(sG + ref * GS + c8, gr);
        const float rs = part == 0 ? sRk[ii] : sRq[ii], bs = sB[ii];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float2 dg = sub2(make_float2(gi[e], gi[e + 1]), make_float2(gr[e], gr[e + 1]));
          const float2 f = make_float2(tc::ex2(fminf(dg.x, 126.f)), tc::ex2(fminf(dg.y, 126.f)));
          float2 xs = mul2(make_float2(raw[e], raw[e + 1]), splat2(rs));
          if (part == 0) xs = mul2(splat2(bs), xs);
          float2 x = mul2(xs, f);
          if (ii >= len) x = splat2(0.f);
          const float2 l = sub2(x, __bfloat1622float2(__float22bfloat162_rn(x)));  // x - bf16(x)
          xh[e] = x.x;
          xh[e + 1] = x.y;
          xl[e] = l.x;
          xl[e + 1] = l.y;
        }
        st_bf16x8(R + R_BP, mnmaj_off(KB_BIG, kr, c8), xh);
        st_bf16x8(R + R_BPL, mnmaj_off(KB_BIG, kr, c8), xl);
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (!*abort_flag && tid == 0) {
      tc::tc_fence_after();
      const uint32_t ap = tc::smem_u32(R + R_AP), bh = tc::smem_u32(R + R_BP), bl = tc::smem_u32(R + R_BPL);
      const uint32_t id = tc::idesc_bf16_f32(64, 128, true, true);
#pragma unroll
      for (int kk = 0; kk < 20; ++kk) {
        const uint32_t k10 = kk % 10;
        tc::mma_bf16(tmem + C_D7, tc::smem_desc_sw128(ap + k10 * 2048, KB_BIG * 128, 1024),
                     tc::smem_desc_sw128((kk < 10 ? bh : bl) + k10 * 2048, KB_BIG * 128, 1024), id,
                     part > 0 || kk > 0);
      }
      tc::mma_commit(bar + 6 + part);
      issued = 6 + part;
    }
    wait_mma(6 + part);
    tc::tc_fence_before();
    __syncthreads();
  }

  // ---- final readout: row r, 64 columns per thread; dq^, dk^, dG (natural
  //      log units) and the dkg.kg parts into shared memory, dbeta parts
  float *fG = reinterpret_cast<float *>(R + R_FG), *fQ = reinterpret_cast<float *>(R + R_FQ);
  float *fK = reinterpret_cast<float *>(R + R_FK), *fP = sQF;  // fP [64][128] over sQF / sDF
  if (!*abort_flag) {
    // every lane works: lane l < 16 and lane l + 16 share row 16 q4 + l, the
    // upper lane taking columns 8..15 of each 16-column load
    const int row = 16 * q4 + (lane & 15), up = lane >> 4, s8 = 8 * up;
    float2 pb2 = splat2(0.f);
    const int rI = 16 * (row >> 4), rJ = rI + 15;
    const float br = sB[row], qd = sQD[row];
    const bool live = row < len;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      const int c0 = 64 * hf + 16 * cc;
      float dq6[16], dd6[16], d7[16], dkb[16];
      const uint32_t lanes = (uint32_t)(32 * q4) << 16;
      __syncwarp();
      tc::tmem_ld16(tmem + C_D2 + lanes + c0, dq6);        // row side, Q rows
      tc::tmem_ld16(tmem + C_D1 + lanes + c0, dd6);        // row side, dL rows
      tc::tmem_ld16(tmem + C_D7 + lanes + c0, d7);         // column side
      tc::tmem_ld16(tmem + C_D2 + 128 + lanes + c0, dkb);  // A^T dw (kept from phase A)
      float dqgv[8], dkgv[8];
      if (live) {
        const float4 *pq = reinterpret_cast<const float4 *>(a.dqg + tok(row, H, h, K) + c0 + s8);
        const float4 *pk = reinterpret_cast<const float4 *>(a.dkg + tok(row, H, h, K) + c0 + s8);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const float4 u = pq[x], w = pk[x];
          dqgv[4 * x] = u.x; dqgv[4 * x + 1] = u.y; dqgv[4 * x + 2] = u.z; dqgv[4 * x + 3] = u.w;
          dkgv[4 * x] = w.x; dkgv[4 * x + 1] = w.y; dkgv[4 * x + 2] = w.z; dkgv[4 * x + 3] = w.w;
        }
      }
      tc::tmem_ld_wait();
      float mq[8], md[8], m7[8], mk[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float tq = __shfl_sync(0xffffffffu, dq6[8 + e], lane & 15);
        const float td = __shfl_sync(0xffffffffu, dd6[8 + e], lane & 15);
        const float t7 = __shfl_sync(0xffffffffu, d7[8 + e], lane & 15);
        const float tk = __shfl_sync(0xffffffffu, dkb[8 + e], lane & 15);
        mq[e] = up ? tq : dq6[e];
        md[e] = up ? td : dd6[e];
        m7[e] = up ? t7 : d7[e];
        mk[e] = up ? tk : dkb[e];
      }
#pragma unroll
      for (int e4 = 0; e4 < 8; e4 += 4) {
        const int cb = c0 + s8 + e4;  // first of this step's four columns
        float oq[4] = {0.f, 0.f, 0.f, 0.f}, ok[4] = {0.f, 0.f, 0.f, 0.f};
        float og[4] = {0.f, 0.f, 0.f, 0.f}, op[4] = {0.f, 0.f, 0.f, 0.f};
        if (live) {
          const float4 G4 = *reinterpret_cast<const float4 *>(sG + row * GS + cb);
          const float4 C4 = *reinterpret_cast<const float4 *>(sG + (len - 1) * GS + cb);
          const float4 I4 = *reinterpret_cast<const float4 *>(sG + rI * GS + cb);
          const float4 J4 = *reinterpret_cast<const float4 *>(sG + rJ * GS + cb);
          const uint2 qr = *reinterpret_cast<const uint2 *>(sQR + row * QS + cb);
          const uint2 kr = *reinterpret_cast<const uint2 *>(sKR + row * QS + cb);
          const float Gv[4] = {G4.x, G4.y, G4.z, G4.w}, Cv[4] = {C4.x, C4.y, C4.z, C4.w};
          const float Iv[4] = {I4.x, I4.y, I4.z, I4.w}, Jv[4] = {J4.x, J4.y, J4.z, J4.w};
          const float2 q01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qr.x));
          const float2 q23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qr.y));
          const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr.x));
          const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr.y));
          const float qv[4] = {q01.x, q01.y, q23.x, q23.y}, kv4[4] = {k01.x, k01.y, k23.x, k23.y};
          const float rq = sRq[row], rk = sRk[row];
#pragma unroll
          for (int x = 0; x < 4; x += 2) {  // two columns at a time (paired fp32)
            const int e = e4 + x;
            auto pr = [&](const float *v, int i) { return make_float2(v[i], v[i + 1]); };
            const float2 G = pr(Gv, x);
            const float2 dI = sub2(G, pr(Iv, x)), dJ = sub2(pr(Jv, x), G), dC = sub2(pr(Cv, x), G);
            const float2 fq = make_float2(tc::ex2(dI.x), tc::ex2(dI.y));                        // <= 1
            const float2 fc = make_float2(tc::ex2(fminf(dJ.x, 0.f)), tc::ex2(fminf(dJ.y, 0.f)));  // <= 1
            const float2 eG = make_float2(tc::ex2(G.x), tc::ex2(G.y));
            const float2 ekg = make_float2(tc::ex2(dC.x), tc::ex2(dC.y));
            const float2 qh = mul2(pr(qv, x), splat2(rq)), kh = mul2(pr(kv4, x), splat2(rk));
            const float2 mke = pr(mk, e), fmd = mul2(fq, pr(md, e));
            const float2 aq = mul2(fq, pr(mq, e)), akr = mul2(splat2(br), fmd), akc = mul2(fc, pr(m7, e));
            const float2 dqs = mul2(pr(dqgv, e), splat2(scale)), dkg = pr(dkgv, e);
            const float2 kbf = mul2(splat2(br), eG);
            const float2 dkh = mul2(dkg, kh);
            const float2 vq = fma2(dqs, eG, fma2(splat2(qd), kh, aq));
            const float2 vk = fma2(dkg, ekg, fma2(mke, kbf, fma2(splat2(qd), qh, add2(akr, akc))));
            const float2 vp = mul2(dkh, ekg);
            float2 vg = fma2(kh, sub2(akr, akc), mul2(qh, aq));
            vg = fma2(mul2(dqs, qh), eG, fma2(mul2(mke, kh), kbf, vg));
            vg = sub2(vg, vp);
            pb2 = fma2(mke, mul2(kh, eG), fma2(kh, fmd, pb2));
            oq[x] = vq.x; oq[x + 1] = vq.y;
            ok[x] = vk.x; ok[x + 1] = vk.y;
            og[x] = vg.x; og[x + 1] = vg.y;
            op[x] = vp.x; op[x + 1] = vp.y;
          }
        }
        *reinterpret_cast<float4 *>(fQ + row * GS + cb) = make_float4(oq[0], oq[1], oq[2], oq[3]);
        *reinterpret_cast<float4 *>(fK + row * GS + cb) = make_float4(ok[0], ok[1], ok[2], ok[3]);
        *reinterpret_cast<float4 *>(fG + row * GS + cb) = make_float4(og[0], og[1], og[2], og[3]);
        *reinterpret_cast<float4 *>(fP + row * GS + cb) = make_float4(op[0], op[1], op[2], op[3]);
      }
    }
    float pb = pb2.x + pb2.y;
    pb += __shfl_xor_sync(0xffffffffu, pb, 16);
    if (!up) sDB[row * 4 + 2 + hf] = pb;
  }
  __syncthreads();

  // global inputs of the last two passes, loaded ahead of them: the chunk-end
  // gate gradient term of this thread's channel and the gate input rows
  const int gc4b = (tid & 31) * 4, grg = tid >> 5;  // gate pass: channels gc4b .., rows grg + 8 m
  float dgc0 = 0.f;
  float4 gxg[8];
  {
    const bool go = !*abort_flag;
    if (go) dgc0 = a.dgc[item * K + (tid & 127)];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int r = grg + 8 * m;
      gxg[m] = (go && gate && r < len) ? *reinterpret_cast<const float4 *>(a.g + tok(r, H, h, K) + gc4b)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  // ---- L2-norm backward: dx = r (dx^ - x^ (x^ . dx^)), one warp per row
  //      (lane = four consecutive channels), two rows (r, r + 8) at a time
  if (!*abort_flag) {
    const int c4n = 4 * lane;
    for (int r0 = warp; r0 < len; r0 += 16) {
      float xq[2][4], xk[2][4], gq[2][4], gk[2][4], pq[2], pk[2];
#pragma unroll
      for (int y = 0; y < 2; ++y) {
        const int r = r0 + 8 * y < len ? r0 + 8 * y : r0;  // a row past the end reads row r0 (unused)
        const uint2 qr = *reinterpret_cast<const uint2 *>(sQR + r * QS + c4n);
        const uint2 kr = *reinterpret_cast<const uint2 *>(sKR + r * QS + c4n);
        const float4 fq4 = *reinterpret_cast<const float4 *>(fQ + r * GS + c4n);
        const float4 fk4 = *reinterpret_cast<const float4 *>(fK + r * GS + c4n);
        const float2 q01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qr.x));
        const float2 q23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qr.y));
        const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr.x));
        const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr.y));
        const float rq = sRq[r], rk = sRk[r];
        xq[y][0] = q01.x * rq; xq[y][1] = q01.y * rq; xq[y][2] = q23.x * rq; xq[y][3] = q23.y * rq;
        xk[y][0] = k01.x * rk; xk[y][1] = k01.y * rk; xk[y][2] = k23.x * rk; xk[y][3] = k23.y * rk;
        gq[y][0] = fq4.x; gq[y][1] = fq4.y; gq[y][2] = fq4.z; gq[y][3] = fq4.w;
        gk[y][0] = fk4.x; gk[y][1] = fk4.y; gk[y][2] = fk4.z; gk[y][3] = fk4.w;
        pq[y] = fmaf(xq[y][3], gq[y][3], fmaf(xq[y][2], gq[y][2], fmaf(xq[y][1], gq[y][1], xq[y][0] * gq[y][0])));
        pk[y] = fmaf(xk[y][3], gk[y][3], fmaf(xk[y][2], gk[y][2], fmaf(xk[y][1], gk[y][1], xk[y][0] * gk[y][0])));
      }
#pragma unroll
      for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int y = 0; y < 2; ++y) {
          pq[y] += __shfl_xor_sync(0xffffffffu, pq[y], o);
          pk[y] += __shfl_xor_sync(0xffffffffu, pk[y], o);
        }
#pragma unroll
      for (int y = 0; y < 2; ++y) {
        const int r = r0 + 8 * y;
        if (r >= len) continue;
        const float sq = l2n ? pq[y] : 0.f, sk = l2n ? pk[y] : 0.f;
        const float rq = sRq[r], rk = sRk[r];
        float oq[4], ok[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          oq[x] = rq * (gq[y][x] - xq[y][x] * sq);
          ok[x] = rk * (gk[y][x] - xk[y][x] * sk);
        }
        const int64_t off = tok(r, H, h, K) + c4n;  // per value head (summed over the group later)
        st4(static_cast<Tdq *>(a.dq) + off, oq);
        st4(static_cast<Tdq *>(a.dk) + off, ok);
      }
    }
  }

  // ---- reverse cumsum over the chunk (dG_C onto every row): fG <- the
  //      gradient of the natural-log gate g of each token.  Thread = (channel,
  //      half of the chunk); the halves exchange their sums of fP and fG.
  {
    float *sHalf = reinterpret_cast<float *>(R + R_FK + 64 * GS * 4);  // [2 halves][fP, fG][128]
    const int cch = tid & 127, hb = tid >> 7, rb = 32 * hb;
    float gv[32];
    float sp = 0.f, sg = 0.f;
    if (!*abort_flag) {
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const bool in = rb + x < len;
        gv[x] = in ? fG[(rb + x) * GS + cch] : 0.f;
        sp += in ? fP[(rb + x) * GS + cch] : 0.f;
      }
#pragma unroll
      for (int x = 0; x < 32; ++x) sg += gv[x];
      sHalf[(2 * hb) * 128 + cch] = sp;
      sHalf[(2 * hb + 1) * 128 + cch] = sg;
    }
    __syncthreads();
    if (!*abort_flag) {
      const float GC = sG[(len - 1) * GS + cch];
      float run = dgc0 * tc::ex2(GC) + sHalf[cch] + sHalf[256 + cch];
      if (hb == 0) run += sHalf[384 + cch];  // fG of the later half
#pragma unroll
      for (int x = 31; x >= 0; --x) {
        run += gv[x];
        if (rb + x < len) fG[(rb + x) * GS + cch] = run;
      }
    }
  }
  __syncthreads();
  // ---- gate backward, all threads (4 channels x every 8th row each):
  //      dz = -exp(a_log) sigmoid(z) dg, z = x + dt_bias; dA_log, ddt_bias parts
  float alog = 0.f;
  float *sPart = fQ;  // [8][128] ddt_bias parts (fQ is free after the norm backward)
  {
    const int c4 = gc4b, rg = grg;
    float dtb[4] = {0.f, 0.f, 0.f, 0.f}, bias[4] = {0.f, 0.f, 0.f, 0.f};
    if (gate && gp.dt_bias)
#pragma unroll
      for (int e = 0; e < 4; ++e) bias[e] = gp.dt_bias[h * K + c4 + e];
    if (!*abort_flag) {
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int r = rg + 8 * m;
        if (r < len) {
          const float xs[4] = {gxg[m].x, gxg[m].y, gxg[m].z, gxg[m].w};
          float o[4];
          const float4 dg4 = *reinterpret_cast<const float4 *>(fG + r * GS + c4);
          const float dgv[4] = {dg4.x, dg4.y, dg4.z, dg4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float dgn = dgv[e];
            if (gate) {
              // t = e^{-|z|}: sigmoid(z) = (z >= 0 ? 1 : t) / (1 + t),
              // softplus(z) = max(z, 0) + ln(1 + t)
              const float z = xs[e] + bias[e];
              const float t = tc::ex2(-fabsf(z) * kLog2e);
              const float sgm = __fdividef(z >= 0.f ? 1.f : t, 1.f + t);
              const float spl = fmaxf(z, 0.f) + tc::lg2(1.f + t) * kLn2;
              const float dz = -A_h * dgn * sgm;
              o[e] = dz;
              dtb[e] += dz;
              alog = fmaf(-A_h * spl, dgn, alog);
            } else {
              o[e] = dgn;
            }
          }
          *reinterpret_cast<float4 *>(a.dg + tok(r, H, h, K) + c4) = make_float4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    if (gate)
#pragma unroll
      for (int e = 0; e < 4; ++e) sPart[rg * K + c4 + e] = dtb[e];
  }
  if (gate) {
    for (int o = 16; o; o >>= 1) alog += __shfl_xor_sync(0xffffffffu, alog, o);
    if (lane == 0) sSRed[warp] = alog;
  }
  __syncthreads();
  if (!*abort_flag && gate && tid < K) {
    float d = 0.f;
    for (int x = 0; x < 8; ++x) d += sPart[x * K + tid];
    a.part_dtb[item * K + tid] = d;
    if (tid == 0) {
      float al = 0.f;
      for (int x = 0; x < 8; ++x) al += sSRed[x];
      a.part_alog[item] = al;
    }
  }
  // ---- beta: parts from -v.beta (phase A) and the final readout; sigmoid backward
  if (!*abort_flag && tid < len) {
    const float d = sDB[tid * 4] + sDB[tid * 4 + 1] + sDB[tid * 4 + 2] + sDB[tid * 4 + 3];
    const float b = sB[tid];
    a.dbeta[(t0 + tid) * H + h] = sig ? d * b * (1.f - b) : d;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (*abort_flag) break;
  }  // items

  if (*abort_flag && tid == 0) {  // bounded drain of the loads and MMAs of the item given up on
    drain_wait(bar, par);
    for (int x = 1; x <= issued; ++x) drain_wait(bar + x, par);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_tc_bwd_intra(const TcIntraArgs &a, const SeqInfo &s, int64_t nchunks, int H, int Hk,
                                const GateParams &gp, cudaStream_t st) {
  if (nchunks == 0 || H == 0) return cudaSuccess;
  CUtensorMap map_do;
  memset(&map_do, 0, sizeof(map_do));  // not read without d_out
  if (a.d_out && (s.T_tot <= 0 || !make_value_map(a.d_out, s.T_tot, H, map_do))) return cudaErrorInvalidValue;
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  const int64_t nitems = nchunks * H;
  dim3 grid((unsigned)(nitems < sms ? nitems : sms));  // persistent: one CTA per SM
  cudaError_t e;
  if (a.dq_is_f32) {
    e = cudaFuncSetAttribute(tc_bwd_intra_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    tc_bwd_intra_kernel<float><<<grid, NT, SMEM_BYTES, st>>>(map_do, a, s, H, Hk, gp, nitems);
  } else {
    e = cudaFuncSetAttribute(tc_bwd_intra_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    tc_bwd_intra_kernel<__nv_bfloat16><<<grid, NT, SMEM_BYTES, st>>>(map_do, a, s, H, Hk, gp, nitems);
  }
  return cudaGetLastError();
}

}  // namespace tcp
}  // namespace kda
