// kda_bwd.cu - chunked KDA backward on CUDA cores (fp32 arithmetic).
//
// Gradients of L = <d_out, o> + <d_final, S_final> with respect to q, k, v,
// beta, the gate input, a_log, dt_bias and the initial state, following the
// six-stage decomposition of "KDA Chunk Backward - TPU/Pallas Kernel Design"
// section 2 (recompute, dAv, reverse state-gradient chain, WY backward,
// intra-chunk backward, reverse cumsum, then gate / L2-norm backward):
//
//   recompute   the forward's per-chunk w, u, qg (= scale q^ e^G),
//               kg (= k^ e^{G_C - G}), Aqk, e^{G_C} and the state h entering
//               every chunk and v_new (the generic forward kernels)
//   bwd_dh      per (sequence, head, 32-column tile), chunks in reverse:
//                 dv_new = Aqk^T dO + kg dh'
//                 dh     = e^{G_C} . dh' + qg^T dO - w^T dv_new
//               (dh' = gradient of the state leaving the chunk; the last is
//               d_final, the first dh is the initial-state gradient)
//   bwd_state   per (chunk, head): d(qg) = dO h^T, dw = -dv_new h^T,
//               dkg = v_new dh'^T, d(e^{G_C}) = sum_v dh' . h
//   bwd_intra   per (chunk, head): dA = dv_new (v.beta)^T + dw (k^.beta.e^G)^T,
//               the triangular inverse backward dL = -A^T dA A^T,
//               dAqk = dO v_new^T, the pairwise terms of L and Aqk over
//               channels, the elementwise terms of qg, kg, w, u, the reverse
//               cumulative sum over the chunk, then the L2-norm, sigmoid and
//               gate backward
//   reductions  dA_log, ddt_bias over chunks; dq, dk over the value heads
//               that share a key head
// All gates are natural-log here (the base-2 form of the forward is only a
// change of base, section 3.1).
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

constexpr int VT = 32;  // column tile of the reverse state-gradient chain

// ---------------------------------------------------------------------------
// Reverse chain of the state gradient: one CTA per (range, head, column tile).
// ---------------------------------------------------------------------------
template <typename Tin, int K>
__global__ void __launch_bounds__(256)
bwd_dh_kernel(SeqInfo s, int H, int V, const float *__restrict__ w, const float *__restrict__ qg,
              const float *__restrict__ kg, const float *__restrict__ aqk,
              const float *__restrict__ gc, const Tin *__restrict__ d_out,
              const float *__restrict__ d_final, float *__restrict__ dhn, float *__restrict__ dvn,
              float *__restrict__ d_initial) {
  extern __shared__ float smem[];
  float *sD = smem;            // [K][VT]  gradient of the state leaving the chunk
  float *sW = sD + K * VT;     // [64][K]
  float *sQg = sW + BT * K;    // [64][K]
  float *sKg = sQg + BT * K;   // [64][K]
  float *sO = sKg + BT * K;    // [64][VT] d_out
  float *sDv = sO + BT * VT;   // [64][VT] dv_new
  float *sA = sDv + BT * VT;   // [64][64] Aqk
  float *sGc = sA + BT * BT;   // [K]      e^{G_C}

  const int n = blockIdx.x / H, h = blockIdx.x % H;
  const int tid = threadIdx.x, j = tid & (VT - 1), rb = tid >> 5;
  const int col = blockIdx.y * VT + j;
  int64_t t0, t1;
  seq_range(s, n, t0, t1);
  const int64_t c0 = seq_first_chunk(s, n);
  const int64_t nch = (t1 - t0 + BT - 1) / BT;
  const int64_t unit = (int64_t)n * H + h;

  for (int cc = rb; cc < K; cc += 8)
    sD[cc * VT + j] = d_final ? d_final[(unit * K + cc) * V + col] : 0.f;

  for (int64_t ci = c0 + nch - 1; ci >= c0; --ci) {
    const int64_t t = t0 + (ci - c0) * BT;
    const int len = (int)((t1 - t) < BT ? (t1 - t) : BT);
    __syncthreads();  // the previous chunk is done with the tiles
    for (int i = tid; i < BT * K; i += 256) {
      const int r = i / K, cc = i % K;
      const bool in = r < len;
      const int64_t off = ((t + r) * H + h) * (int64_t)K + cc;
      sW[i] = in ? w[off] : 0.f;
      sQg[i] = in ? qg[off] : 0.f;
      sKg[i] = in ? kg[off] : 0.f;
    }
    for (int r = rb; r < BT; r += 8)
      sO[r * VT + j] = (r < len && d_out) ? to_f32(d_out[((t + r) * H + h) * (int64_t)V + col]) : 0.f;
    for (int i = tid; i < BT * BT; i += 256) {
      const int r = i / BT;
      sA[i] = r < len ? aqk[((t + r) * H + h) * BT + (i % BT)] : 0.f;
    }
    for (int cc = tid; cc < K; cc += 256) sGc[cc] = gc[(ci * H + h) * K + cc];
    if (dhn)
      for (int cc = rb; cc < K; cc += 8) dhn[((ci * H + h) * K + cc) * V + col] = sD[cc * VT + j];
    __syncthreads();

    // dv_new = Aqk^T dO + kg dh'
    for (int r = rb; r < BT; r += 8) {
      float acc = 0.f;
      if (r < len) {
        for (int s2 = r; s2 < len; ++s2) acc = fmaf(sA[s2 * BT + r], sO[s2 * VT + j], acc);
        for (int cc = 0; cc < K; ++cc) acc = fmaf(sKg[r * K + cc], sD[cc * VT + j], acc);
        if (dvn) dvn[((t + r) * H + h) * (int64_t)V + col] = acc;
      }
      sDv[r * VT + j] = acc;
    }
    __syncthreads();

    // dh = e^{G_C} . dh' + qg^T dO - w^T dv_new
    for (int cc = rb; cc < K; cc += 8) {
      float acc = sGc[cc] * sD[cc * VT + j];
      for (int r = 0; r < len; ++r) {
        acc = fmaf(sQg[r * K + cc], sO[r * VT + j], acc);
        acc = fmaf(-sW[r * K + cc], sDv[r * VT + j], acc);
      }
      sD[cc * VT + j] = acc;
    }
  }
  __syncthreads();
  if (d_initial)
    for (int cc = rb; cc < K; cc += 8) d_initial[(unit * K + cc) * V + col] = sD[cc * VT + j];
}

// ---------------------------------------------------------------------------
// State-contraction terms: one CTA per (chunk, head); thread = (channel,
// every NP-th row).
// ---------------------------------------------------------------------------
template <typename Tin, int K>
__global__ void __launch_bounds__(256)
bwd_state_kernel(SeqInfo s, int H, int V, const float *__restrict__ hst,
                 const float *__restrict__ dhn, const Tin *__restrict__ d_out,
                 const float *__restrict__ dvn, const float *__restrict__ vn,
                 float *__restrict__ dqg, float *__restrict__ dw, float *__restrict__ dkg,
                 float *__restrict__ dgc) {
  constexpr int NP = 256 / K, NR = BT / NP, KP = K + 1;
  extern __shared__ float smem[];
  float *sH = smem;            // [VT][K+1]  h, column-major in the tile
  float *sDh = sH + VT * KP;   // [VT][K+1]  dh'
  float *sO = sDh + VT * KP;   // [64][VT]
  float *sDv = sO + BT * VT;   // [64][VT]
  float *sVn = sDv + BT * VT;  // [64][VT]

  const int64_t c = blockIdx.x;
  const int h = blockIdx.y;
  int n, len;
  int64_t t0;
  if (!chunk_lookup(s, c, n, t0, len)) return;
  const int tid = threadIdx.x, cc = tid % K, part = tid / K;
  float aq[NR], aw[NR], ak[NR], agc = 0.f;
#pragma unroll
  for (int m = 0; m < NR; ++m) aq[m] = aw[m] = ak[m] = 0.f;

  for (int v0 = 0; v0 < V; v0 += VT) {
    __syncthreads();
    for (int i = tid; i < K * VT; i += 256) {
      const int r = i / VT, jj = i % VT;
      const int64_t off = ((c * H + h) * K + r) * (int64_t)V + v0 + jj;
      sH[jj * KP + r] = hst[off];
      sDh[jj * KP + r] = dhn[off];
    }
    for (int i = tid; i < BT * VT; i += 256) {
      const int r = i / VT, jj = i % VT;
      const bool in = r < len;
      const int64_t off = ((t0 + r) * H + h) * (int64_t)V + v0 + jj;
      sO[i] = (in && d_out) ? to_f32(d_out[off]) : 0.f;
      sDv[i] = in ? dvn[off] : 0.f;
      sVn[i] = in ? vn[off] : 0.f;
    }
    __syncthreads();
    for (int jj = 0; jj < VT; ++jj) {
      const float hv = sH[jj * KP + cc], dh = sDh[jj * KP + cc];
      agc = fmaf(dh, hv, agc);
#pragma unroll
      for (int m = 0; m < NR; ++m) {
        const int r = part + NP * m;
        aq[m] = fmaf(sO[r * VT + jj], hv, aq[m]);
        aw[m] = fmaf(-sDv[r * VT + jj], hv, aw[m]);
        ak[m] = fmaf(sVn[r * VT + jj], dh, ak[m]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < NR; ++m) {
    const int r = part + NP * m;
    if (r < len) {
      const int64_t off = ((t0 + r) * H + h) * (int64_t)K + cc;
      dqg[off] = aq[m];
      dw[off] = aw[m];
      dkg[off] = ak[m];
    }
  }
  if (part == 0) dgc[(c * H + h) * K + cc] = agc;
}

// ---------------------------------------------------------------------------
// Intra-chunk backward: one CTA per (chunk, head).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float softplus_f(float z) { return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))); }

// Row-pair mapping of a 64 x 64 product: thread -> row i = tid / 4, columns
// j = (tid & 3) + 4 m.
template <int K, int V>
struct IntraSmem {
  static constexpr int KP = K + 1, XP = (K > V ? K : V) + 1;
  static constexpr int oQ = 0, oK = oQ + BT * KP, oG = oK + BT * KP;
  static constexpr int oX = oG + BT * KP, oY = oX + BT * XP;
  static constexpr int oA = oY + BT * XP, oP = oA + BT * 65, oM = oP + BT * 65;
  static constexpr int oB = oM + BT * 65, oRq = oB + BT, oRk = oRq + BT;
  static constexpr int oRedV = oRk + BT;            // [64][4]  dbeta parts over v
  static constexpr int oRedK = oRedV + BT * 4;      // [64][4]  dbeta parts over channels
  static constexpr int oRedC = oRedK + BT * 4;      // [4][K]   dG_C parts
  static constexpr int oRedS = oRedC + 4 * K;       // [8]      dA_log parts
  static constexpr int total = oRedS + 8;
};

// The tensor-core path's bf16 tile images of -dv_new, v_new and dw (16 KB
// per (chunk, head), [token][column] in the 64-row MN-major SW128 layout),
// and the list of the items to process, for the list mode of
// bwd_intra_kernel; unused (null) otherwise.
struct ImgSrc {
  const uint8_t *dvn_neg, *vn, *dw;
  const uint32_t *count, *list;
};

__device__ __forceinline__ float img_at(const uint8_t *img, int64_t item, int r, int col) {
  return __bfloat162float(
      *reinterpret_cast<const __nv_bfloat16 *>(img + item * 16384 + tcp::mnmaj_off(64, r, col)));
}

// LIST = false: one CTA per (chunk, head) of the grid, fp32 intermediates.
// LIST = true: the CTAs loop over the items of img.list (chunk * H + head)
// and read dv_new, v_new and dw from img's tile images - the exact pass over
// the chunks the tensor-core kernel cannot take (strong decay).
template <typename Tin, typename Tdq, int K, int V, bool LIST = false>
__global__ void __launch_bounds__(256, 1)
bwd_intra_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                 const float *__restrict__ g, const float *__restrict__ beta, GateParams gp,
                 SeqInfo s, int H, int Hk, const Tin *__restrict__ d_out,
                 const float *__restrict__ dvn, const float *__restrict__ vn,
                 const float *__restrict__ dqg, const float *__restrict__ dw,
                 const float *__restrict__ dkg, const float *__restrict__ dgc,
                 Tdq *__restrict__ dq_out, Tdq *__restrict__ dk_out, Tin *__restrict__ dv_out,
                 float *__restrict__ dg_out, float *__restrict__ dbeta_out,
                 float *__restrict__ part_alog, float *__restrict__ part_dtb,
                 const float *__restrict__ a_in, ImgSrc img) {
  using L = IntraSmem<K, V>;
  constexpr int KP = L::KP, XP = L::XP;
  constexpr int NP = 256 / K, NR = BT / NP;  // channel mapping: rows part + NP m
  constexpr int NPV = 256 / V;               // column mapping over v
  extern __shared__ float smem[];
  float *sQ = smem + L::oQ, *sK = smem + L::oK, *sG = smem + L::oG;
  float *X = smem + L::oX, *Y = smem + L::oY;
  float *sA = smem + L::oA, *sP = smem + L::oP, *sM = smem + L::oM;
  float *sB = smem + L::oB, *sRq = smem + L::oRq, *sRk = smem + L::oRk;
  float *sRedV = smem + L::oRedV, *sRedK = smem + L::oRedK, *sRedC = smem + L::oRedC;
  float *sRedS = smem + L::oRedS;

  const uint32_t n_list = LIST ? *img.count : 1u;
  for (uint32_t li = LIST ? blockIdx.x : 0u; li < n_list; li += LIST ? gridDim.x : 1u) {
  if (LIST) __syncthreads();  // the previous item is done with shared memory
  const int64_t c = LIST ? (int64_t)(img.list[li] / (uint32_t)H) : (int64_t)blockIdx.x;
  const int h = LIST ? (int)(img.list[li] % (uint32_t)H) : (int)blockIdx.y;
  const int64_t item = c * H + h;
  int n, len;
  int64_t t0;
  if (!chunk_lookup(s, c, n, t0, len)) continue;  // uniform over the CTA
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hk = h / (H / Hk);
  const bool gate = (gp.flags & KDA_GATE_IN_KERNEL) != 0;
  const bool sig = (gp.flags & KDA_BETA_SIGMOID) != 0;
  const float A_h = gate ? expf(gp.a_log[h]) : 0.f;
  const float scale = gp.scale;
  auto row_off = [&](int r, int heads, int head, int D) {
    return ((t0 + r) * heads + head) * (int64_t)D;
  };

  // 1. q, k (raw), natural-log gate, beta (rows past the end are zero)
  for (int i = tid; i < BT * K; i += 256) {
    const int r = i / K, cc = i % K;
    float qv = 0.f, kv = 0.f, gv = 0.f;
    if (r < len) {
      qv = to_f32(q[row_off(r, Hk, hk, K) + cc]);
      kv = to_f32(k[row_off(r, Hk, hk, K) + cc]);
      gv = g[row_off(r, H, h, K) + cc];
      if (gate) gv = -A_h * softplus_f(gv + (gp.dt_bias ? gp.dt_bias[h * K + cc] : 0.f));
    }
    sQ[r * KP + cc] = qv;
    sK[r * KP + cc] = kv;
    sG[r * KP + cc] = gv;
  }
  if (tid < BT) {
    float b = 0.f;
    if (tid < len) {
      b = beta[(t0 + tid) * H + h];
      if (sig) b = 1.f / (1.f + expf(-b));
    }
    sB[tid] = b;
  }
  __syncthreads();

  // 2. row norms (q^ = q r_q), the chunk-local inclusive cumsum of the gate
  for (int r = warp; r < BT; r += 8) {
    float sq = 0.f, sk = 0.f;
    for (int cc = lane; cc < K; cc += 32) {
      const float a = sQ[r * KP + cc], b = sK[r * KP + cc];
      sq += a * a;
      sk += b * b;
    }
    for (int o = 16; o; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    const bool l2 = (gp.flags & KDA_L2NORM_QK) != 0;
    const float rq = l2 ? rsqrtf(sq + gp.eps) : 1.f, rk = l2 ? rsqrtf(sk + gp.eps) : 1.f;
    for (int cc = lane; cc < K; cc += 32) {
      sQ[r * KP + cc] *= rq;
      sK[r * KP + cc] *= rk;
    }
    if (lane == 0) {
      sRq[r] = rq;
      sRk[r] = rk;
    }
  }
  if (tid < K) {
    float acc = 0.f;
    for (int r = 0; r < BT; ++r) {
      acc += sG[r * KP + tid];
      sG[r * KP + tid] = acc;
    }
  }
  __syncthreads();

  // 3. A = (I + L)^-1 into sA: from the forward's intra-chunk stage when it
  //    kept it, else L (strictly lower, beta-weighted) into sP and forward
  //    substitution
  if (a_in) {
    const float *src = a_in + (c * H + h) * (BT * BT);
    for (int i = tid; i < BT * BT; i += 256) sA[(i >> 6) * 65 + (i & 63)] = src[i];
  } else {
  for (int p = tid; p < BT * BT; p += 256) {
    const int r = p / BT, j = p % BT;
    float acc = 0.f;
    if (j < r && r < len) {
      for (int cc = 0; cc < K; ++cc)
        acc = fmaf(sK[r * KP + cc], sK[j * KP + cc] * expf(sG[r * KP + cc] - sG[j * KP + cc]), acc);
      acc *= sB[r];
    }
    sP[r * 65 + j] = acc;
  }
  __syncthreads();
  {
    const int col = tid >> 2, part = tid & 3;
    for (int i = 0; i < BT; ++i) {
      float acc = 0.f;
      for (int m = col + part; m < i; m += 4) acc = fmaf(sP[i * 65 + m], sA[m * 65 + col], acc);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (part == 0) sA[i * 65 + col] = (i == col) ? 1.f : (i > col ? -acc : 0.f);
      __syncwarp();
    }
  }
  }
  __syncthreads();

  // channel-mapped accumulators: rows part + NP m of channel cc
  const int cc = tid % K, part = tid / K;
  float aq[NR], ak[NR], ag[NR], ab[NR];
#pragma unroll
  for (int m = 0; m < NR; ++m) aq[m] = ak[m] = ag[m] = ab[m] = 0.f;

  // 4a. X = dv_new, Y = v:  dA_ij = beta_j sum_v X_iv Y_jv (j < i) into sM;
  //     dvb = A^T dv_new, dv = beta dvb, dbeta += sum_v dvb v
  for (int i = tid; i < BT * V; i += 256) {
    const int r = i / V, cv = i % V;
    const bool in = r < len;
    X[r * XP + cv] = in ? (LIST ? -img_at(img.dvn_neg, item, r, cv) : dvn[row_off(r, H, h, V) + cv]) : 0.f;
    Y[r * XP + cv] = in ? to_f32(v[row_off(r, H, h, V) + cv]) : 0.f;
  }
  __syncthreads();
  {
    const int i = tid >> 2;
    for (int m = 0; m < 16; ++m) {
      const int j = (tid & 3) + 4 * m;
      float acc = 0.f;
      if (j < i)
        for (int cv = 0; cv < V; ++cv) acc = fmaf(X[i * XP + cv], Y[j * XP + cv], acc);
      sM[i * 65 + j] = acc * sB[j];
    }
  }
  {
    const int cv = tid % V, pv = tid / V;
    for (int j = pv; j < BT; j += NPV) {
      float acc = 0.f;
      for (int i = j; i < len; ++i) acc = fmaf(sA[i * 65 + j], X[i * XP + cv], acc);
      if (j < len) dv_out[row_off(j, H, h, V) + cv] = from_f32<Tin>(acc * sB[j]);
      float pb = acc * Y[j * XP + cv];
      for (int o = 16; o; o >>= 1) pb += __shfl_xor_sync(0xffffffffu, pb, o);
      if (lane == 0) sRedV[j * 4 + (cv >> 5)] = pb;
    }
  }
  __syncthreads();

  // 4b. X = dw, Y = k^ beta e^G:  dA_ij += sum_c X_ic Y_jc (j < i);
  //     dkb = A^T dw -> dk^, dbeta, dG
  for (int i = tid; i < BT * K; i += 256) {
    const int r = i / K, c2 = i % K;
    X[r * XP + c2] = r < len ? (LIST ? img_at(img.dw, item, r, c2) : dw[row_off(r, H, h, K) + c2]) : 0.f;
    Y[r * XP + c2] = sK[r * KP + c2] * sB[r] * expf(sG[r * KP + c2]);
  }
  __syncthreads();
  {
    const int i = tid >> 2;
    for (int m = 0; m < 16; ++m) {
      const int j = (tid & 3) + 4 * m;
      if (j < i) {
        float acc = 0.f;
        for (int c2 = 0; c2 < K; ++c2) acc = fmaf(X[i * XP + c2], Y[j * XP + c2], acc);
        sM[i * 65 + j] += acc;
      }
    }
  }
#pragma unroll
  for (int m = 0; m < NR; ++m) {
    const int j = part + NP * m;
    if (j < len) {
      float acc = 0.f;
      for (int i = j; i < len; ++i) acc = fmaf(sA[i * 65 + j], X[i * XP + cc], acc);
      const float e = expf(sG[j * KP + cc]);
      ak[m] = fmaf(acc, sB[j] * e, ak[m]);
      ab[m] = fmaf(acc, sK[j * KP + cc] * e, ab[m]);
      ag[m] = fmaf(acc, Y[j * XP + cc], ag[m]);
    }
  }
  __syncthreads();

  // 5. dL = -A^T dA A^T (strictly lower): sP = A^T dA, then sM = dL
  {
    const int p = tid >> 2;
    for (int m = 0; m < 16; ++m) {
      const int qq = (tid & 3) + 4 * m;
      float acc = 0.f;
      for (int i = (p > qq + 1 ? p : qq + 1); i < BT; ++i) acc = fmaf(sA[i * 65 + p], sM[i * 65 + qq], acc);
      sP[p * 65 + qq] = acc;
    }
  }
  __syncthreads();
  {
    const int i = tid >> 2;
    for (int m = 0; m < 16; ++m) {
      const int j = (tid & 3) + 4 * m;
      float acc = 0.f;
      if (j < i)
        for (int qq = 0; qq <= j; ++qq) acc = fmaf(sP[i * 65 + qq], sA[j * 65 + qq], acc);
      sM[i * 65 + j] = -acc;
    }
  }
  __syncthreads();

  // 6. X = dO, Y = v_new:  sP = scale dAqk (j <= i)
  for (int i = tid; i < BT * V; i += 256) {
    const int r = i / V, cv = i % V;
    const bool in = r < len;
    X[r * XP + cv] = (in && d_out) ? to_f32(d_out[row_off(r, H, h, V) + cv]) : 0.f;
    Y[r * XP + cv] = in ? (LIST ? img_at(img.vn, item, r, cv) : vn[row_off(r, H, h, V) + cv]) : 0.f;
  }
  __syncthreads();
  {
    const int i = tid >> 2;
    for (int m = 0; m < 16; ++m) {
      const int j = (tid & 3) + 4 * m;
      float acc = 0.f;
      if (j <= i)
        for (int cv = 0; cv < V; ++cv) acc = fmaf(X[i * XP + cv], Y[j * XP + cv], acc);
      sP[i * 65 + j] = scale * acc;
    }
  }
  __syncthreads();

  // 7. pairwise terms of L (D = dL) and Aqk (Q = scale dAqk) over channel cc:
  //    row side (row i over j <= i), then column side (row j over i >= j)
#pragma unroll
  for (int m = 0; m < NR; ++m) {
    const int i = part + NP * m;
    if (i < len) {
      const float qi = sQ[i * KP + cc], ki = sK[i * KP + cc], Gi = sG[i * KP + cc], bi = sB[i];
      float a_q = 0.f, a_k = 0.f, a_b = 0.f, a_g = 0.f;
      for (int j = 0; j <= i; ++j) {
        const float e = expf(Gi - sG[j * KP + cc]);
        const float t = sK[j * KP + cc] * e;
        const float Q = sP[i * 65 + j], D = (j < i) ? sM[i * 65 + j] : 0.f;
        a_q = fmaf(Q, t, a_q);
        a_k = fmaf(D, t, a_k);
        a_g = fmaf(bi * D * ki + Q * qi, t, a_g);
      }
      a_b = a_k * ki;
      aq[m] += a_q;
      ak[m] = fmaf(bi, a_k, ak[m]);
      ab[m] += a_b;
      ag[m] += a_g;
    }
  }
#pragma unroll
  for (int m = 0; m < NR; ++m) {
    const int j = part + NP * m;
    if (j < len) {
      const float kj = sK[j * KP + cc], Gj = sG[j * KP + cc];
      float a_k = 0.f;
      for (int i = j; i < len; ++i) {
        const float e = expf(sG[i * KP + cc] - Gj);
        const float D = (i > j) ? sM[i * 65 + j] : 0.f;
        const float x = sB[i] * D * sK[i * KP + cc] + sP[i * 65 + j] * sQ[i * KP + cc];
        a_k = fmaf(x, e, a_k);
      }
      ak[m] += a_k;
      ag[m] = fmaf(-a_k, kj, ag[m]);
    }
  }

  // 8. elementwise terms of qg = scale q^ e^G and kg = k^ e^{G_C - G}
  const float GC = sG[(len - 1) * KP + cc];
  float agc = 0.f;
#pragma unroll
  for (int m = 0; m < NR; ++m) {
    const int r = part + NP * m;
    if (r < len) {
      const int64_t off = row_off(r, H, h, K) + cc;
      const float G = sG[r * KP + cc], eg = expf(G), ekg = expf(GC - G);
      const float a = dqg[off] * scale * eg;
      aq[m] = fmaf(a, 1.f, aq[m]);
      ag[m] = fmaf(a, sQ[r * KP + cc], ag[m]);
      const float b = dkg[off] * ekg;
      ak[m] += b;
      ag[m] = fmaf(-b, sK[r * KP + cc], ag[m]);
      agc = fmaf(b, sK[r * KP + cc], agc);
    }
  }
  __syncthreads();  // everyone is done with X, Y, sP, sM

  // 9. dG into X, dG_C onto the last row, reverse cumsum -> gradient of g
  sRedC[part * K + cc] = agc;
#pragma unroll
  for (int m = 0; m < NR; ++m) {
    const int r = part + NP * m;
    X[r * XP + cc] = ag[m];
    Y[r * XP + cc] = aq[m];
    sA[r * KP + cc] = ak[m];  // dk^ (the sA, sP, sM block is free)
  }
  // dbeta parts over channels (rows of this warp's part)
#pragma unroll
  for (int m = 0; m < NR; ++m) {
    float pb = ab[m];
    for (int o = 16; o; o >>= 1) pb += __shfl_xor_sync(0xffffffffu, pb, o);
    if (lane == 0) sRedK[(part + NP * m) * 4 + (cc >> 5)] = pb;
  }
  __syncthreads();
  if (tid < K) {
    float dgcC = 0.f;
    for (int p = 0; p < NP; ++p) dgcC += sRedC[p * K + tid];
    dgcC = fmaf(dgc[(c * H + h) * K + tid], expf(sG[(len - 1) * KP + tid]), dgcC);
    float run = dgcC;
    for (int r = len - 1; r >= 0; --r) {
      run += X[r * XP + tid];
      X[r * XP + tid] = run;
    }
  }
  __syncthreads();

  // 10. L2-norm backward: dx = r (dx^ - x^ (x^ . dx^)), one warp per row
  float *sDk = sA;
  for (int r = warp; r < len; r += 8) {
    float pq = 0.f, pk = 0.f;
    for (int c2 = lane; c2 < K; c2 += 32) {
      pq = fmaf(sQ[r * KP + c2], Y[r * XP + c2], pq);
      pk = fmaf(sK[r * KP + c2], sDk[r * KP + c2], pk);
    }
    for (int o = 16; o; o >>= 1) {
      pq += __shfl_xor_sync(0xffffffffu, pq, o);
      pk += __shfl_xor_sync(0xffffffffu, pk, o);
    }
    if (!(gp.flags & KDA_L2NORM_QK)) pq = pk = 0.f;
    const float rq = sRq[r], rk = sRk[r];
    for (int c2 = lane; c2 < K; c2 += 32) {
      const int64_t off = row_off(r, H, h, K) + c2;
      dq_out[off] = from_f32<Tdq>(rq * (Y[r * XP + c2] - sQ[r * KP + c2] * pq));
      dk_out[off] = from_f32<Tdq>(rk * (sDk[r * KP + c2] - sK[r * KP + c2] * pk));
    }
  }

  // 11. gate backward: dz = -exp(a_log) sigmoid(z) dg, z = x + dt_bias
  float dtb = 0.f, alog = 0.f;
  for (int r = part; r < len; r += NP) {
    const int64_t off = row_off(r, H, h, K) + cc;
    const float dgn = X[r * XP + cc];
    if (gate) {
      const float z = g[off] + (gp.dt_bias ? gp.dt_bias[h * K + cc] : 0.f);
      const float sgm = 1.f / (1.f + expf(-z));
      const float dz = -A_h * sgm * dgn;
      dg_out[off] = dz;
      dtb += dz;
      alog = fmaf(-A_h * softplus_f(z), dgn, alog);
    } else {
      dg_out[off] = dgn;
    }
  }
  if (gate) {
    sRedC[part * K + cc] = dtb;
    for (int o = 16; o; o >>= 1) alog += __shfl_xor_sync(0xffffffffu, alog, o);
    if (lane == 0) sRedS[warp] = alog;
  }
  __syncthreads();
  if (gate && tid < K) {
    float d = 0.f;
    for (int p = 0; p < NP; ++p) d += sRedC[p * K + tid];
    part_dtb[(c * H + h) * K + tid] = d;
  }
  if (gate && tid == 0) {
    float a = 0.f;
    for (int w2 = 0; w2 < 8; ++w2) a += sRedS[w2];
    part_alog[c * H + h] = a;
  }

  // 12. beta: d(beta) from v.beta, k^.beta.e^G and L; sigmoid backward
  if (tid < len) {
    float d = 0.f;
    for (int x = 0; x < V / 32; ++x) d += sRedV[tid * 4 + x];
    for (int x = 0; x < K / 32; ++x) d += sRedK[tid * 4 + x];
    const float b = sB[tid];
    dbeta_out[(t0 + tid) * H + h] = sig ? d * b * (1.f - b) : d;
  }
  }  // items
}

// ---------------------------------------------------------------------------
// Reductions.
// ---------------------------------------------------------------------------
__global__ void bwd_param_reduce_kernel(int64_t nchunks, int H, int K, const float *__restrict__ part_alog,
                                        const float *__restrict__ part_dtb, float *__restrict__ da_log,
                                        float *__restrict__ ddt_bias) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // (h, channel)
  if (i >= H * K) return;
  const int h = i / K, cc = i % K;
  float d = 0.f, a = 0.f;
  for (int64_t c = 0; c < nchunks; ++c) {
    d += part_dtb[(c * H + h) * K + cc];
    if (cc == 0) a += part_alog[c * H + h];
  }
  if (ddt_bias) ddt_bias[i] = d;
  if (da_log && cc == 0) da_log[h] = a;
}

template <typename Tin>
__global__ void bwd_group_sum_kernel(int64_t rows, int H, int Hk, int K, const float *__restrict__ dqv,
                                     const float *__restrict__ dkv, Tin *__restrict__ dq,
                                     Tin *__restrict__ dk) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (token, key head, channel)
  if (i >= rows * Hk * K) return;
  const int cc = (int)(i % K);
  const int64_t th = i / K;
  const int hk = (int)(th % Hk);
  const int64_t t = th / Hk;
  const int grp = H / Hk;
  float a = 0.f, b = 0.f;
  for (int x = 0; x < grp; ++x) {
    const int64_t off = (t * H + hk * grp + x) * (int64_t)K + cc;
    a += dqv[off];
    b += dkv[off];
  }
  dq[i] = from_f32<Tin>(a);
  dk[i] = from_f32<Tin>(b);
}

template <typename Tin, int K>
cudaError_t dh_dispatch(const BwdLaunch &b, int V, cudaStream_t st) {
  const size_t smem = sizeof(float) * (K * VT + 3 * BT * K + 2 * BT * VT + BT * BT + K);
  auto kern = bwd_dh_kernel<Tin, K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((int64_t)b.s.N * b.H), V / VT);
  if (grid.x == 0) return cudaSuccess;
  kern<<<grid, 256, smem, st>>>(b.s, b.H, V, b.w, b.qg, b.kg, b.aqk, b.gc,
                                static_cast<const Tin *>(b.d_out), b.d_final, b.dhn, b.dvn,
                                b.d_initial);
  return cudaGetLastError();
}

template <typename Tin, int K, int V>
cudaError_t bwd_dispatch(const BwdLaunch &b, bool with_dh, bool with_state, cudaStream_t st) {
  const SeqInfo &s = b.s;
  const int H = b.H, Hk = b.Hk;
  const Tin *dO = static_cast<const Tin *>(b.d_out);
  // B1: reverse chain of the state gradient (unless the caller ran it)
  if (with_dh) {
    cudaError_t e0 = dh_dispatch<Tin, K>(b, V, st);
    if (e0 != cudaSuccess) return e0;
  }
  if (b.nchunks == 0) return cudaSuccess;
  // B2: state-contraction terms (unless the caller ran them)
  if (with_state) {
    const size_t smem = sizeof(float) * (2 * VT * (K + 1) + 3 * BT * VT);
    auto kern = bwd_state_kernel<Tin, K>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)b.nchunks, H);
    kern<<<grid, 256, smem, st>>>(s, H, V, b.h, b.dhn, dO, b.dvn, b.vn, b.dqg, b.dw, b.dkg, b.dgc);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // B3: intra-chunk backward
  {
    const size_t smem = sizeof(float) * IntraSmem<K, V>::total;
    const bool grouped = Hk != H;
    dim3 grid((unsigned)b.nchunks, H);
    cudaError_t e;
    if (grouped) {
      auto kern = bwd_intra_kernel<Tin, float, K, V>;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      kern<<<grid, 256, smem, st>>>(
          static_cast<const Tin *>(b.q), static_cast<const Tin *>(b.k), static_cast<const Tin *>(b.v),
          b.g, b.beta, b.gp, s, H, Hk, dO, b.dvn, b.vn, b.dqg, b.dw, b.dkg, b.dgc, b.dqv, b.dkv,
          static_cast<Tin *>(b.dv), b.dg, b.dbeta, b.part_alog, b.part_dtb, b.a_in, ImgSrc{});
    } else {
      auto kern = bwd_intra_kernel<Tin, Tin, K, V>;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      kern<<<grid, 256, smem, st>>>(
          static_cast<const Tin *>(b.q), static_cast<const Tin *>(b.k), static_cast<const Tin *>(b.v),
          b.g, b.beta, b.gp, s, H, Hk, dO, b.dvn, b.vn, b.dqg, b.dw, b.dkg, b.dgc,
          static_cast<Tin *>(b.dq), static_cast<Tin *>(b.dk), static_cast<Tin *>(b.dv), b.dg, b.dbeta,
          b.part_alog, b.part_dtb, b.a_in, ImgSrc{});
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (grouped) {
      const int64_t n = s.T_tot * Hk * K;
      bwd_group_sum_kernel<Tin><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
          s.T_tot, H, Hk, K, b.dqv, b.dkv, static_cast<Tin *>(b.dq), static_cast<Tin *>(b.dk));
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_generic_bwd(kda_dtype dt, int K, int V, const BwdLaunch &b, cudaStream_t st,
                               bool with_dh, bool with_state) {
#define KDA_BWD(T_, K_, V_) \
  if (K == K_ && V == V_) return bwd_dispatch<T_, K_, V_>(b, with_dh, with_state, st);
  if (dt == KDA_F32) {
    KDA_BWD(float, 64, 64) KDA_BWD(float, 64, 128) KDA_BWD(float, 128, 64) KDA_BWD(float, 128, 128)
  } else {
    KDA_BWD(__nv_bfloat16, 64, 64) KDA_BWD(__nv_bfloat16, 64, 128)
    KDA_BWD(__nv_bfloat16, 128, 64) KDA_BWD(__nv_bfloat16, 128, 128)
  }
#undef KDA_BWD
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_intra_list(const BwdLaunch &b, const uint8_t *dvn_neg_img, const uint8_t *vn_img,
                                  const uint8_t *dw_img, const uint32_t *count, const uint32_t *list,
                                  cudaStream_t st) {
  constexpr int K = 128, V = 128;
  using Tin = __nv_bfloat16;
  const int64_t nitems = b.nchunks * b.H;
  if (nitems == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 148;
  const size_t smem = sizeof(float) * IntraSmem<K, V>::total;
  const ImgSrc img{dvn_neg_img, vn_img, dw_img, count, list};
  const int grid = (int)(nitems < sms ? nitems : sms);
  const Tin *dO = static_cast<const Tin *>(b.d_out);
  cudaError_t e;
  if (b.Hk != b.H) {
    auto kern = bwd_intra_kernel<Tin, float, K, V, true>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 256, smem, st>>>(
        static_cast<const Tin *>(b.q), static_cast<const Tin *>(b.k), static_cast<const Tin *>(b.v), b.g,
        b.beta, b.gp, b.s, b.H, b.Hk, dO, nullptr, nullptr, b.dqg, nullptr, b.dkg, b.dgc, b.dqv, b.dkv,
        static_cast<Tin *>(b.dv), b.dg, b.dbeta, b.part_alog, b.part_dtb, b.a_in, img);
  } else {
    auto kern = bwd_intra_kernel<Tin, Tin, K, V, true>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 256, smem, st>>>(
        static_cast<const Tin *>(b.q), static_cast<const Tin *>(b.k), static_cast<const Tin *>(b.v), b.g,
        b.beta, b.gp, b.s, b.H, b.Hk, dO, nullptr, nullptr, b.dqg, nullptr, b.dkg, b.dgc,
        static_cast<Tin *>(b.dq), static_cast<Tin *>(b.dk), static_cast<Tin *>(b.dv), b.dg, b.dbeta,
        b.part_alog, b.part_dtb, b.a_in, img);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_dh(kda_dtype dt, int K, int V, const BwdLaunch &b, cudaStream_t st) {
  if (dt == KDA_F32) {
    if (K == 64) return dh_dispatch<float, 64>(b, V, st);
    if (K == 128) return dh_dispatch<float, 128>(b, V, st);
  } else {
    if (K == 64) return dh_dispatch<__nv_bfloat16, 64>(b, V, st);
    if (K == 128) return dh_dispatch<__nv_bfloat16, 128>(b, V, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_group_sum(kda_dtype dt, int64_t rows, int H, int Hk, int K, const float *dqv,
                                 const float *dkv, void *dq, void *dk, cudaStream_t st) {
  const int64_t n = rows * Hk * K;
  if (n == 0) return cudaSuccess;
  if (dt == KDA_F32)
    bwd_group_sum_kernel<float><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
        rows, H, Hk, K, dqv, dkv, static_cast<float *>(dq), static_cast<float *>(dk));
  else
    bwd_group_sum_kernel<__nv_bfloat16><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
        rows, H, Hk, K, dqv, dkv, static_cast<__nv_bfloat16 *>(dq), static_cast<__nv_bfloat16 *>(dk));
  return cudaGetLastError();
}

cudaError_t launch_bwd_param_reduce(int64_t nchunks, int H, int K, const float *part_alog,
                                    const float *part_dtb, float *da_log, float *ddt_bias,
                                    cudaStream_t st) {
  if (!da_log && !ddt_bias) return cudaSuccess;
  const int n = H * K;
  bwd_param_reduce_kernel<<<(n + 255) / 256, 256, 0, st>>>(nchunks, H, K, part_alog, part_dtb, da_log,
                                                           ddt_bias);
  return cudaGetLastError();
}

}  // namespace kda
