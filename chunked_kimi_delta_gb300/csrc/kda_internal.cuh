// kda_internal.cuh - definitions shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int BT = 64;  // chunk length

// ---------------------------------------------------------------------------
// Sequences and chunks.  A problem is a set of N token ranges ("sequences":
// the batch rows, the packed sequences of cu_seqlens, or the segments of a
// summary) over a token axis of T_tot tokens.  Chunks restart at every range
// start; chunk ids are numbered range by range.
// ---------------------------------------------------------------------------
struct SeqInfo {
  const int32_t *bounds;     // device [N+1] range offsets, or null: range n = [n*T, (n+1)*T)
  const int32_t *chunk_off;  // device [N+1] first chunk id of each range (when bounds)
  int64_t T_tot;             // tokens on the token axis
  int32_t T;                 // fixed range length (bounds == null)
  int32_t N;                 // number of ranges
};

// Range n, clamped into the token axis (defends the kernels against a bad
// cu_seqlens: out-of-range or decreasing offsets become empty ranges).
__device__ __forceinline__ void seq_range(const SeqInfo &s, int n, int64_t &t0, int64_t &t1) {
  if (s.bounds) {
    int64_t a = s.bounds[n], b = s.bounds[n + 1];
    a = a < 0 ? 0 : (a > s.T_tot ? s.T_tot : a);
    b = b < a ? a : (b > s.T_tot ? s.T_tot : b);
    t0 = a;
    t1 = b;
  } else {
    t0 = (int64_t)n * s.T;
    t1 = t0 + s.T;
  }
}

__device__ __forceinline__ int64_t seq_first_chunk(const SeqInfo &s, int n) {
  if (s.bounds) return s.chunk_off[n];
  return (int64_t)n * ((s.T + BT - 1) / BT);
}

// Global chunk id -> (range n, first token, length).  False when c is past
// the last chunk (grids are sized by an upper bound).
__device__ __forceinline__ bool chunk_lookup(const SeqInfo &s, int64_t c, int &n, int64_t &t0,
                                             int &len) {
  if (s.bounds) {
    if (c >= s.chunk_off[s.N]) return false;
    int lo = 0, hi = s.N - 1;  // largest n with chunk_off[n] <= c
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (s.chunk_off[mid] <= c) lo = mid; else hi = mid - 1;
    }
    n = lo;
  } else {
    const int64_t per = (s.T + BT - 1) / BT;
    if (per == 0 || c >= per * s.N) return false;
    n = (int)(c / per);
  }
  int64_t a, b;
  seq_range(s, n, a, b);
  const int64_t local = c - seq_first_chunk(s, n);
  t0 = a + local * BT;
  const int64_t rem = b - t0;
  len = (int)(rem < BT ? rem : BT);
  return len > 0;
}

// Upper bound on the number of chunks.
inline int64_t chunks_upper_bound(int64_t T_tot, int32_t N, bool ragged, int32_t T) {
  if (!ragged) return (int64_t)N * ((T + BT - 1) / BT);
  return (T_tot + BT - 1) / BT + N;
}

// ---------------------------------------------------------------------------
// Workspace of the forward / summary (generic path).  Byte offsets from the
// workspace base; every block is 256-byte aligned.
// ---------------------------------------------------------------------------
struct FwdPlan {
  int64_t T_tot, nchunks;
  int32_t N, H, K, V;
  int32_t Hk;  // heads of q and k; value head h reads key head h / (H / Hk)
  size_t off_chunk_off, off_w, off_u, off_qg, off_kg, off_aqk, off_gc, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

inline FwdPlan make_plan(int64_t T_tot, int32_t N, bool ragged, int32_t T, int H, int K, int V) {
  FwdPlan p{};
  p.T_tot = T_tot;
  p.N = N;
  p.H = H;
  p.Hk = H;
  p.K = K;
  p.V = V;
  p.nchunks = chunks_upper_bound(T_tot, N, ragged, T);
  size_t o = 256;  // [0,256): device status word
  p.off_chunk_off = o; o = align256(o + sizeof(int32_t) * (size_t)(N + 1));
  const size_t th = (size_t)T_tot * H;
  p.off_w = o;   o = align256(o + 4 * th * K);
  p.off_u = o;   o = align256(o + 4 * th * V);
  p.off_qg = o;  o = align256(o + 4 * th * K);
  p.off_kg = o;  o = align256(o + 4 * th * K);
  p.off_aqk = o; o = align256(o + 4 * th * BT);
  p.off_gc = o;  o = align256(o + 4 * (size_t)p.nchunks * H * K);
  p.total = o;
  return p;
}

// Device error word (first 4 bytes of a workspace).
constexpr uint32_t DEV_ERR_TIMEOUT = 1u;

// ---------------------------------------------------------------------------
// Element conversions.
// ---------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ---------------------------------------------------------------------------
// Launchers (host side), implemented in the .cu files.
// ---------------------------------------------------------------------------
struct GateParams {
  const float *a_log, *dt_bias;
  float scale, eps;
  uint32_t flags;
  // head widths of the call (the tensor-core kernels work 128 wide: narrower
  // heads are read with the extra channels held at zero)
  int32_t dk = 128, dv = 128;
};

cudaError_t launch_chunk_map(const SeqInfo &s, int32_t *chunk_off, cudaStream_t st);

// n fp32 matrices R x C -> C x R (kda_layout.cu); with count_ptr only the
// first (*count_ptr) * per_count matrices.
// dst[m] = the rows_dst x row_bytes_dst window of src[m] (rows_src x
// row_bytes_src), `fill` (a 32-bit pattern) outside src; n matrices, row
// bytes multiples of 16.  With count_ptr only matrices below
// (*count_ptr) * per_count are written.
cudaError_t launch_window_copy(const void *src, void *dst, int64_t n, int rows_src, int row_bytes_src,
                               int rows_dst, int row_bytes_dst, uint32_t fill, const int32_t *count_ptr,
                               int per_count, cudaStream_t st);
cudaError_t launch_transpose_states(const float *src, float *dst, int64_t n, int R, int C,
                                    const int32_t *count_ptr, int per_count, cudaStream_t st);
// [B, H, T, row] <-> [B, T, H, row] (row_bytes a multiple of 4).
cudaError_t launch_swap_token_head(const void *src, void *dst, int64_t B, int H, int64_t T,
                                   int row_bytes, bool to_token_major, cudaStream_t st);

// Recurrent decode step on pool rows (kda_decode.cu).
cudaError_t launch_decode(kda_dtype qkv_dtype, kda_dtype cache_dtype, kda_index_dtype idx_dtype,
                          int dk, int dv, int N, int T, int H, int Hk, const void *q, const void *k,
                          const void *v, const float *g, const float *beta, const GateParams &gp,
                          void *out, void *cache, int64_t num_rows, int64_t row_stride,
                          const void *idx, const bool *init_flags, bool vfirst, cudaStream_t st);

// Generic (CUDA-core, fp32 arithmetic) intra-chunk stage: writes w, u, qg, kg,
// Aqk, gC of the plan.
cudaError_t launch_generic_intra(kda_dtype dt, const void *q, const void *k, const void *v,
                                 const float *g, const float *beta, const GateParams &gp,
                                 const SeqInfo &s, const FwdPlan &p, char *ws, cudaStream_t st);

// Generic inter-chunk chain.  summary = false: forward (o, final, h_out,
// v_new_out); summary = true: augmented [S~ | M] chain written to S_tilde / M.
struct InterOut {
  void *out;
  float *final_state, *h_out, *v_new_out;
  const float *initial_state;
  float *S_tilde, *M;
};
cudaError_t launch_generic_inter(kda_dtype dt, bool summary, const InterOut &io, const SeqInfo &s,
                                 const FwdPlan &p, const char *ws, cudaStream_t st);

// Backward on CUDA cores (kda_bwd.cu): pointers of one call.  w, qg, kg, aqk,
// gc, h and vn are the forward's recomputed intermediates; dhn, dvn, dqg,
// dw, dkg, dgc, part_* and (grouped key heads) dqv, dkv are scratch.
struct BwdLaunch {
  SeqInfo s;
  int H, Hk;
  int64_t nchunks;
  const void *q, *k, *v;
  const float *g, *beta;
  GateParams gp;
  const void *d_out;
  const float *d_final;
  const float *w, *qg, *kg, *aqk, *gc, *h, *vn;
  float *dhn, *dvn, *dqg, *dw, *dkg, *dgc, *part_alog, *part_dtb, *dqv, *dkv;
  void *dq, *dk, *dv;
  float *dg, *dbeta, *d_initial;
  const float *a_in;  // [nchunks, H, 64, 64] A = (I + L)^-1 from the forward, or null (recomputed)
};
// with_dh = false: dvn and d_initial come from the tensor-core reverse chain;
// with_state = false: dqg, dw, dkg, dgc from the tensor-core state kernel.
cudaError_t launch_generic_bwd(kda_dtype dt, int K, int V, const BwdLaunch &b, cudaStream_t st,
                               bool with_dh = true, bool with_state = true);
// The intra-chunk backward of the (chunk, head) items in list (count on the
// device) on the CUDA cores, bf16 d_k = d_v = 128, from the tensor-core
// path's tile images of -dv_new, v_new and dw (b.dvn, b.vn, b.dw unused):
// the exact pass for the chunks under strong decay, written over what the
// tensor-core kernel left for them.
cudaError_t launch_bwd_intra_list(const BwdLaunch &b, const uint8_t *dvn_neg_img, const uint8_t *vn_img,
                                  const uint8_t *dw_img, const uint32_t *count, const uint32_t *list,
                                  cudaStream_t st);
// The reverse state-gradient chain alone (dhn / dvn may be null: not written).
cudaError_t launch_bwd_dh(kda_dtype dt, int K, int V, const BwdLaunch &b, cudaStream_t st);
// dq, dk of each key head = the sum over the value heads of its group.
cudaError_t launch_bwd_group_sum(kda_dtype dt, int64_t rows, int H, int Hk, int K, const float *dqv,
                                 const float *dkv, void *dq, void *dk, cudaStream_t st);
cudaError_t launch_bwd_param_reduce(int64_t nchunks, int H, int K, const float *part_alog,
                                    const float *part_dtb, float *da_log, float *ddt_bias,
                                    cudaStream_t st);

// reverse = false: S_in[j] = S; S = M_j S + S~_j over j = 0 .. S-1.
// reverse = true:  S_in[j] = S; S = M_j^T S + S~_j over j = S-1 .. 0.
cudaError_t launch_prefix_scan(const float *M, const float *S_tilde, const float *S0, int C,
                               int S, int H, int K, int V, float *S_in, float *S_final,
                               cudaStream_t st, bool reverse = false);

cudaError_t launch_state_gather(const void *cache, kda_dtype dt, int64_t num_rows,
                                int64_t row_stride, int64_t payload, const void *idx,
                                kda_index_dtype it, const bool *flags, int64_t n_sel,
                                void *packed, cudaStream_t st);
cudaError_t launch_state_scatter(void *cache, kda_dtype dt, int64_t num_rows, int64_t row_stride,
                                 int64_t payload, const void *idx, kda_index_dtype it,
                                 const void *packed, kda_dtype pdt, int64_t n_sel,
                                 cudaStream_t st);

}  // namespace kda
