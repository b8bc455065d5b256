// kda_tc.cuh - shared definitions of the tensor-core (tcgen05) forward path
// for bf16 inputs with d_k = d_v = 128.
//
// The path has three kernels:
//   prep    (kda_tc_prep.cu): per (chunk, head) - gate, cumulative decay, L2
//           norms, the decay-weighted A_kk / A_qk products, the triangular
//           inverse and the WY products w = A (k.beta.e^G), u = A (v.beta);
//   chain   (kda_tc_chain.cu): per (sequence, head) - the sequential state
//           recurrence v_new = u - w h, o = qg h + Aqk v_new,
//           h' = e^{G_C} h + kg^T v_new;
//   summary (kda_tc_summary.cu): per (segment, head) - the same recurrence
//           on the augmented state [S~ | M] for the segment summary.
// prep hands each chunk to the others as a "package": a byte image of the
// shared memory tiles they feed to the tensor cores, so it moves with bulk
// copies and no re-layout.
#pragma once

#include <cuda.h>

#include "kda_internal.cuh"
#include "tc_primitives.cuh"

namespace kda {
namespace tcp {

constexpr int K = 128, V = 128;

// Package of one (chunk, head), byte offsets.  All tiles are bf16 SW128 except
// U (bf16 rows of 256 bytes, 16-byte chunks of row r permuted by XOR with
// r % 16) and GC (fp32).
//   WQ : [qg (rows 0-63); w (rows 64-127)] x 128 channels, K-major, two
//        64-channel panels of 128 rows           -> A operand of [qg; w] h
//   U  : u [64 tokens][128] bf16 (the precision of the other WY tiles)
//   KG : kg = k^ e^{G_C - G} as [token][channel], MN-major, two 64-channel
//        panels of 64 token rows                  -> A operand of kg^T v_new
//   AQK: Aqk [64 rows][64 tokens], K-major        -> A operand of Aqk v_new
//   GC : e^{G_C} [128] fp32 (decay of the whole chunk per key channel)
// WQ and U (read first) and KG, AQK, GC (read last) are contiguous, so that
// the two halves can be moved separately.
constexpr uint32_t PK_WQ = 0;
constexpr uint32_t PK_U = 32768;
constexpr uint32_t PK_KG = 49152;
constexpr uint32_t PK_AQK = 65536;
constexpr uint32_t PK_GC = 73728;
constexpr uint32_t PK_BYTES = 74240;
constexpr uint32_t PK_FIRST = PK_KG;  // bytes of the first half (WQ, U)

__host__ __device__ __forceinline__ uint32_t u_offset(uint32_t row, uint32_t col) {
  // bf16 element (row, col) of the U tile
  const uint32_t chunk = (col >> 3) ^ (row & 15u);
  return row * 256u + chunk * 16u + (col & 7u) * 2u;
}

// K-major SW128 tile with `rows` rows per 64-element K panel: byte offset of
// bf16 element (row, k).
__host__ __device__ __forceinline__ uint32_t kmaj_off(uint32_t rows, uint32_t row, uint32_t k) {
  return (k >> 6) * rows * 128u + tc::sw128_offset(row, (k & 63u) * 2u);
}
// MN-major SW128 tile with `krows` K rows per 64-element MN panel: byte offset
// of bf16 element (k, mn).
__host__ __device__ __forceinline__ uint32_t mnmaj_off(uint32_t krows, uint32_t k, uint32_t mn) {
  return (mn >> 6) * krows * 128u + tc::sw128_offset(k, (mn & 63u) * 2u);
}

// Bounded waits: give up after this many nanoseconds.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for an mbarrier phase; on timeout (limit_ns) record the device error
// word and return false.
__device__ __forceinline__ bool wait_or_flag(uint64_t *bar, uint32_t parity, uint32_t *err,
                                             unsigned long long limit_ns = WAIT_LIMIT_NS) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 256; ++i)
      if (tc::mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) {
      atomicOr(err, DEV_ERR_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait used when a CTA winds down after a timeout: lets copies or
// MMAs it started finish before it releases its memory; ignores the result.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!tc::mbar_try_wait(bar, parity) && globaltimer() - t0 < WAIT_LIMIT_NS) {
  }
}

// 3-D TMA load (coordinates: channel, head, token).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(tc::smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
         "r"(tc::smem_u32(bar))
      : "memory");
}

// Prefetch a 3-D TMA box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int32_t x, int32_t y,
                                                   int32_t z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
               :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z) : "memory");
}

// Bulk copy shared -> global (16-byte aligned, size multiple of 16), tracked
// by the issuing thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               :: "l"(reinterpret_cast<uint64_t>(dst)), "r"(tc::smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the shared-memory sources of all committed bulk stores have
// been read (the smem may then be rewritten).
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until all committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Plain bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(tc::smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
         "r"(tc::smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Paired fp32 arithmetic: one packed instruction for two values, each
// rounded to nearest exactly as the scalar operation would be.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
// a - b (the product b * -1 is exact, so this rounds as the subtraction does)
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.f, -1.f), a); }
__device__ __forceinline__ float2 splat2(float a) { return make_float2(a, a); }

// Host side --------------------------------------------------------------------
struct TcMaps {
  CUtensorMap q, k, v, x;
};

// Encodes the four input tensor maps (q, k, gate input with dk channels, v
// with dv); false when the driver entry point is unavailable or a map is
// rejected.
bool make_input_maps(const void *q, const void *k, const void *v, const float *x, int64_t T_tot,
                     int dk, int dv, int H, int Hk, TcMaps &maps);

// Strong decay: in an item in which some channel's chunk-local gate (log2
// units) moves by more than this inside one 16-token sub-block, the prep
// computes the factored products' at-risk parts from exact gate differences
// (for every other item the factors stay inside [2^-96, 2^96]).
constexpr float STRONG_DECAY_LOG2 = 96.f;

// The prep of every (chunk, head).  flag_count (one word, cleared here) and
// flag_list ([nchunks * H] entries, item = chunk * H + head) receive the
// items under strong decay, for the backward's exact pass.
cudaError_t launch_tc_prep(const TcMaps &maps, const void *q, const void *k, const void *v,
                           const float *x, const float *beta, const GateParams &gp,
                           const SeqInfo &s, int64_t nchunks, int H, int Hk, char *pkg,
                           uint32_t *err, uint32_t *flag_count, uint32_t *flag_list,
                           cudaStream_t st, float *a_out = nullptr);
// a_out: when given, [nchunks, H, 64, 64] fp32 receives A = (I + L)^-1 of
// every item (the backward's intra-chunk stage reuses it).

struct ChainArgs {
  const char *pkg;
  void *out;                    // bf16 [T_tot, H, dv] or null (not written)
  const float *initial_state;   // [N, H, dk, dv] or null
  float *final_state;           // [N, H, dk, dv] or null
  float *h_out;                 // [nchunks, H, dk, dv] or null
  float *v_new_out;             // [T_tot, H, dv] or null
  // head widths of the caller's tensors (64 or 128); the chain works 128
  // wide (the packages of narrow heads carry zeros in the extra channels)
  int dk = 128, dv = 128;
  // bf16 byte images of the chain's operand tiles, per (chunk, head), for
  // the backward (or null): h entering the chunk (32 KB, MN-major K = 128
  // channels), v_new (16 KB, MN-major K = 64 tokens)
  uint8_t *h_img, *vn_img;
  uint32_t *err;
  // test only: one extra wait, on a barrier nothing completes, with a 1 ms
  // limit (the failure path of the bounded waits, without a hang)
  bool test_wait_timeout;
};

cudaError_t launch_tc_chain(const ChainArgs &a, const SeqInfo &s, int H, cudaStream_t st);

// Reverse chain of the state gradient (kda_tc_bwd.cu), from the packages of
// the forward: dh' of every chunk, dv_new and the initial-state gradient.
struct BwdChainArgs {
  const char *pkg;
  const void *d_out;            // bf16 [T_tot, H, V] or null (zeros)
  const float *d_final;         // [N, H, K, V] or null (zeros)
  float *dhn;                   // [nchunks, H, K, V]: gradient of the state leaving each chunk, or null
  float *dvn;                   // [T_tot, H, V] fp32 or null
  float *d_initial;             // [N, H, K, V] or null
  // bf16 byte images per (chunk, head), or null: dh' (the gradient of the
  // state leaving the chunk, 32 KB, layout of the forward's h tile) and
  // -dv_new (16 KB, layout of the forward's v_new tile)
  uint8_t *dh_img, *dv_img;
  uint32_t *err;
};

// State-contraction terms of the backward per (chunk, head), on the tensor
// cores, from the chains' tile images: d(qg) = dO h^T, dw = -dv_new h^T,
// dkg = v_new dh'^T (fp32 [T_tot, H, K]) and d(e^{G_C}) = sum_v dh' . h (fp32
// [nchunks, H, K]).
struct BwdStateArgs {
  const uint8_t *h_img, *vn_img, *dh_img, *dv_img;
  const void *d_out;            // bf16 [T_tot, H, V] or null (zeros)
  float *dqg, *dw, *dkg, *dgc;  // dw fp32 unless dw_img
  uint8_t *dw_img;              // or dw as a bf16 tile image (16 KB per (chunk, head),
                                // rows past the chunk end zero)
  uint32_t *err;
};

// Intra-chunk backward on the tensor cores (kda_tc_bwd_intra.cu).
struct TcIntraArgs {
  const void *q, *k, *v;        // bf16 inputs (q, k with Hk heads)
  const float *g, *beta;        // raw gate input / natural-log g, beta (logits or beta)
  const float *a_in;            // [nchunks, H, 64, 64] A = (I + L)^-1 from the prep
  const float *dqg, *dkg, *dgc; // from the state kernel
  const void *d_out;            // bf16 [T_tot, H, V] or null
  const uint8_t *dv_img, *dw_img, *vn_img;  // -dv_new, dw, v_new tile images
  void *dq, *dk;                // [T_tot, H, K]: bf16, or fp32 per value head (dq_is_f32)
  void *dv;                     // bf16 [T_tot, H, V]
  float *dg, *dbeta;
  float *part_alog, *part_dtb;  // [nchunks, H], [nchunks, H, K]
  uint32_t *err;
  bool dq_is_f32;
};
cudaError_t launch_tc_bwd_intra(const TcIntraArgs &a, const SeqInfo &s, int64_t nchunks, int H, int Hk,
                                const GateParams &gp, cudaStream_t st);
cudaError_t launch_tc_bwd_state(const BwdStateArgs &a, const SeqInfo &s, int64_t nchunks, int H,
                                cudaStream_t st);
cudaError_t launch_tc_bwd_dh(const BwdChainArgs &a, const SeqInfo &s, int H, int64_t T_tot,
                             cudaStream_t st);

// TMA map of a bf16 [T_tot, H, 128] tensor in the forward's v-tile layout.
bool make_value_map(const void *x, int64_t T_tot, int H, CUtensorMap &map);
// The chain's output o, bf16 [T_tot, H, dv]: boxes of 64 channels x 64 tokens
// of one head, 128-byte swizzle (the layout of the chain's staging tile).
bool make_out_map(const void *o, int64_t T_tot, int H, int dv, CUtensorMap &map);

// Segment summary (kda_tc_summary.cu): M [.., dk, dk] and S~ [.., dk, dv] of
// every (segment, head) from the packages of its chunks.
cudaError_t launch_tc_summary(const char *pkg, float *S_tilde, float *M, const SeqInfo &s, int H, int dk,
                              int dv, uint32_t *err, cudaStream_t st);

}  // namespace tcp
}  // namespace kda
