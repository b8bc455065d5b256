// kda_api.cu - the C ABI of include/kda.h: host-side argument checks, the
// workspace plan, and the launch sequence of each call.
//
// Every check runs before anything is enqueued; a failed check returns its
// code and launches nothing.  The library allocates no device memory: all
// scratch lives in the caller's workspace.
#include <stdint.h>
#include <string.h>

#include "kda_profile.h"
#include "kda_internal.cuh"
#include "kda_tc.cuh"

using namespace kda;

namespace {

inline bool mis16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

constexpr uint32_t kKnownFlags = KDA_L2NORM_QK | KDA_BETA_SIGMOID | KDA_GATE_IN_KERNEL |
                                 KDA_USE_EXP2 | KDA_REUSE_PREP | KDA_SAFE_GATE |
                                 KDA_ALLOW_NEG_EIGVAL | KDA_STATE_V_FIRST;
constexpr uint32_t kRejectedFlags = KDA_SAFE_GATE | KDA_ALLOW_NEG_EIGVAL | KDA_STATE_V_FIRST;

// Checks shared by the forward and the summary (everything but the outputs).
kda_status check_common(const kda_fwd_args *a) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (a->B < 1 || a->T < 0 || a->H < 1) return KDA_ERR_INVALID_ARG;
  if (a->flags & ~kKnownFlags) return KDA_ERR_INVALID_ARG;
  if (a->qkv_dtype != KDA_F32 && a->qkv_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  const bool any_tokens = (int64_t)a->B * a->T > 0;
  if (any_tokens && (!a->q || !a->k || !a->v || !a->g || !a->beta)) return KDA_ERR_INVALID_ARG;
  if ((a->flags & KDA_GATE_IN_KERNEL) && !a->a_log) return KDA_ERR_INVALID_ARG;
  if ((a->dk != 64 && a->dk != 128) || (a->dv != 64 && a->dv != 128)) return KDA_ERR_UNSUPPORTED;
  if (a->chunk != BT) return KDA_ERR_UNSUPPORTED;
  if (a->flags & kRejectedFlags) return KDA_ERR_UNSUPPORTED;
  if ((int64_t)a->B * a->T > INT32_MAX) return KDA_ERR_UNSUPPORTED;  // token ids are 32-bit
  if (mis16(a->q) || mis16(a->k) || mis16(a->v) || mis16(a->g) || mis16(a->beta) ||
      mis16(a->a_log) || mis16(a->dt_bias))
    return KDA_ERR_ALIGNMENT;
  return KDA_OK;
}

kda_status check_fwd(const kda_fwd_args *a) {
  kda_status s = check_common(a);
  if (s != KDA_OK) return s;
  if (!a->out && (int64_t)a->B * a->T > 0) return KDA_ERR_INVALID_ARG;
  if (a->cu_seqlens && (a->B != 1 || a->num_seqs < 1)) return KDA_ERR_INVALID_ARG;
  if (mis16(a->out) || mis16(a->initial_state) || mis16(a->final_state) || mis16(a->h_out) ||
      mis16(a->v_new_out) || mis16(a->cu_seqlens))
    return KDA_ERR_ALIGNMENT;
  return KDA_OK;
}

FwdPlan fwd_plan(const kda_fwd_args *a) {
  const bool ragged = a->cu_seqlens != nullptr;
  const int64_t T_tot = (int64_t)a->B * a->T;
  const int32_t N = ragged ? a->num_seqs : a->B;
  return make_plan(T_tot, N, ragged, a->T, a->H, a->dk, a->dv);
}

FwdPlan summary_plan(const kda_fwd_args *a, int32_t num_segments) {
  const int64_t T_tot = (int64_t)a->B * a->T;
  return make_plan(T_tot, num_segments, true, a->T, a->H, a->dk, a->dv);
}

// The tensor-core path takes bf16 inputs with d_k = d_v = 128; every other
// case runs on the CUDA-core path.
bool use_tc(const kda_fwd_args *a) {
  return a->qkv_dtype == KDA_BF16 && a->dk == 128 && a->dv == 128 && (int64_t)a->B * a->T > 0;
}

// Tensor-core workspace: error word, chunk offsets, one package per (chunk, head).
struct TcPlan {
  size_t off_chunk_off, off_pkg, total;
};
TcPlan tc_plan(const FwdPlan &p) {
  TcPlan t{};
  size_t o = 256;
  t.off_chunk_off = o; o = align256(o + sizeof(int32_t) * (size_t)(p.N + 1));
  t.off_pkg = o; o = align256(o + (size_t)p.nchunks * p.H * tcp::PK_BYTES);
  t.total = o;
  return t;
}

size_t plan_bytes(const kda_fwd_args *a, const FwdPlan &p) {
  return use_tc(a) ? tc_plan(p).total : p.total;
}

kda_status check_workspace(const kda_fwd_args *a, const FwdPlan &p) {
  if (!a->workspace || a->workspace_bytes < plan_bytes(a, p)) return KDA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return KDA_ERR_ALIGNMENT;
  return KDA_OK;
}

GateParams gate_params(const kda_fwd_args *a) {
  GateParams gp;
  gp.a_log = a->a_log;
  gp.dt_bias = a->dt_bias;
  gp.scale = a->scale;
  gp.eps = a->eps;
  gp.flags = a->flags;
  return gp;
}

inline kda_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

}  // namespace

extern "C" {

const char *kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_ALIGNMENT: return "KDA_ERR_ALIGNMENT";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_DEVICE_TIMEOUT: return "KDA_ERR_DEVICE_TIMEOUT";
  }
  return "KDA_ERR_UNKNOWN";
}

size_t kda_chunk_fwd_workspace_size(const kda_fwd_args *a) {
  if (check_fwd(a) != KDA_OK) return 0;
  return plan_bytes(a, fwd_plan(a));
}

size_t kda_segment_summary_workspace_size(const kda_fwd_args *a, int32_t num_segments) {
  if (check_common(a) != KDA_OK || num_segments < 1) return 0;
  return plan_bytes(a, summary_plan(a, num_segments));
}

// Launch sequence of the forward.  When events are given, events[i] is
// recorded before stage i and events[count] after the last stage.
static kda_status run_fwd(const kda_fwd_args *a, cudaStream_t st, cudaEvent_t const *ev,
                          int32_t nev) {
  kda_status s = check_fwd(a);
  if (s != KDA_OK) return s;
  const FwdPlan p = fwd_plan(a);
  if ((s = check_workspace(a, p)) != KDA_OK) return s;
  char *ws = static_cast<char *>(a->workspace);

  SeqInfo si{};
  si.bounds = a->cu_seqlens;
  si.chunk_off = reinterpret_cast<int32_t *>(ws + p.off_chunk_off);
  si.T_tot = p.T_tot;
  si.T = a->T;
  si.N = p.N;

  int32_t stage = 0;
  auto mark = [&]() -> cudaError_t {
    cudaError_t r = cudaSuccess;
    if (ev && stage < nev) r = cudaEventRecord(ev[stage], st);
    ++stage;
    return r;
  };
  const bool tc = use_tc(a);
  const size_t off_co = tc ? tc_plan(p).off_chunk_off : p.off_chunk_off;
  si.chunk_off = reinterpret_cast<int32_t *>(ws + off_co);
  tcp::TcMaps maps;
  if (tc && !tcp::make_input_maps(a->q, a->k, a->v, a->g, p.T_tot, a->H, maps)) return KDA_ERR_CUDA;

  const bool reuse = (a->flags & KDA_REUSE_PREP) != 0;
  cudaError_t e = cudaMemsetAsync(ws, 0, 4, st);  // device error word
  if (e == cudaSuccess && si.bounds && !reuse) {
    e = mark();
    if (e == cudaSuccess) e = launch_chunk_map(si, const_cast<int32_t *>(si.chunk_off), st);
  }
  if (tc) {
    char *pkg = ws + tc_plan(p).off_pkg;
    uint32_t *err = reinterpret_cast<uint32_t *>(ws);
    if (e == cudaSuccess && !reuse) e = mark();
    if (e == cudaSuccess && !reuse)
      e = tcp::launch_tc_prep(maps, a->q, a->k, a->g, a->beta, gate_params(a), si, p.nchunks, a->H, pkg, err, st);
    if (e == cudaSuccess) e = mark();
    if (e == cudaSuccess) {
      tcp::ChainArgs ca{};
      ca.pkg = pkg;
      ca.out = a->out;
      ca.initial_state = a->initial_state;
      ca.final_state = a->final_state;
      ca.h_out = a->h_out;
      ca.v_new_out = a->v_new_out;
      ca.err = err;
      e = tcp::launch_tc_chain(tcp::CHAIN_FWD, ca, si, a->H, st);
    }
  } else {
    if (e == cudaSuccess && !reuse) e = mark();
    if (e == cudaSuccess && !reuse)
      e = launch_generic_intra(a->qkv_dtype, a->q, a->k, a->v, a->g, a->beta, gate_params(a), si, p, ws, st);
    if (e == cudaSuccess) e = mark();
    if (e == cudaSuccess) {
      InterOut io{};
      io.out = a->out;
      io.final_state = a->final_state;
      io.h_out = a->h_out;
      io.v_new_out = a->v_new_out;
      io.initial_state = a->initial_state;
      e = launch_generic_inter(a->qkv_dtype, false, io, si, p, ws, st);
    }
  }
  if (e == cudaSuccess) e = mark();
  return cuda_status(e);
}

kda_status kda_chunk_fwd(const kda_fwd_args *a, kda_stream_t stream) {
  return run_fwd(a, reinterpret_cast<cudaStream_t>(stream), nullptr, 0);
}

int32_t kda_chunk_fwd_stages(const kda_fwd_args *a, const char **names, int32_t max_names) {
  if (check_fwd(a) != KDA_OK) return 0;
  const char *list[3];
  int32_t n = 0;
  const bool reuse = (a->flags & KDA_REUSE_PREP) != 0;
  if (a->cu_seqlens && !reuse) list[n++] = "chunk_map";
  if (use_tc(a)) {
    if (!reuse) list[n++] = "tc_prep";
    list[n++] = "tc_chain";
  } else {
    if (!reuse) list[n++] = "intra_generic";
    list[n++] = "inter_generic";
  }
  for (int32_t i = 0; names && i < n && i < max_names; ++i) names[i] = list[i];
  return n;
}

kda_status kda_chunk_fwd_profiled(const kda_fwd_args *a, kda_stream_t stream,
                                  void *const *events, int32_t num_events) {
  const int32_t n = kda_chunk_fwd_stages(a, nullptr, 0);
  if (n == 0) return check_fwd(a) != KDA_OK ? check_fwd(a) : KDA_ERR_INVALID_ARG;
  if (!events || num_events < n + 1) return KDA_ERR_INVALID_ARG;
  for (int32_t i = 0; i <= n; ++i)
    if (!events[i]) return KDA_ERR_INVALID_ARG;
  return run_fwd(a, reinterpret_cast<cudaStream_t>(stream),
                 reinterpret_cast<cudaEvent_t const *>(events), num_events);
}

kda_status kda_segment_summary(const kda_fwd_args *a, const int32_t *seg_bounds,
                               int32_t num_segments, float *M, float *S_tilde,
                               kda_stream_t stream) {
  kda_status s = check_common(a);
  if (s != KDA_OK) return s;
  if (num_segments < 1 || !seg_bounds || !M || !S_tilde) return KDA_ERR_INVALID_ARG;
  if (mis16(seg_bounds) || mis16(M) || mis16(S_tilde)) return KDA_ERR_ALIGNMENT;
  const FwdPlan p = summary_plan(a, num_segments);
  if ((s = check_workspace(a, p)) != KDA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(a->workspace);

  SeqInfo si{};
  si.bounds = seg_bounds;
  si.T_tot = p.T_tot;
  si.T = a->T;
  si.N = num_segments;
  const bool tc = use_tc(a);
  si.chunk_off = reinterpret_cast<int32_t *>(ws + (tc ? tc_plan(p).off_chunk_off : p.off_chunk_off));
  tcp::TcMaps maps;
  if (tc && !tcp::make_input_maps(a->q, a->k, a->v, a->g, p.T_tot, a->H, maps)) return KDA_ERR_CUDA;

  cudaError_t e = cudaMemsetAsync(ws, 0, 4, st);
  if (e == cudaSuccess) e = launch_chunk_map(si, const_cast<int32_t *>(si.chunk_off), st);
  if (tc) {
    char *pkg = ws + tc_plan(p).off_pkg;
    uint32_t *err = reinterpret_cast<uint32_t *>(ws);
    if (e == cudaSuccess)
      e = tcp::launch_tc_prep(maps, a->q, a->k, a->g, a->beta, gate_params(a), si, p.nchunks, a->H, pkg, err, st);
    if (e == cudaSuccess) {
      tcp::ChainArgs ca{};
      ca.pkg = pkg;
      ca.S_tilde = S_tilde;
      ca.M = M;
      ca.err = err;
      e = tcp::launch_tc_chain(tcp::CHAIN_SUMMARY, ca, si, a->H, st);
    }
  } else {
    if (e == cudaSuccess)
      e = launch_generic_intra(a->qkv_dtype, a->q, a->k, a->v, a->g, a->beta, gate_params(a), si, p, ws, st);
    if (e == cudaSuccess) {
      InterOut io{};
      io.S_tilde = S_tilde;
      io.M = M;
      e = launch_generic_inter(a->qkv_dtype, true, io, si, p, ws, st);
    }
  }
  return cuda_status(e);
}

kda_status kda_state_prefix_scan(const float *M, const float *S_tilde, const float *S0,
                                 int32_t num_chains, int32_t num_segments, int32_t H, int32_t dk,
                                 int32_t dv, float *S_in, float *S_final, kda_stream_t stream) {
  if (!M || !S_tilde || !S_in) return KDA_ERR_INVALID_ARG;
  if (num_chains < 1 || num_segments < 1 || H < 1) return KDA_ERR_INVALID_ARG;
  if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return KDA_ERR_UNSUPPORTED;
  if ((int64_t)num_chains * H > INT32_MAX) return KDA_ERR_UNSUPPORTED;
  if (mis16(M) || mis16(S_tilde) || mis16(S0) || mis16(S_in) || mis16(S_final))
    return KDA_ERR_ALIGNMENT;
  return cuda_status(launch_prefix_scan(M, S_tilde, S0, num_chains, num_segments, H, dk, dv, S_in,
                                        S_final, reinterpret_cast<cudaStream_t>(stream)));
}

static kda_status check_copy(const void *cache, kda_dtype cd, int64_t num_rows, int64_t row_stride,
                             int64_t payload, const void *idx, kda_index_dtype it,
                             const void *packed, kda_dtype pd, int64_t n_sel) {
  if (n_sel < 0 || n_sel > INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (num_rows < 1 || payload < 1 || row_stride < payload) return KDA_ERR_INVALID_ARG;
  if ((cd != KDA_F32 && cd != KDA_BF16) || (pd != KDA_F32 && pd != KDA_BF16))
    return KDA_ERR_INVALID_ARG;
  if (it != KDA_I32 && it != KDA_I64) return KDA_ERR_INVALID_ARG;
  if (n_sel > 0 && (!cache || !idx || !packed)) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

kda_status kda_state_gather(const void *cache, kda_dtype cache_dtype, int64_t num_rows,
                            int64_t row_stride_elems, int64_t payload_elems, const void *idx,
                            kda_index_dtype idx_dtype, const bool *flags, int64_t n_sel,
                            void *packed, kda_stream_t stream) {
  kda_status s = check_copy(cache, cache_dtype, num_rows, row_stride_elems, payload_elems, idx,
                            idx_dtype, packed, cache_dtype, n_sel);
  if (s != KDA_OK || n_sel == 0) return s;
  return cuda_status(launch_state_gather(cache, cache_dtype, num_rows, row_stride_elems,
                                         payload_elems, idx, idx_dtype, flags, n_sel, packed,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_state_scatter(void *cache, kda_dtype cache_dtype, int64_t num_rows,
                             int64_t row_stride_elems, int64_t payload_elems, const void *idx,
                             kda_index_dtype idx_dtype, const void *packed, kda_dtype packed_dtype,
                             int64_t n_sel, kda_stream_t stream) {
  kda_status s = check_copy(cache, cache_dtype, num_rows, row_stride_elems, payload_elems, idx,
                            idx_dtype, packed, packed_dtype, n_sel);
  if (s != KDA_OK || n_sel == 0) return s;
  return cuda_status(launch_state_scatter(cache, cache_dtype, num_rows, row_stride_elems,
                                          payload_elems, idx, idx_dtype, packed, packed_dtype,
                                          n_sel, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_get_device_status(void *workspace, kda_stream_t stream) {
  if (!workspace) return KDA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && word) e = cudaMemsetAsync(workspace, 0, 4, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return KDA_ERR_CUDA;
  return word ? KDA_ERR_DEVICE_TIMEOUT : KDA_OK;
}

}  // extern "C"
