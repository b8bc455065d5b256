// kda_api.cu - the C ABI of include/kda.h: host-side argument checks, the
// workspace plan, and the launch sequence of each call.
//
// Every check runs before anything is enqueued; a failed check returns its
// code and launches nothing.  The library allocates no device memory: all
// scratch lives in the caller's workspace.
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "kda_profile.h"
#include "kda_internal.cuh"
#include "kda_tc.cuh"

using namespace kda;

namespace {

inline bool mis16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

constexpr uint32_t kKnownFlags = KDA_L2NORM_QK | KDA_BETA_SIGMOID | KDA_GATE_IN_KERNEL |
                                 KDA_USE_EXP2 | KDA_REUSE_PREP | KDA_SAFE_GATE |
                                 KDA_ALLOW_NEG_EIGVAL | KDA_STATE_V_FIRST |
                                 KDA_LAYOUT_HEAD_MAJOR | KDA_TEST_WAIT_TIMEOUT;
constexpr uint32_t kRejectedFlags = KDA_SAFE_GATE | KDA_ALLOW_NEG_EIGVAL;

inline bool v_first(const kda_fwd_args *a) { return (a->flags & KDA_STATE_V_FIRST) != 0; }
inline bool head_major(const kda_fwd_args *a) { return (a->flags & KDA_LAYOUT_HEAD_MAJOR) != 0; }

// Checks shared by the forward and the summary (everything but the outputs).
kda_status check_common(const kda_fwd_args *a) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (a->B < 1 || a->T < 0 || a->H < 1) return KDA_ERR_INVALID_ARG;
  if (a->Hk < 0 || (a->Hk > 0 && a->H % a->Hk != 0)) return KDA_ERR_INVALID_ARG;
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

// Heads of q and k (grouped key heads when fewer than H).
inline int key_heads(const kda_fwd_args *a) { return a->Hk > 0 ? a->Hk : a->H; }

FwdPlan fwd_plan(const kda_fwd_args *a) {
  const bool ragged = a->cu_seqlens != nullptr;
  const int64_t T_tot = (int64_t)a->B * a->T;
  const int32_t N = ragged ? a->num_seqs : a->B;
  FwdPlan p = make_plan(T_tot, N, ragged, a->T, a->H, a->dk, a->dv);
  p.Hk = key_heads(a);
  return p;
}

FwdPlan summary_plan(const kda_fwd_args *a, int32_t num_segments) {
  const int64_t T_tot = (int64_t)a->B * a->T;
  FwdPlan p = make_plan(T_tot, num_segments, true, a->T, a->H, a->dk, a->dv);
  p.Hk = key_heads(a);
  return p;
}

// The tensor-core path takes bf16 inputs (d_k, d_v of 64 or 128: the
// forward kernels read narrow heads with the extra channels held at zero);
// fp32 inputs run on the CUDA-core path.
bool use_tc(const kda_fwd_args *a) {
  return a->qkv_dtype == KDA_BF16 && (int64_t)a->B * a->T > 0;
}

// Tensor-core workspace: error word (and, 64 bytes in, the count of the
// strong-decay list), chunk offsets, the strong-decay list, one package per
// (chunk, head).
constexpr size_t kFlagCountOff = 64;
struct TcPlan {
  size_t off_chunk_off, off_flags, off_pkg, total;
};
TcPlan tc_plan(const FwdPlan &p) {
  TcPlan t{};
  size_t o = 256;
  t.off_chunk_off = o; o = align256(o + sizeof(int32_t) * (size_t)(p.N + 1));
  t.off_flags = o; o = align256(o + sizeof(uint32_t) * (size_t)p.nchunks * p.H);
  t.off_pkg = o; o = align256(o + (size_t)p.nchunks * p.H * tcp::PK_BYTES);
  t.total = o;
  return t;
}
inline uint32_t *flag_count(char *ws) { return reinterpret_cast<uint32_t *>(ws + kFlagCountOff); }
inline uint32_t *flag_list(char *ws, const FwdPlan &p) {
  return reinterpret_cast<uint32_t *>(ws + tc_plan(p).off_flags);
}

// K-first copies of the caller's V-first states (initial, final, h_out),
// after the forward's own workspace.
struct VfPlan {
  size_t off_init, off_fin, off_hout, total;
};
VfPlan vf_plan(const kda_fwd_args *a, const FwdPlan &p, size_t base) {
  VfPlan v{};
  size_t o = base;
  if (v_first(a)) {
    const size_t SS = (size_t)p.N * p.H * p.K * p.V * 4;
    if (a->initial_state) { v.off_init = o; o = align256(o + SS); }
    if (a->final_state) { v.off_fin = o; o = align256(o + SS); }
    if (a->h_out) { v.off_hout = o; o = align256(o + (size_t)p.nchunks * p.H * p.K * p.V * 4); }
  }
  v.total = o;
  return v;
}

// Token-major copies of a head-major call's per-token tensors, after the
// rest of the workspace.  The inputs always; out / v_new_out / d_out when
// the call has them (with_out: out is written by the call).
struct HmPlan {
  size_t off_q, off_k, off_v, off_g, off_b, off_o, off_vn, total;
};
HmPlan hm_plan(const kda_fwd_args *a, bool with_out, size_t base) {
  HmPlan m{};
  const size_t tok = (size_t)a->B * a->T, esz = a->qkv_dtype == KDA_BF16 ? 2 : 4;
  const size_t Hk = a->Hk > 0 ? a->Hk : a->H;
  size_t o = base;
  m.off_q = o; o = align256(o + tok * Hk * a->dk * esz);
  m.off_k = o; o = align256(o + tok * Hk * a->dk * esz);
  m.off_v = o; o = align256(o + tok * a->H * a->dv * esz);
  m.off_g = o; o = align256(o + tok * a->H * a->dk * 4);
  m.off_b = o; o = align256(o + tok * a->H * 4);
  m.off_o = m.off_vn = 0;
  if (with_out) { m.off_o = o; o = align256(o + tok * a->H * a->dv * esz); }
  if (with_out && a->v_new_out) { m.off_vn = o; o = align256(o + tok * a->H * a->dv * 4); }
  m.total = o;
  return m;
}

// (batch, tokens per batch row) of the swap between the layouts.
inline void hm_dims(const kda_fwd_args *a, int64_t &B, int64_t &T) {
  B = a->cu_seqlens ? 1 : a->B;
  T = a->cu_seqlens ? (int64_t)a->B * a->T : a->T;
}

// Head-major inputs -> token-major copies in the workspace ws; b points at them.
cudaError_t hm_inputs_in(const kda_fwd_args *a, char *ws, const HmPlan &m, kda_fwd_args *b,
                         cudaStream_t st) {
  int64_t B, T;
  hm_dims(a, B, T);
  const int esz = a->qkv_dtype == KDA_BF16 ? 2 : 4, Hk = a->Hk > 0 ? a->Hk : a->H;
  b->flags &= ~(uint32_t)KDA_LAYOUT_HEAD_MAJOR;
  b->q = ws + m.off_q;
  b->k = ws + m.off_k;
  b->v = ws + m.off_v;
  b->g = reinterpret_cast<float *>(ws + m.off_g);
  b->beta = reinterpret_cast<float *>(ws + m.off_b);
  cudaError_t e = launch_swap_token_head(a->q, ws + m.off_q, B, Hk, T, a->dk * esz, true, st);
  if (e == cudaSuccess) e = launch_swap_token_head(a->k, ws + m.off_k, B, Hk, T, a->dk * esz, true, st);
  if (e == cudaSuccess) e = launch_swap_token_head(a->v, ws + m.off_v, B, a->H, T, a->dv * esz, true, st);
  if (e == cudaSuccess) e = launch_swap_token_head(a->g, ws + m.off_g, B, a->H, T, a->dk * 4, true, st);
  if (e == cudaSuccess) e = launch_swap_token_head(a->beta, ws + m.off_b, B, a->H, T, 4, true, st);
  return e;
}

// Narrow heads (bf16, d_k or d_v = 64) in the backward and the backward
// summary: their 128-wide tensor-core kernels run on zero-padded copies in
// the workspace (the forward and the summary read narrow heads directly).
// Exact: a padded key channel has zero q and k and no decay (gate input
// -1e30 through the in-kernel softplus, or a zero log-decay), a padded value
// channel zero v, so the padded rows and columns of every state stay zero and
// the real channels see the unpadded problem; the padded outputs are dropped.
bool narrow_tc(const kda_fwd_args *a) {
  return a->qkv_dtype == KDA_BF16 && (a->dk != 128 || a->dv != 128) && (int64_t)a->B * a->T > 0;
}
kda_fwd_args wide_args(const kda_fwd_args *a) {
  kda_fwd_args w = *a;
  w.dk = w.dv = 128;
  return w;
}
constexpr size_t kWideState = 128 * 128 * 4;  // one padded fp32 state

// Padded q, k, v, gate input, dt_bias (and initial state) from offset o on.
struct PadIn {
  size_t off_q, off_k, off_v, off_g, off_dtb, off_init, end;
};
PadIn pad_in_plan(const kda_fwd_args *a, size_t o, bool with_init) {
  PadIn m{};
  const size_t tok = (size_t)a->B * a->T, Hk = key_heads(a);
  m.off_q = o; o = align256(o + tok * Hk * 256);
  m.off_k = o; o = align256(o + tok * Hk * 256);
  m.off_v = o; o = align256(o + tok * a->H * 256);
  m.off_g = o; o = align256(o + tok * a->H * 512);
  if (a->dt_bias) { m.off_dtb = o; o = align256(o + (size_t)a->H * 512); }
  if (with_init && a->initial_state) {
    m.off_init = o;
    o = align256(o + (size_t)fwd_plan(a).N * a->H * kWideState);
  }
  m.end = o;
  return m;
}

// Rows of w elements (esz bytes) widened to 128 with `fill`, and back.
cudaError_t widen_rows(const void *src, void *dst, int64_t rows, int w, int esz, uint32_t fill,
                       cudaStream_t st) {
  return launch_window_copy(src, dst, rows, 1, w * esz, 1, 128 * esz, fill, nullptr, 0, st);
}
cudaError_t narrow_rows(const void *src, void *dst, int64_t rows, int w, int esz, cudaStream_t st) {
  return launch_window_copy(src, dst, rows, 1, 128 * esz, 1, w * esz, 0u, nullptr, 0, st);
}
// fp32 r x c states (the caller's state dimensions) in 128 x 128 ones, and back.
cudaError_t widen_states(const float *src, float *dst, int64_t n, int r, int c, cudaStream_t st) {
  return launch_window_copy(src, dst, n, r, c * 4, 128, 512, 0u, nullptr, 0, st);
}
cudaError_t narrow_states(const float *src, float *dst, int64_t n, int r, int c, const int32_t *count,
                          int per_count, cudaStream_t st) {
  return launch_window_copy(src, dst, n, 128, 512, r, c * 4, 0u, count, per_count, st);
}

// w's q, k, v, g, dt_bias moved onto 128-wide copies (copied when `copy`);
// tensors that are 128 wide already are used in place.
cudaError_t pad_inputs(const kda_fwd_args *a, char *ws, const PadIn &m, kda_fwd_args *w, bool copy,
                       cudaStream_t st) {
  const int64_t tok = (int64_t)a->B * a->T, Hk = key_heads(a);
  float gfill = (a->flags & KDA_GATE_IN_KERNEL) ? -1e30f : 0.f;  // no decay on padded channels
  uint32_t gbits;
  memcpy(&gbits, &gfill, 4);
  cudaError_t e = cudaSuccess;
  if (a->dk != 128) {
    w->q = ws + m.off_q;
    w->k = ws + m.off_k;
    w->g = reinterpret_cast<float *>(ws + m.off_g);
    w->dt_bias = a->dt_bias ? reinterpret_cast<float *>(ws + m.off_dtb) : nullptr;
    if (copy) {
      e = widen_rows(a->q, ws + m.off_q, tok * Hk, a->dk, 2, 0u, st);
      if (e == cudaSuccess) e = widen_rows(a->k, ws + m.off_k, tok * Hk, a->dk, 2, 0u, st);
      if (e == cudaSuccess) e = widen_rows(a->g, ws + m.off_g, tok * a->H, a->dk, 4, gbits, st);
      if (e == cudaSuccess && a->dt_bias) e = widen_rows(a->dt_bias, ws + m.off_dtb, a->H, a->dk, 4, 0u, st);
    }
  }
  if (a->dv != 128) {
    w->v = ws + m.off_v;
    if (copy && e == cudaSuccess) e = widen_rows(a->v, ws + m.off_v, tok * a->H, a->dv, 2, 0u, st);
  }
  return e;
}

// The forward's or the segment summary's own workspace, before the layout
// copies.
size_t inner_bytes(const kda_fwd_args *a, const FwdPlan &p) {
  return use_tc(a) ? tc_plan(p).total : p.total;
}
// Where the chunk offsets (and, for packed sequences, the chunk count) live.
size_t chunk_off_pos(const kda_fwd_args *a, const FwdPlan &p) {
  return use_tc(a) ? tc_plan(p).off_chunk_off : p.off_chunk_off;
}

size_t plan_bytes(const kda_fwd_args *a, const FwdPlan &p) {
  const size_t base = vf_plan(a, p, inner_bytes(a, p)).total;
  return head_major(a) ? hm_plan(a, true, base).total : base;
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
  gp.dk = a->dk;
  gp.dv = a->dv;
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
// recorded before stage i and events[count] after the last stage.  The device
// error word is cleared first unless keep_err (the blocks of a host-IO call
// share one word, cleared once).
static kda_status run_fwd_kfirst(const kda_fwd_args *a, cudaStream_t st, cudaEvent_t const *ev,
                                 int32_t nev, bool keep_err);

// V-first states: converted to K-first copies in the workspace around the
// K-first forward ("Hyper-Parallel Chunk KDA current implementation design",
// section 4.1, state_v_first).
static kda_status run_fwd(const kda_fwd_args *a, cudaStream_t st, cudaEvent_t const *ev,
                          int32_t nev, bool keep_err = false) {
  kda_status s = check_fwd(a);
  if (s != KDA_OK) return s;
  if (head_major(a) && (int64_t)a->B * a->T > 0) {
    // head-major tensors: token-major copies around the token-major forward
    const FwdPlan p = fwd_plan(a);
    if ((s = check_workspace(a, p)) != KDA_OK) return s;
    kda_fwd_args b = *a;
    b.flags &= ~(uint32_t)KDA_LAYOUT_HEAD_MAJOR;
    const size_t base = plan_bytes(&b, p);
    const HmPlan m = hm_plan(a, true, base);
    char *ws = static_cast<char *>(a->workspace);
    cudaError_t e = hm_inputs_in(a, ws, m, &b, st);
    b.out = ws + m.off_o;
    b.v_new_out = a->v_new_out ? reinterpret_cast<float *>(ws + m.off_vn) : nullptr;
    b.workspace_bytes = base;
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if ((s = run_fwd(&b, st, ev, nev, keep_err)) != KDA_OK) return s;
    int64_t B, T;
    hm_dims(a, B, T);
    const int esz = a->qkv_dtype == KDA_BF16 ? 2 : 4;
    e = launch_swap_token_head(b.out, a->out, B, a->H, T, a->dv * esz, false, st);
    if (e == cudaSuccess && a->v_new_out)
      e = launch_swap_token_head(b.v_new_out, a->v_new_out, B, a->H, T, a->dv * 4, false, st);
    return cuda_status(e);
  }
  if (!v_first(a)) return run_fwd_kfirst(a, st, ev, nev, keep_err);
  const FwdPlan p = fwd_plan(a);
  if ((s = check_workspace(a, p)) != KDA_OK) return s;
  char *ws = static_cast<char *>(a->workspace);
  const VfPlan v = vf_plan(a, p, inner_bytes(a, p));
  kda_fwd_args b = *a;
  b.flags &= ~(uint32_t)KDA_STATE_V_FIRST;
  b.workspace_bytes = v.off_init ? v.off_init : (v.off_fin ? v.off_fin : (v.off_hout ? v.off_hout : v.total));
  cudaError_t e = cudaSuccess;
  if (a->initial_state) {
    b.initial_state = reinterpret_cast<float *>(ws + v.off_init);
    e = launch_transpose_states(a->initial_state, const_cast<float *>(b.initial_state),
                                (int64_t)p.N * p.H, p.V, p.K, nullptr, 0, st);
  }
  if (a->final_state) b.final_state = reinterpret_cast<float *>(ws + v.off_fin);
  if (a->h_out) b.h_out = reinterpret_cast<float *>(ws + v.off_hout);
  if (e != cudaSuccess) return KDA_ERR_CUDA;
  if ((s = run_fwd_kfirst(&b, st, ev, nev, keep_err)) != KDA_OK) return s;
  if (a->final_state)
    e = launch_transpose_states(b.final_state, a->final_state, (int64_t)p.N * p.H, p.K, p.V, nullptr,
                                0, st);
  if (e == cudaSuccess && a->h_out) {
    // only the chunks that exist: their count is on the device for packed sequences
    const int32_t *count =
        a->cu_seqlens ? reinterpret_cast<const int32_t *>(ws + chunk_off_pos(a, p)) + p.N : nullptr;
    e = launch_transpose_states(b.h_out, a->h_out, p.nchunks * p.H, p.K, p.V, count, p.H, st);
  }
  return cuda_status(e);
}

static kda_status run_fwd_kfirst(const kda_fwd_args *a, cudaStream_t st, cudaEvent_t const *ev,
                                 int32_t nev, bool keep_err) {
  kda_status s;
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
  const bool reuse = (a->flags & KDA_REUSE_PREP) != 0;
  tcp::TcMaps maps;  // the prep's input maps (no prep with KDA_REUSE_PREP)
  if (tc && !reuse &&
      !tcp::make_input_maps(a->q, a->k, a->v, a->g, p.T_tot, a->dk, a->dv, a->H, p.Hk, maps))
    return KDA_ERR_CUDA;

  cudaError_t e = keep_err ? cudaSuccess : cudaMemsetAsync(ws, 0, 4, st);  // device error word
  if (e == cudaSuccess && si.bounds && !reuse) {
    e = mark();
    if (e == cudaSuccess) e = launch_chunk_map(si, const_cast<int32_t *>(si.chunk_off), st);
  }
  if (tc) {
    char *pkg = ws + tc_plan(p).off_pkg;
    uint32_t *err = reinterpret_cast<uint32_t *>(ws);
    if (e == cudaSuccess && !reuse) e = mark();
    if (e == cudaSuccess && !reuse)
      e = tcp::launch_tc_prep(maps, a->q, a->k, a->v, a->g, a->beta, gate_params(a), si, p.nchunks,
                              a->H, p.Hk, pkg, err, flag_count(ws), flag_list(ws, p), st);
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
      ca.dk = a->dk;
      ca.dv = a->dv;
      ca.test_wait_timeout = (a->flags & KDA_TEST_WAIT_TIMEOUT) != 0;
      e = tcp::launch_tc_chain(ca, si, a->H, st);
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

}  // extern "C"

namespace {

// Host-IO forward: the batch in blocks of KDA_HOST_BLOCK_TOKENS tokens of
// every sequence, with the copies on two streams of the library's own.
struct HostPlan {
  int64_t Tb;                        // tokens per block (last block: fewer)
  int64_t nblk;
  size_t off_sub, sub_bytes;         // workspace of one block's forward
  size_t off_in[2], in_bytes;        // staged q, k, v, g, beta of a block
  size_t off_out[2], out_bytes;      // staged o of a block
  size_t off_state, state_bytes;     // carried state when final_state is NULL
  size_t total;
  size_t esz;                        // bytes per q/k/v/o element
};

kda_status check_host(const kda_fwd_args *a) {
  kda_status s = check_fwd(a);
  if (s != KDA_OK) return s;
  if (a->cu_seqlens || a->h_out || a->v_new_out || (a->flags & (KDA_REUSE_PREP | KDA_LAYOUT_HEAD_MAJOR)))
    return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

// Sub-problem of block t: the same arguments on [B, Tb_t] staged tokens.
kda_fwd_args block_args(const kda_fwd_args *a, int64_t Tb_t) {
  kda_fwd_args b = *a;
  b.T = (int32_t)Tb_t;
  return b;
}

HostPlan host_plan(const kda_fwd_args *a) {
  HostPlan h{};
  h.esz = a->qkv_dtype == KDA_BF16 ? 2 : 4;
  h.Tb = a->T < KDA_HOST_BLOCK_TOKENS ? a->T : KDA_HOST_BLOCK_TOKENS;
  h.nblk = h.Tb > 0 ? (a->T + h.Tb - 1) / h.Tb : 0;
  kda_fwd_args b = block_args(a, h.Tb);
  if (v_first(a)) {  // every block converts its entering and leaving state (size only)
    static const float placeholder[4] = {0.f, 0.f, 0.f, 0.f};
    b.initial_state = b.final_state = const_cast<float *>(placeholder);
  }
  size_t o = 0;
  h.off_sub = o;
  h.sub_bytes = plan_bytes(&b, fwd_plan(&b));
  o = align256(o + h.sub_bytes);
  const size_t tok = (size_t)a->B * h.Tb * a->H;  // token-heads of a block
  const size_t tok_k = (size_t)a->B * h.Tb * key_heads(a);
  h.in_bytes = tok_k * 2 * a->dk * h.esz + tok * ((size_t)a->dv * h.esz + (size_t)a->dk * 4 + 4);
  h.out_bytes = tok * a->dv * h.esz;
  for (int j = 0; j < 2; ++j) { h.off_in[j] = o; o = align256(o + h.in_bytes); }
  for (int j = 0; j < 2; ++j) { h.off_out[j] = o; o = align256(o + h.out_bytes); }
  h.state_bytes = a->final_state ? 0 : (size_t)a->B * a->H * a->dk * a->dv * 4;
  h.off_state = o;
  o = align256(o + h.state_bytes);
  h.total = o;
  return h;
}

struct HostStreams {
  cudaStream_t in = nullptr, out = nullptr;
};

// The library's two copy streams on the current device, created once.
kda_status host_streams(HostStreams *hs) {
  static std::mutex mu;
  static HostStreams cache[64];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  HostStreams &c = cache[dev];
  if (!c.in) {
    if (cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking) != cudaSuccess) {
      cudaStreamDestroy(c.in);
      c.in = nullptr;
      return KDA_ERR_CUDA;
    }
  }
  *hs = c;
  return KDA_OK;
}

// Copy rows [t0, t0 + n) of every sequence of a [B, T, H, width] host tensor
// into a contiguous [B, n, H, width] device block.
cudaError_t copy_in(void *dst, const void *src, int64_t B, int64_t T, int64_t t0, int64_t n,
                    size_t row_bytes, cudaStream_t s) {
  return cudaMemcpy2DAsync(dst, n * row_bytes, static_cast<const char *>(src) + t0 * row_bytes,
                           T * row_bytes, n * row_bytes, B, cudaMemcpyHostToDevice, s);
}

}  // namespace

extern "C" {

size_t kda_chunk_fwd_host_workspace_size(const kda_fwd_args *a) {
  if (check_host(a) != KDA_OK) return 0;
  return host_plan(a).total;
}

kda_status kda_chunk_fwd_host(const kda_fwd_args *a, kda_stream_t stream) {
  kda_status s = check_host(a);
  if (s != KDA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((int64_t)a->B * a->T == 0) return run_fwd(a, st, nullptr, 0);  // no tokens: no copies
  const HostPlan hp = host_plan(a);
  if (!a->workspace || a->workspace_bytes < hp.total) return KDA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return KDA_ERR_ALIGNMENT;
  HostStreams hs;
  if ((s = host_streams(&hs)) != KDA_OK) return s;
  char *ws = static_cast<char *>(a->workspace);
  float *carry = a->final_state ? a->final_state : reinterpret_cast<float *>(ws + hp.off_state);

  cudaEvent_t ev[7] = {};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 7 && e == cudaSuccess; ++i)
    e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
  cudaEvent_t ev_start = ev[6], *ev_in = ev, *ev_comp = ev + 2, *ev_out = ev + 4;
  // the workspace and the device buffers are free once earlier work on `stream` is done
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + hp.off_sub, 0, 4, st);  // shared error word
  if (e == cudaSuccess) e = cudaEventRecord(ev_start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hs.in, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hs.out, ev_start, 0);

  const int64_t B = a->B, T = a->T, H = a->H;
  const size_t rq = (size_t)key_heads(a) * a->dk * hp.esz, rv = (size_t)H * a->dv * hp.esz;
  const size_t rg = (size_t)H * a->dk * 4, rb = (size_t)H * 4;
  for (int64_t t = 0; t < hp.nblk && e == cudaSuccess; ++t) {
    const int j = (int)(t & 1);
    const int64_t t0 = t * hp.Tb, n = (T - t0) < hp.Tb ? (T - t0) : hp.Tb;
    char *in = ws + hp.off_in[j];
    const size_t nb = (size_t)B * n;  // staged rows
    void *dq = in, *dk = in + nb * rq, *dv = in + 2 * nb * rq, *dg = in + 2 * nb * rq + nb * rv;
    void *db = static_cast<char *>(dg) + nb * rg;
    // inputs of block t (after block t - 2 has finished reading this buffer)
    if (t >= 2) e = cudaStreamWaitEvent(hs.in, ev_comp[j], 0);
    if (e == cudaSuccess) e = copy_in(dq, a->q, B, T, t0, n, rq, hs.in);
    if (e == cudaSuccess) e = copy_in(dk, a->k, B, T, t0, n, rq, hs.in);
    if (e == cudaSuccess) e = copy_in(dv, a->v, B, T, t0, n, rv, hs.in);
    if (e == cudaSuccess) e = copy_in(dg, a->g, B, T, t0, n, rg, hs.in);
    if (e == cudaSuccess) e = copy_in(db, a->beta, B, T, t0, n, rb, hs.in);
    if (e == cudaSuccess) e = cudaEventRecord(ev_in[j], hs.in);
    // the forward of block t (after block t - 2's o has left this buffer)
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_in[j], 0);
    if (e == cudaSuccess && t >= 2) e = cudaStreamWaitEvent(st, ev_out[j], 0);
    if (e != cudaSuccess) break;
    kda_fwd_args b = block_args(a, n);
    b.q = dq; b.k = dk; b.v = dv; b.g = static_cast<float *>(dg); b.beta = static_cast<float *>(db);
    b.out = ws + hp.off_out[j];
    b.initial_state = t == 0 ? a->initial_state : carry;
    b.final_state = carry;
    b.workspace = ws + hp.off_sub;
    b.workspace_bytes = hp.sub_bytes;
    if ((s = run_fwd(&b, st, nullptr, 0, true)) != KDA_OK) break;
    e = cudaEventRecord(ev_comp[j], st);
    // o of block t back to the host
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hs.out, ev_comp[j], 0);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(static_cast<char *>(a->out) + t0 * rv, T * rv, ws + hp.off_out[j], n * rv,
                            n * rv, B, cudaMemcpyDeviceToHost, hs.out);
    if (e == cudaSuccess) e = cudaEventRecord(ev_out[j], hs.out);
  }
  // `stream` passes the call once the last copy out is done
  if (e == cudaSuccess && s == KDA_OK) e = cudaStreamWaitEvent(st, ev_out[(hp.nblk - 1) & 1], 0);
  for (int i = 0; i < 7; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  if (s != KDA_OK) return s;
  return cuda_status(e);
}

kda_status kda_segment_summary(const kda_fwd_args *a, const int32_t *seg_bounds,
                               int32_t num_segments, float *M, float *S_tilde,
                               kda_stream_t stream) {
  kda_status s = check_common(a);
  if (s != KDA_OK) return s;
  if (v_first(a)) return KDA_ERR_UNSUPPORTED;  // summaries are K-first
  if (num_segments < 1 || !seg_bounds || !M || !S_tilde) return KDA_ERR_INVALID_ARG;
  if (mis16(seg_bounds) || mis16(M) || mis16(S_tilde)) return KDA_ERR_ALIGNMENT;
  if (head_major(a) && (int64_t)a->B * a->T > 0) {  // token-major copies of the inputs
    kda_fwd_args b = *a;
    b.flags &= ~(uint32_t)KDA_LAYOUT_HEAD_MAJOR;
    const size_t base = plan_bytes(&b, summary_plan(&b, num_segments));
    const HmPlan m = hm_plan(a, false, base);
    if (!a->workspace || a->workspace_bytes < m.total) return KDA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return KDA_ERR_ALIGNMENT;
    cudaStream_t st0 = reinterpret_cast<cudaStream_t>(stream);
    if (hm_inputs_in(a, static_cast<char *>(a->workspace), m, &b, st0) != cudaSuccess) return KDA_ERR_CUDA;
    b.workspace_bytes = base;
    return kda_segment_summary(&b, seg_bounds, num_segments, M, S_tilde, stream);
  }
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
  if (tc && !tcp::make_input_maps(a->q, a->k, a->v, a->g, p.T_tot, a->dk, a->dv, a->H, p.Hk, maps))
    return KDA_ERR_CUDA;

  cudaError_t e = cudaMemsetAsync(ws, 0, 4, st);
  if (e == cudaSuccess) e = launch_chunk_map(si, const_cast<int32_t *>(si.chunk_off), st);
  if (tc) {
    char *pkg = ws + tc_plan(p).off_pkg;
    uint32_t *err = reinterpret_cast<uint32_t *>(ws);
    if (e == cudaSuccess)
      e = tcp::launch_tc_prep(maps, a->q, a->k, a->v, a->g, a->beta, gate_params(a), si, p.nchunks,
                              a->H, p.Hk, pkg, err, flag_count(ws), flag_list(ws, p), st);
    if (e == cudaSuccess) e = tcp::launch_tc_summary(pkg, S_tilde, M, si, a->H, a->dk, a->dv, err, st);
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

kda_status kda_recurrent_step(const kda_decode_args *a, kda_stream_t stream) {
  if (!a || a->N < 0 || a->T < 1 || a->H < 1) return KDA_ERR_INVALID_ARG;
  if (a->Hk < 0 || (a->Hk > 0 && a->H % a->Hk != 0)) return KDA_ERR_INVALID_ARG;
  if (a->flags & ~kKnownFlags) return KDA_ERR_INVALID_ARG;
  if (a->flags & (kRejectedFlags | KDA_REUSE_PREP | KDA_LAYOUT_HEAD_MAJOR))
    return KDA_ERR_UNSUPPORTED;  // V-first is taken
  if ((a->dk != 64 && a->dk != 128) || (a->dv != 64 && a->dv != 128)) return KDA_ERR_UNSUPPORTED;
  if (a->qkv_dtype != KDA_F32 && a->qkv_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (a->cache_dtype != KDA_F32 && a->cache_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (a->idx_dtype != KDA_I32 && a->idx_dtype != KDA_I64) return KDA_ERR_INVALID_ARG;
  if (a->num_rows < 1 || a->row_stride_elems < (int64_t)a->H * a->dk * a->dv) return KDA_ERR_INVALID_ARG;
  if ((a->flags & KDA_GATE_IN_KERNEL) && !a->a_log) return KDA_ERR_INVALID_ARG;
  if (a->N == 0) return KDA_OK;
  if (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->out || !a->cache || !a->idx)
    return KDA_ERR_INVALID_ARG;
  if ((int64_t)a->N * a->T * a->H > INT32_MAX) return KDA_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  GateParams gp;
  gp.a_log = a->a_log;
  gp.dt_bias = a->dt_bias;
  gp.scale = a->scale;
  gp.eps = a->eps;
  gp.flags = a->flags;
  return cuda_status(launch_decode(a->qkv_dtype, a->cache_dtype, a->idx_dtype, a->dk, a->dv, a->N,
                                   a->T, a->H, a->Hk > 0 ? a->Hk : a->H, a->q, a->k, a->v, a->g,
                                   a->beta, gp, a->out, a->cache,
                                   a->num_rows, a->row_stride_elems, a->idx, a->init_flags,
                                   (a->flags & KDA_STATE_V_FIRST) != 0, st));
}

}  // extern "C"

namespace {

kda_status check_bwd(const kda_bwd_args *b) {
  if (!b) return KDA_ERR_INVALID_ARG;
  const kda_fwd_args *a = &b->fwd;
  kda_status s = check_common(a);
  if (s != KDA_OK) return s;
  if (a->cu_seqlens && (a->B != 1 || a->num_seqs < 1)) return KDA_ERR_INVALID_ARG;
  if (a->flags & KDA_REUSE_PREP) return KDA_ERR_UNSUPPORTED;
  if ((int64_t)a->B * a->T > 0 && (!b->dq || !b->dk || !b->dv || !b->dg || !b->dbeta))
    return KDA_ERR_INVALID_ARG;
  if (mis16(a->initial_state) || mis16(a->cu_seqlens) || mis16(b->d_out) || mis16(b->d_final_state) ||
      mis16(b->dq) || mis16(b->dk) || mis16(b->dv) || mis16(b->dg) || mis16(b->dbeta) ||
      mis16(b->da_log) || mis16(b->ddt_bias) || mis16(b->d_initial_state))
    return KDA_ERR_ALIGNMENT;
  return KDA_OK;
}

// Backward workspace: the generic forward plan (recomputed intermediates),
// then the states, state gradients and per-token scratch of the backward.
struct BwdPlan {
  FwdPlan f;
  size_t off_h, off_vn, off_dhn, off_dvn, off_dqg, off_dw, off_dkg, off_dgc, off_palog, off_pdtb;
  size_t off_himg, off_vnimg, off_dhimg, off_dvimg, off_dwimg;  // bf16 tile images (tensor-core path)
  size_t off_dqv, off_dkv;
  size_t off_ainv;                                // A of every chunk (tensor-core recompute)
  size_t off_vf_init, off_vf_dfin, off_vf_dinit;  // K-first copies of V-first states
  size_t total;
};

// The recompute runs on the tensor-core forward (packages) where the forward
// does, else on the generic one (fp32 per-token intermediates).
BwdPlan bwd_plan(const kda_bwd_args *b) {
  BwdPlan p{};
  p.f = fwd_plan(&b->fwd);
  const size_t th = (size_t)p.f.T_tot * p.f.H, ch = (size_t)p.f.nchunks * p.f.H;
  const size_t K = p.f.K, V = p.f.V;
  const bool tc = use_tc(&b->fwd);
  size_t o = tc ? tc_plan(p.f).total : p.f.total;
  p.off_h = p.off_dhn = p.off_himg = p.off_vnimg = p.off_dhimg = p.off_dvimg = p.off_dwimg = 0;
  p.off_vn = p.off_dvn = p.off_dw = 0;
  if (tc) {  // states and state gradients travel as bf16 operand-tile images
    p.off_himg = o;  o = align256(o + ch * 32768);
    p.off_vnimg = o; o = align256(o + ch * 16384);
    p.off_dhimg = o; o = align256(o + ch * 32768);
    p.off_dvimg = o; o = align256(o + ch * 16384);
    p.off_dwimg = o; o = align256(o + ch * 16384);
  } else {  // fp32 states, state gradients, v_new and its gradient, dw (CUDA-core path only)
    p.off_h = o;     o = align256(o + 4 * ch * K * V);
    p.off_dhn = o;   o = align256(o + 4 * ch * K * V);
    p.off_vn = o;    o = align256(o + 4 * th * V);
    p.off_dvn = o;   o = align256(o + 4 * th * V);
    p.off_dw = o;    o = align256(o + 4 * th * K);
  }
  p.off_dqg = o;   o = align256(o + 4 * th * K);
  p.off_dkg = o;   o = align256(o + 4 * th * K);
  p.off_dgc = o;   o = align256(o + 4 * ch * K);
  p.off_palog = o; o = align256(o + 4 * ch);
  p.off_pdtb = o;  o = align256(o + 4 * ch * K);
  p.off_dqv = p.off_dkv = 0;
  if (p.f.Hk != p.f.H) {
    p.off_dqv = o; o = align256(o + 4 * th * K);
    p.off_dkv = o; o = align256(o + 4 * th * K);
  }
  p.off_ainv = 0;
  if (use_tc(&b->fwd)) { p.off_ainv = o; o = align256(o + 4 * ch * BT * BT); }
  p.off_vf_init = p.off_vf_dfin = p.off_vf_dinit = 0;
  if (v_first(&b->fwd)) {
    const size_t SS = 4 * (size_t)p.f.N * p.f.H * K * V;
    if (b->fwd.initial_state) { p.off_vf_init = o; o = align256(o + SS); }
    if (b->d_final_state) { p.off_vf_dfin = o; o = align256(o + SS); }
    if (b->d_initial_state) { p.off_vf_dinit = o; o = align256(o + SS); }
  }
  p.total = o;
  return p;
}

// Backward of a narrow-head problem: the wide backward's workspace, the padded
// inputs and cotangents, then 128-wide gradients.
struct PadBwd {
  size_t inner;
  PadIn in;
  size_t off_dfin, off_do, off_dq, off_dk, off_dv, off_dg, off_ddtb, off_dinit, total;
};
kda_bwd_args wide_bwd(const kda_bwd_args *b) {
  kda_bwd_args c = *b;
  c.fwd = wide_args(&b->fwd);
  return c;
}
PadBwd pad_bwd_plan(const kda_bwd_args *b) {
  PadBwd f{};
  const kda_fwd_args *a = &b->fwd;
  const kda_bwd_args c = wide_bwd(b);
  f.inner = bwd_plan(&c).total;
  f.in = pad_in_plan(a, f.inner, true);
  size_t o = f.in.end;
  const size_t tok = (size_t)a->B * a->T, Hk = key_heads(a), ns = (size_t)fwd_plan(a).N * a->H;
  if (b->d_final_state) { f.off_dfin = o; o = align256(o + ns * kWideState); }
  if (b->d_out) { f.off_do = o; o = align256(o + tok * a->H * 256); }
  f.off_dq = o; o = align256(o + tok * Hk * 256);
  f.off_dk = o; o = align256(o + tok * Hk * 256);
  f.off_dv = o; o = align256(o + tok * a->H * 256);
  f.off_dg = o; o = align256(o + tok * a->H * 512);
  if (b->ddt_bias) { f.off_ddtb = o; o = align256(o + (size_t)a->H * 512); }
  if (b->d_initial_state) { f.off_dinit = o; o = align256(o + ns * kWideState); }
  f.total = o;
  return f;
}
size_t bwd_total(const kda_bwd_args *b) {
  return narrow_tc(&b->fwd) ? pad_bwd_plan(b).total : bwd_plan(b).total;
}

// Segment backward summary of a narrow-head problem: padded d_out, 128-wide E.
struct PadSegBwd {
  size_t inner;
  PadIn in;
  size_t off_do, off_E, total;
};
PadSegBwd pad_segbwd_plan(const kda_fwd_args *a, int32_t S) {
  PadSegBwd f{};
  const kda_fwd_args w = wide_args(a);
  f.inner = tc_plan(summary_plan(&w, S)).total;
  f.in = pad_in_plan(a, f.inner, false);
  size_t o = f.in.end;
  f.off_do = o; o = align256(o + (size_t)a->B * a->T * a->H * 256);
  f.off_E = o; o = align256(o + (size_t)S * a->H * kWideState);
  f.total = o;
  return f;
}
size_t segbwd_total(const kda_fwd_args *a, int32_t S) {
  if (narrow_tc(a)) return pad_segbwd_plan(a, S).total;
  const FwdPlan p = summary_plan(a, S);  // packages or generic intermediates
  return use_tc(a) ? tc_plan(p).total : p.total;
}

// Narrow heads: the 128-wide backward on padded copies, gradients cut back;
// dbeta and dA_log (no head-width dimension) go to the caller's buffers.
kda_status run_bwd_narrow(const kda_bwd_args *b, kda_stream_t stream) {
  const kda_fwd_args *a = &b->fwd;
  const PadBwd m = pad_bwd_plan(b);
  if (!b->workspace || b->workspace_bytes < m.total) return KDA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(b->workspace) & 255u) return KDA_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(b->workspace);
  auto f32 = [&](size_t off) { return reinterpret_cast<float *>(ws + off); };
  kda_bwd_args c = wide_bwd(b);
  c.workspace_bytes = m.inner;
  const int64_t tok = (int64_t)a->B * a->T, Hk = key_heads(a), ns = (int64_t)fwd_plan(a).N * a->H;
  const bool vf = v_first(a);
  const int sr = vf ? a->dv : a->dk, sc = vf ? a->dk : a->dv;  // the caller's state dimensions
  const bool nk = a->dk != 128, nv = a->dv != 128;
  cudaError_t e = pad_inputs(a, ws, m.in, &c.fwd, true, st);
  if (e == cudaSuccess && a->initial_state) {
    c.fwd.initial_state = f32(m.in.off_init);
    e = widen_states(a->initial_state, f32(m.in.off_init), ns, sr, sc, st);
  }
  if (e == cudaSuccess && b->d_final_state) {
    c.d_final_state = f32(m.off_dfin);
    e = widen_states(b->d_final_state, f32(m.off_dfin), ns, sr, sc, st);
  }
  if (e == cudaSuccess && b->d_out && nv) {
    c.d_out = ws + m.off_do;
    e = widen_rows(b->d_out, ws + m.off_do, tok * a->H, a->dv, 2, 0u, st);
  }
  if (nk) {
    c.dq = ws + m.off_dq;
    c.dk = ws + m.off_dk;
    c.dg = f32(m.off_dg);
    c.ddt_bias = b->ddt_bias ? f32(m.off_ddtb) : nullptr;
  }
  if (nv) c.dv = ws + m.off_dv;
  c.d_initial_state = b->d_initial_state ? f32(m.off_dinit) : nullptr;
  if (e != cudaSuccess) return KDA_ERR_CUDA;
  kda_status s = kda_chunk_bwd(&c, stream);
  if (s != KDA_OK) return s;
  if (nk) {
    e = narrow_rows(c.dq, b->dq, tok * Hk, a->dk, 2, st);
    if (e == cudaSuccess) e = narrow_rows(c.dk, b->dk, tok * Hk, a->dk, 2, st);
    if (e == cudaSuccess) e = narrow_rows(c.dg, b->dg, tok * a->H, a->dk, 4, st);
    if (e == cudaSuccess && b->ddt_bias) e = narrow_rows(c.ddt_bias, b->ddt_bias, a->H, a->dk, 4, st);
  }
  if (e == cudaSuccess && nv) e = narrow_rows(c.dv, b->dv, tok * a->H, a->dv, 2, st);
  if (e == cudaSuccess && b->d_initial_state)
    e = narrow_states(c.d_initial_state, b->d_initial_state, ns, sr, sc, nullptr, 0, st);
  return cuda_status(e);
}

}  // namespace

extern "C" {

// Head-major backward: token-major copies of the inputs and d_out (the
// forward's out region), then of the gradients dq, dk, dv, dg, dbeta.
struct HmBwd {
  HmPlan in;
  size_t off_dq, off_dk, off_dv, off_dg, off_db, total;
};
HmBwd hm_bwd_plan(const kda_bwd_args *b, size_t base) {
  HmBwd h{};
  const kda_fwd_args *a = &b->fwd;
  h.in = hm_plan(a, true, base);
  const size_t tok = (size_t)a->B * a->T, esz = a->qkv_dtype == KDA_BF16 ? 2 : 4;
  const size_t Hk = a->Hk > 0 ? a->Hk : a->H;
  size_t o = h.in.total;
  h.off_dq = o; o = align256(o + tok * Hk * a->dk * esz);
  h.off_dk = o; o = align256(o + tok * Hk * a->dk * esz);
  h.off_dv = o; o = align256(o + tok * a->H * a->dv * esz);
  h.off_dg = o; o = align256(o + tok * a->H * a->dk * 4);
  h.off_db = o; o = align256(o + tok * a->H * 4);
  h.total = o;
  return h;
}

size_t kda_chunk_bwd_workspace_size(const kda_bwd_args *b) {
  if (check_bwd(b) != KDA_OK) return 0;
  const size_t base = bwd_total(b);
  return head_major(&b->fwd) ? hm_bwd_plan(b, base).total : base;
}

kda_status kda_chunk_bwd(const kda_bwd_args *b, kda_stream_t stream) {
  kda_status s = check_bwd(b);
  if (s != KDA_OK) return s;
  const kda_fwd_args *a = &b->fwd;
  if (head_major(a) && (int64_t)a->B * a->T > 0) {
    const size_t base = bwd_total(b);
    const HmBwd m = hm_bwd_plan(b, base);
    if (!b->workspace || b->workspace_bytes < m.total) return KDA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(b->workspace) & 255u) return KDA_ERR_ALIGNMENT;
    cudaStream_t st0 = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(b->workspace);
    int64_t B, T;
    hm_dims(a, B, T);
    const int esz = a->qkv_dtype == KDA_BF16 ? 2 : 4, Hk = a->Hk > 0 ? a->Hk : a->H;
    kda_bwd_args c = *b;
    cudaError_t e = hm_inputs_in(a, ws, m.in, &c.fwd, st0);
    if (e == cudaSuccess && b->d_out) {
      e = launch_swap_token_head(b->d_out, ws + m.in.off_o, B, a->H, T, a->dv * esz, true, st0);
      c.d_out = ws + m.in.off_o;
    }
    c.dq = ws + m.off_dq;
    c.dk = ws + m.off_dk;
    c.dv = ws + m.off_dv;
    c.dg = reinterpret_cast<float *>(ws + m.off_dg);
    c.dbeta = reinterpret_cast<float *>(ws + m.off_db);
    c.workspace_bytes = base;
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if ((s = kda_chunk_bwd(&c, stream)) != KDA_OK) return s;
    e = launch_swap_token_head(c.dq, b->dq, B, Hk, T, a->dk * esz, false, st0);
    if (e == cudaSuccess) e = launch_swap_token_head(c.dk, b->dk, B, Hk, T, a->dk * esz, false, st0);
    if (e == cudaSuccess) e = launch_swap_token_head(c.dv, b->dv, B, a->H, T, a->dv * esz, false, st0);
    if (e == cudaSuccess) e = launch_swap_token_head(c.dg, b->dg, B, a->H, T, a->dk * 4, false, st0);
    if (e == cudaSuccess) e = launch_swap_token_head(c.dbeta, b->dbeta, B, a->H, T, 4, false, st0);
    return cuda_status(e);
  }
  if (narrow_tc(a)) return run_bwd_narrow(b, stream);
  const BwdPlan p = bwd_plan(b);
  if (!b->workspace || b->workspace_bytes < p.total) return KDA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(b->workspace) & 255u) return KDA_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(b->workspace);
  auto f32 = [&](size_t off) { return reinterpret_cast<float *>(ws + off); };

  const bool tc = use_tc(a);
  SeqInfo si{};
  si.bounds = a->cu_seqlens;
  si.chunk_off = reinterpret_cast<int32_t *>(ws + (tc ? tc_plan(p.f).off_chunk_off : p.f.off_chunk_off));
  si.T_tot = p.f.T_tot;
  si.T = a->T;
  si.N = p.f.N;
  const GateParams gp = gate_params(a);
  uint32_t *err = reinterpret_cast<uint32_t *>(ws);
  char *pkg = ws + tc_plan(p.f).off_pkg;
  tcp::TcMaps maps;
  if (tc && !tcp::make_input_maps(a->q, a->k, a->v, a->g, p.f.T_tot, a->dk, a->dv, a->H, p.f.Hk, maps))
    return KDA_ERR_CUDA;

  // V-first states: K-first copies in the workspace
  const float *init = a->initial_state, *dfin = b->d_final_state;
  float *dinit = b->d_initial_state;
  const int64_t nstates = (int64_t)p.f.N * p.f.H;
  cudaError_t e = cudaSuccess;
  if (v_first(a)) {
    if (init) {
      e = launch_transpose_states(init, f32(p.off_vf_init), nstates, p.f.V, p.f.K, nullptr, 0, st);
      init = f32(p.off_vf_init);
    }
    if (e == cudaSuccess && dfin) {
      e = launch_transpose_states(dfin, f32(p.off_vf_dfin), nstates, p.f.V, p.f.K, nullptr, 0, st);
      dfin = f32(p.off_vf_dfin);
    }
    if (dinit) dinit = f32(p.off_vf_dinit);
  }

  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, 4, st);
  if (e == cudaSuccess && si.bounds) e = launch_chunk_map(si, const_cast<int32_t *>(si.chunk_off), st);
  // recompute: the per-chunk intermediates, the state entering every chunk, v_new
  if (tc) {
    if (e == cudaSuccess)
      e = tcp::launch_tc_prep(maps, a->q, a->k, a->v, a->g, a->beta, gp, si, p.f.nchunks, a->H, p.f.Hk,
                              pkg, err, flag_count(ws), flag_list(ws, p.f), st, f32(p.off_ainv));
    if (e == cudaSuccess) {
      tcp::ChainArgs ca{};
      ca.pkg = pkg;
      ca.initial_state = init;
      ca.v_new_out = nullptr;  // v_new travels as the bf16 tile image
      ca.h_img = reinterpret_cast<uint8_t *>(ws + p.off_himg);
      ca.vn_img = reinterpret_cast<uint8_t *>(ws + p.off_vnimg);
      ca.err = err;
      e = tcp::launch_tc_chain(ca, si, a->H, st);
    }
  } else {
    if (e == cudaSuccess && p.f.T_tot > 0)
      e = launch_generic_intra(a->qkv_dtype, a->q, a->k, a->v, a->g, a->beta, gp, si, p.f, ws, st);
    if (e == cudaSuccess && p.f.T_tot > 0) {
      InterOut io{};
      io.h_out = f32(p.off_h);
      io.v_new_out = f32(p.off_vn);
      io.initial_state = init;
      e = launch_generic_inter(a->qkv_dtype, false, io, si, p.f, ws, st);
    }
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + p.off_palog, 0, p.off_pdtb - p.off_palog, st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(ws + p.off_pdtb, 0, 4 * (size_t)p.f.nchunks * p.f.H * p.f.K, st);
  if (e == cudaSuccess) {
    BwdLaunch l{};
    l.s = si;
    l.H = p.f.H;
    l.Hk = p.f.Hk;
    l.nchunks = p.f.T_tot > 0 ? p.f.nchunks : 0;
    l.q = a->q; l.k = a->k; l.v = a->v; l.g = a->g; l.beta = a->beta;
    l.gp = gp;
    l.d_out = b->d_out;
    l.d_final = dfin;
    if (!tc) {  // the generic intermediates (the tensor-core path keeps packages instead)
      l.w = f32(p.f.off_w); l.qg = f32(p.f.off_qg); l.kg = f32(p.f.off_kg);
      l.aqk = f32(p.f.off_aqk); l.gc = f32(p.f.off_gc);
    }
    l.h = tc ? nullptr : f32(p.off_h);
    l.vn = tc ? nullptr : f32(p.off_vn);
    l.dhn = tc ? nullptr : f32(p.off_dhn);
    l.dvn = tc ? nullptr : f32(p.off_dvn);
    l.dw = tc ? nullptr : f32(p.off_dw);
    l.dqg = f32(p.off_dqg);
    l.dkg = f32(p.off_dkg); l.dgc = f32(p.off_dgc);
    l.part_alog = f32(p.off_palog); l.part_dtb = f32(p.off_pdtb);
    l.dqv = p.off_dqv ? f32(p.off_dqv) : nullptr;
    l.dkv = p.off_dkv ? f32(p.off_dkv) : nullptr;
    l.dq = b->dq; l.dk = b->dk; l.dv = b->dv;
    l.dg = b->dg; l.dbeta = b->dbeta; l.d_initial = dinit;
    l.a_in = tc ? f32(p.off_ainv) : nullptr;
    if (tc) {  // reverse chain on the tensor cores from the packages
      tcp::BwdChainArgs ba{};
      ba.pkg = pkg;
      ba.d_out = b->d_out;
      ba.d_final = dfin;
      ba.dvn = l.dvn;
      ba.d_initial = dinit;
      ba.dh_img = reinterpret_cast<uint8_t *>(ws + p.off_dhimg);
      ba.dv_img = reinterpret_cast<uint8_t *>(ws + p.off_dvimg);
      ba.err = err;
      e = tcp::launch_tc_bwd_dh(ba, si, a->H, p.f.T_tot, st);
      uint8_t *sa_dw_img = reinterpret_cast<uint8_t *>(ws + p.off_dwimg);
      if (e == cudaSuccess) {  // the state-contraction terms on the tensor cores
        tcp::BwdStateArgs sa{};
        sa.h_img = reinterpret_cast<const uint8_t *>(ws + p.off_himg);
        sa.vn_img = reinterpret_cast<const uint8_t *>(ws + p.off_vnimg);
        sa.dh_img = ba.dh_img;
        sa.dv_img = ba.dv_img;
        sa.d_out = b->d_out;
        sa.dqg = l.dqg; sa.dw = l.dw; sa.dkg = l.dkg; sa.dgc = l.dgc;
        sa.dw_img = reinterpret_cast<uint8_t *>(ws + p.off_dwimg);
        sa.err = err;
        e = tcp::launch_tc_bwd_state(sa, si, p.f.nchunks, a->H, st);
      }
      if (e == cudaSuccess) {  // the intra-chunk backward on the tensor cores
        const bool grouped = p.f.Hk != p.f.H;
        tcp::TcIntraArgs ia{};
        ia.q = a->q; ia.k = a->k; ia.v = a->v; ia.g = a->g; ia.beta = a->beta;
        ia.a_in = l.a_in;
        ia.dqg = l.dqg; ia.dkg = l.dkg; ia.dgc = l.dgc;
        ia.d_out = b->d_out;
        ia.dv_img = ba.dv_img;
        ia.dw_img = sa_dw_img;
        ia.vn_img = reinterpret_cast<const uint8_t *>(ws + p.off_vnimg);
        ia.dq = grouped ? static_cast<void *>(l.dqv) : b->dq;
        ia.dk = grouped ? static_cast<void *>(l.dkv) : b->dk;
        ia.dq_is_f32 = grouped;
        ia.dv = b->dv; ia.dg = b->dg; ia.dbeta = b->dbeta;
        ia.part_alog = l.part_alog; ia.part_dtb = l.part_dtb;
        ia.err = err;
        e = tcp::launch_tc_bwd_intra(ia, si, p.f.nchunks, a->H, p.f.Hk, gp, st);
        // the chunks the prep listed under strong decay, again, exactly
        if (e == cudaSuccess)
          e = launch_bwd_intra_list(l, ba.dv_img, ia.vn_img, sa_dw_img, flag_count(ws), flag_list(ws, p.f),
                                    st);
        if (e == cudaSuccess && grouped)
          e = launch_bwd_group_sum(a->qkv_dtype, p.f.T_tot, a->H, p.f.Hk, a->dk, l.dqv, l.dkv, b->dq, b->dk,
                                   st);
      }
    } else {
      e = launch_generic_bwd(a->qkv_dtype, a->dk, a->dv, l, st);
    }
  }
  if (e == cudaSuccess)
    e = launch_bwd_param_reduce(p.f.nchunks, p.f.H, p.f.K, f32(p.off_palog), f32(p.off_pdtb), b->da_log,
                                b->ddt_bias, st);
  if (e == cudaSuccess && v_first(a) && dinit)
    e = launch_transpose_states(dinit, b->d_initial_state, nstates, p.f.K, p.f.V, nullptr, 0, st);
  return cuda_status(e);
}

size_t kda_segment_bwd_summary_workspace_size(const kda_fwd_args *a, int32_t num_segments) {
  if (check_common(a) != KDA_OK || num_segments < 1) return 0;
  const size_t base = segbwd_total(a, num_segments);
  return head_major(a) ? hm_plan(a, true, base).total : base;  // + token-major inputs and d_out
}

kda_status kda_segment_bwd_summary(const kda_fwd_args *a, const void *d_out,
                                   const int32_t *seg_bounds, int32_t num_segments, float *E,
                                   kda_stream_t stream) {
  kda_status s = check_common(a);
  if (s != KDA_OK) return s;
  if (a->flags & (KDA_REUSE_PREP | KDA_STATE_V_FIRST)) return KDA_ERR_UNSUPPORTED;
  if (num_segments < 1 || !seg_bounds || !E) return KDA_ERR_INVALID_ARG;
  if (mis16(seg_bounds) || mis16(E) || mis16(d_out)) return KDA_ERR_ALIGNMENT;
  if (head_major(a) && (int64_t)a->B * a->T > 0) {  // token-major copies of the inputs, d_out
    kda_fwd_args b = *a;
    b.flags &= ~(uint32_t)KDA_LAYOUT_HEAD_MAJOR;
    const size_t base = segbwd_total(&b, num_segments);
    const HmPlan m = hm_plan(a, true, base);
    if (!a->workspace || a->workspace_bytes < m.total) return KDA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return KDA_ERR_ALIGNMENT;
    cudaStream_t st0 = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(a->workspace);
    cudaError_t e = hm_inputs_in(a, ws, m, &b, st0);
    const void *dO = nullptr;
    if (e == cudaSuccess && d_out) {
      int64_t B, T;
      hm_dims(a, B, T);
      e = launch_swap_token_head(d_out, ws + m.off_o, B, a->H, T,
                                 a->dv * (a->qkv_dtype == KDA_BF16 ? 2 : 4), true, st0);
      dO = ws + m.off_o;
    }
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    b.workspace_bytes = base;
    return kda_segment_bwd_summary(&b, dO, seg_bounds, num_segments, E, stream);
  }
  if (narrow_tc(a)) {  // the 128-wide reverse chain on padded copies, E cut back
    const PadSegBwd m = pad_segbwd_plan(a, num_segments);
    if (!a->workspace || a->workspace_bytes < m.total) return KDA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return KDA_ERR_ALIGNMENT;
    cudaStream_t st0 = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(a->workspace);
    kda_fwd_args w = wide_args(a);
    w.workspace_bytes = m.inner;
    cudaError_t e = pad_inputs(a, ws, m.in, &w, true, st0);
    const void *dO = d_out;
    if (e == cudaSuccess && d_out && a->dv != 128) {
      e = widen_rows(d_out, ws + m.off_do, (int64_t)a->B * a->T * a->H, a->dv, 2, 0u, st0);
      dO = ws + m.off_do;
    }
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    float *Ew = reinterpret_cast<float *>(ws + m.off_E);
    if ((s = kda_segment_bwd_summary(&w, dO, seg_bounds, num_segments, Ew, stream)) != KDA_OK) return s;
    return cuda_status(narrow_states(Ew, E, (int64_t)num_segments * a->H, a->dk, a->dv, nullptr, 0, st0));
  }
  const FwdPlan p = summary_plan(a, num_segments);
  const bool tc = use_tc(a);
  if (!a->workspace || a->workspace_bytes < (tc ? tc_plan(p).total : p.total)) return KDA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return KDA_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(a->workspace);
  auto f32 = [&](size_t off) { return reinterpret_cast<float *>(ws + off); };
  SeqInfo si{};
  si.bounds = seg_bounds;
  si.chunk_off = reinterpret_cast<int32_t *>(ws + (tc ? tc_plan(p).off_chunk_off : p.off_chunk_off));
  si.T_tot = p.T_tot;
  si.T = a->T;
  si.N = num_segments;
  tcp::TcMaps maps;
  if (tc && !tcp::make_input_maps(a->q, a->k, a->v, a->g, p.T_tot, a->dk, a->dv, a->H, p.Hk, maps))
    return KDA_ERR_CUDA;
  cudaError_t e = cudaMemsetAsync(ws, 0, 4, st);
  if (e == cudaSuccess) e = launch_chunk_map(si, const_cast<int32_t *>(si.chunk_off), st);
  if (tc) {  // the packages, then the reverse chain on the tensor cores
    char *pkg = ws + tc_plan(p).off_pkg;
    uint32_t *err = reinterpret_cast<uint32_t *>(ws);
    if (e == cudaSuccess)
      e = tcp::launch_tc_prep(maps, a->q, a->k, a->v, a->g, a->beta, gate_params(a), si, p.nchunks, a->H,
                              p.Hk, pkg, err, flag_count(ws), flag_list(ws, p), st);
    if (e == cudaSuccess) {
      tcp::BwdChainArgs ba{};
      ba.pkg = pkg;
      ba.d_out = d_out;
      ba.d_initial = E;  // d_final = 0, dhn / dvn not kept
      ba.err = err;
      e = tcp::launch_tc_bwd_dh(ba, si, a->H, p.T_tot, st);
    }
    return cuda_status(e);
  }
  if (e == cudaSuccess && p.T_tot > 0)
    e = launch_generic_intra(a->qkv_dtype, a->q, a->k, a->v, a->g, a->beta, gate_params(a), si, p, ws,
                             st);
  if (e == cudaSuccess) {
    BwdLaunch l{};
    l.s = si;
    l.H = p.H;
    l.Hk = p.Hk;
    l.d_out = d_out;
    l.w = f32(p.off_w); l.qg = f32(p.off_qg); l.kg = f32(p.off_kg);
    l.aqk = f32(p.off_aqk); l.gc = f32(p.off_gc);
    l.d_initial = E;  // d_final = 0, dhn / dvn not kept
    e = launch_bwd_dh(a->qkv_dtype, a->dk, a->dv, l, st);
  }
  return cuda_status(e);
}

kda_status kda_state_grad_scan(const float *M, const float *E, const float *dS_final,
                               int32_t num_chains, int32_t num_segments, int32_t H, int32_t dk,
                               int32_t dv, float *dS_out, float *dS_initial, kda_stream_t stream) {
  if (!M || !E || !dS_out) return KDA_ERR_INVALID_ARG;
  if (num_chains < 1 || num_segments < 1 || H < 1) return KDA_ERR_INVALID_ARG;
  if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return KDA_ERR_UNSUPPORTED;
  if ((int64_t)num_chains * H > INT32_MAX) return KDA_ERR_UNSUPPORTED;
  if (mis16(M) || mis16(E) || mis16(dS_final) || mis16(dS_out) || mis16(dS_initial))
    return KDA_ERR_ALIGNMENT;
  return cuda_status(launch_prefix_scan(M, E, dS_final, num_chains, num_segments, H, dk, dv, dS_out,
                                        dS_initial, reinterpret_cast<cudaStream_t>(stream), true));
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
