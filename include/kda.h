/*
 * kda.h - C ABI of the GB300 (sm_103a) chunked Kimi Delta Attention library.
 *
 * The library computes, on one GPU, the forward pass of KDA, the per-channel
 * gated delta rule
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = scale * S_t^T q_t,          alpha_t = exp(g_t) per key channel,
 * in chunks of 64 tokens, together with the segment affine summary (M, S~)
 * of a token range, the ordered prefix scan S <- M_j S + S~_j that composes
 * summaries, and the gather/scatter of per-request states between a cache
 * pool and packed rows.
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers unless a comment says "host".
 *    The caller allocates and owns every buffer; the library allocates no
 *    device memory, keeps no pointer after a call returns, and holds no
 *    global state besides a lazily filled per-process table of driver entry
 *    points.
 *  - Calls are asynchronous on the given stream (NULL = legacy default
 *    stream).  Argument checks run on the host before anything is launched;
 *    a failed check returns an error code and launches nothing.  A launch
 *    failure returns KDA_ERR_CUDA.  No call aborts, traps or prints.
 *  - Tensors are dense and row-major ("contiguous") in the shapes given.
 *    Every tensor pointer must be 16-byte aligned (KDA_ERR_ALIGNMENT).
 *  - Recurrent states are fp32 and K-first: state[..., c, j] with c a key
 *    channel (d_k) and j a value channel (d_v).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stdbool.h>
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the same handle type), spelled without CUDA headers. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,    /* null required pointer, bad size or shape      */
  KDA_ERR_UNSUPPORTED = 2,    /* a valid request this library does not compute */
  KDA_ERR_ALIGNMENT = 3,      /* a tensor pointer is not 16-byte aligned       */
  KDA_ERR_WORKSPACE = 4,      /* workspace missing or smaller than required    */
  KDA_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed          */
  KDA_ERR_DEVICE_TIMEOUT = 6  /* a bounded device-side wait gave up            */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;
typedef enum { KDA_I32 = 0, KDA_I64 = 1 } kda_index_dtype;

/* Flags of kda_fwd_args.flags.  The first four follow the keyword arguments
 * use_qk_l2norm_in_kernel, use_beta_sigmoid_in_kernel, use_gate_in_kernel and
 * use_exp2 of npu_chunk_kda ("Hyper-Parallel Chunk KDA current implementation
 * design", section 4 and 4.1). */
enum {
  KDA_L2NORM_QK = 1u << 0,      /* q^ = q (sum q^2 + eps)^-1/2, same for k       */
  KDA_BETA_SIGMOID = 1u << 1,   /* beta = 1 / (1 + exp(-b)) of the given logits  */
  KDA_GATE_IN_KERNEL = 1u << 2, /* g = -exp(a_log[h]) softplus(x + dt_bias[h,c]) */
  KDA_USE_EXP2 = 1u << 3,       /* work in base 2 internally; same result        */
  /* kda_chunk_fwd only: the workspace already holds this call's intra-chunk
   * results (the per-chunk preparation of q, k, v, g, beta: "FwdPrepare" of
   * "Hyper-Parallel Chunk KDA current implementation design" section 6.3),
   * left there by the immediately preceding kda_segment_summary on the same
   * inputs, flags and workspace with seg_bounds equal to this call's
   * cu_seqlens (or by a kda_chunk_fwd with the same arguments); only the
   * inter-chunk chain runs.  Caller precondition, not checked. */
  KDA_REUSE_PREP = 1u << 4,
  /* Named on the pages without a formula (safe_gate/lower_bound,
   * allow_neg_eigval): always rejected with KDA_ERR_UNSUPPORTED. */
  KDA_SAFE_GATE = 1u << 8,
  KDA_ALLOW_NEG_EIGVAL = 1u << 9,
  /* state_v_first (same design, section 4.1): every recurrent state the call
   * takes or returns - initial_state, final_state, h_out of the forward;
   * initial_state, d_final_state, d_initial_state of the backward; the pool
   * states of kda_recurrent_step - has its last two dimensions as [dv, dk]
   * instead of [dk, dv].  The library computes K-first and converts at the
   * boundary (through workspace copies, included in the workspace sizes).
   * kda_segment_summary and kda_segment_bwd_summary return K-first summaries
   * and reject the flag with KDA_ERR_UNSUPPORTED. */
  KDA_STATE_V_FIRST = 1u << 10,
  /* Head-major token layouts (same design, section 4.2): BNSD [B, H, T, D]
   * instead of BSND [B, T, H, D] without cu_seqlens, NTD [H, T_total, D]
   * instead of TND [T_total, H, D] with it.  Applies to q, k (Hk heads), v,
   * g, beta ([B, H, T] / [H, T_total]), out and v_new_out of the forward and
   * summaries, and to d_out, dq, dk, dv, dg, dbeta of the backward.  The
   * kernels work token-major; the library converts at the boundary through
   * workspace copies (included in the workspace sizes).  Rejected with
   * KDA_ERR_UNSUPPORTED by kda_chunk_fwd_host and kda_recurrent_step. */
  KDA_LAYOUT_HEAD_MAJOR = 1u << 11,
  /* Test only (no counterpart on the pages): exercises the device-side
   * failure path without faulting or hanging the GPU.  In a kda_chunk_fwd
   * (or kda_chunk_fwd_static_scratch) that runs the tensor-core chain, the
   * chain kernel also waits, once, on a barrier that nothing completes,
   * with a 1 ms limit; it then records KDA_ERR_DEVICE_TIMEOUT in the
   * workspace's error word, lets the copies it started land, releases its
   * tensor memory and returns.  The call itself returns KDA_OK; its outputs
   * are undefined; kda_get_device_status (kda_static_scratch_status) then
   * reports the timeout.  Ignored by the CUDA-core path (no waits there). */
  KDA_TEST_WAIT_TIMEOUT = 1u << 30
};

/*
 * Arguments of the chunked forward ("Hyper-Parallel Chunk KDA current
 * implementation design", section 4, npu_chunk_kda; "KDA Chunk Backward -
 * TPU/Pallas Kernel Design", section 1 and 1.2 for the chunk formulas).
 *
 * Layout: tokens are BSND [B, T, H, D] when cu_seqlens is NULL, or TND
 * [T_total, H, D] packed sequences when cu_seqlens is given (then B must be
 * 1 and T = T_total).  q and k have d_k channels, v and out d_v channels.
 * Grouped key heads (same design, section 4.2: q/k may have fewer heads
 * than v): q and k carry Hk heads, v, g, beta, out and every state carry the
 * H value heads; value head h reads key head h / (H / Hk).  Hk = 0 means
 * Hk = H (every field named H below is the value-head count).
 * Every sequence starts from its own initial state (section 6.5 of the same
 * design); chunks restart at every sequence start, the last one may be
 * partial.
 */
typedef struct {
  int32_t B, T, H;          /* batch, tokens per sequence (or T_total), heads    */
  int32_t dk, dv;           /* head dims; each must be 64 or 128                 */
  int32_t chunk;            /* chunk length; must be 64                          */
  kda_dtype qkv_dtype;      /* dtype of q, k, v and out                          */
  const void *q, *k;        /* [B,T,H,dk] or [T_total,H,dk], qkv_dtype           */
  const void *v;            /* [B,T,H,dv] or [T_total,H,dv], qkv_dtype           */
  const float *g;           /* [.., H, dk] fp32: raw gate input x when           */
                            /* KDA_GATE_IN_KERNEL, else natural-log decay g <= 0 */
  const float *a_log;       /* [H] fp32; required with KDA_GATE_IN_KERNEL        */
  const float *dt_bias;     /* [H, dk] fp32 or NULL (= zeros)                    */
  const float *beta;        /* [.., H] fp32: logits with KDA_BETA_SIGMOID        */
  float scale;              /* output scale, usually dk^-1/2                     */
  float eps;                /* L2-norm epsilon, usually 1e-6                     */
  const float *initial_state; /* [N, H, dk, dv] fp32 or NULL (= zeros); [N, H,    */
                              /* dv, dk] with KDA_STATE_V_FIRST (so every state) */
  const int32_t *cu_seqlens;  /* device [num_seqs+1] token offsets or NULL;      */
                              /* caller precondition: 0 = cu[0] <= .. <= cu[N] = T */
  int32_t num_seqs;         /* N when cu_seqlens is given; ignored otherwise     */
  uint32_t flags;           /* KDA_* flags above                                 */
  void *out;                /* [.., H, dv] qkv_dtype, written                    */
  float *final_state;       /* [N, H, dk, dv] fp32 or NULL (not written)         */
  float *h_out;             /* [num_chunks, H, dk, dv] fp32 state entering each  */
                            /* chunk (chunks numbered sequence by sequence), or  */
                            /* NULL; num_chunks = sum over sequences of ceil(len/64) */
  float *v_new_out;         /* [.., H, dv] fp32 corrected values u - w h, or NULL */
  void *workspace;          /* device scratch, >= kda_chunk_fwd_workspace_size   */
  size_t workspace_bytes;   /* and 256-byte aligned                              */
  int32_t Hk;               /* key heads of q and k: 0 (= H) or a divisor of H;  */
                            /* q, k are [.., Hk, dk]; otherwise INVALID_ARG      */
} kda_fwd_args;

/* Bytes of workspace kda_chunk_fwd needs for these arguments (0 when the
 * arguments are invalid).  Depends only on sizes, dtype, flags and which
 * optional outputs are requested. */
size_t kda_chunk_fwd_workspace_size(const kda_fwd_args *args);

/* The chunked KDA forward: out, and final_state / h_out / v_new_out when
 * given.  N = B without cu_seqlens, num_seqs with it.
 * Arithmetic: bf16 inputs with dk = dv = 128 run on the tensor cores (bf16
 * operands, fp32 accumulation, inverse and state); in a chunk in which some
 * channel's gate falls by more than 96 log2 units (about 66 nats) inside one
 * of its 16-token sub-blocks, the parts of the decay-factored products that
 * could leave the floating-point range are computed from exact gate
 * differences in fp32 on the CUDA cores, so strong decay costs time, not
 * accuracy.  bf16 heads with dk or dv = 64 run the same 128-wide kernels,
 * which read the narrow tensors directly and hold the missing channels at
 * zero (zero q and k, no decay, zero v: the extra state rows and columns stay
 * zero) and write only the caller's channels: exact.  fp32 inputs run in
 * fp32 on the CUDA cores.
 * With no tokens (B*T == 0, or only empty sequences) the final state is the
 * initial state; q/k/v/g/beta/out may then be NULL.
 * Errors: KDA_ERR_INVALID_ARG (null q/k/v/g/beta/out with tokens, B or H < 1,
 * T < 0, Hk < 0 or not dividing H, a_log missing with KDA_GATE_IN_KERNEL,
 * cu_seqlens with B != 1), KDA_ERR_UNSUPPORTED
 * (dk or dv not 64/128, chunk != 64, KDA_SAFE_GATE / KDA_ALLOW_NEG_EIGVAL),
 * KDA_ERR_ALIGNMENT, KDA_ERR_WORKSPACE, KDA_ERR_CUDA. */
kda_status kda_chunk_fwd(const kda_fwd_args *args, kda_stream_t stream);

/* Size of the library's own scratch array used by
 * kda_chunk_fwd_static_scratch: 32 MiB on every GPU the library runs on. */
#define KDA_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * kda_chunk_fwd for callers that cannot allocate device memory (the pages
 * have no counterpart of this call).  A plugin whose host owns all device
 * memory, or a latency-critical path where cudaMalloc is not allowed, passes
 * its inputs and outputs exactly as for kda_chunk_fwd; args->workspace and
 * args->workspace_bytes are ignored and the scratch comes from a fixed
 * KDA_STATIC_SCRATCH_BYTES array inside the library, which no call allocates
 * or frees (it exists from the time the library is loaded on a GPU until the
 * process exits).
 *  - Limit: the problem's kda_chunk_fwd_workspace_size must not exceed
 *    KDA_STATIC_SCRATCH_BYTES, else KDA_ERR_WORKSPACE and nothing is
 *    launched (roughly: up to about 450 chunk-heads on the bf16 d=128 path,
 *    e.g. B=1, T=2048, H=14).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls share the one array: calls that overlap on the GPU (e.g. on
 *    two streams) race and must be serialised by the caller.  Leftover
 *    contents of earlier calls do not affect results: every call rewrites
 *    what it reads, and KDA_REUSE_PREP (which would read an earlier call's
 *    preparation back) is refused with KDA_ERR_UNSUPPORTED.
 *  - A device-side wait that gave up is recorded in the array's error word:
 *    read it with kda_static_scratch_status after the call and before the
 *    next one (each call clears the word when it starts).
 *  - Other errors as kda_chunk_fwd; KDA_ERR_CUDA if the address lookup fails.
 */
kda_status kda_chunk_fwd_static_scratch(const kda_fwd_args *args, kda_stream_t stream);

/* kda_get_device_status for the static scratch array of the current device
 * (the callers of kda_chunk_fwd_static_scratch never see its address):
 * synchronises `stream`, returns KDA_ERR_DEVICE_TIMEOUT if a bounded wait of
 * the last call gave up (and clears the word), else KDA_OK.  Copies 4 bytes
 * to a host variable; allocates nothing. */
kda_status kda_static_scratch_status(kda_stream_t stream);

/* Tokens per block of kda_chunk_fwd_host. */
#define KDA_HOST_BLOCK_TOKENS 1024

/* Bytes of device workspace kda_chunk_fwd_host needs (0 when the arguments
 * are invalid for it). */
size_t kda_chunk_fwd_host_workspace_size(const kda_fwd_args *args);

/*
 * kda_chunk_fwd with q, k, v, g, beta and out in HOST memory (the pages have
 * no counterpart of this call: they assume device-resident inputs).  The
 * forward streams the batch through the device workspace in blocks of
 * KDA_HOST_BLOCK_TOKENS tokens of every sequence: the host-to-device copies
 * of block t+1 and the device-to-host copy of o of block t-1 run on two
 * internal streams while block t computes on `stream`; the state moves from
 * block to block on the device.  Blocks end on chunk boundaries and the fp32
 * state is handed over as is, so the results are bit-identical to
 * kda_chunk_fwd's on the same inputs.
 *  - Host buffers: same layouts as kda_chunk_fwd (BSND only); page-locked
 *    memory lets the copies overlap the kernels (pageable memory works but
 *    the copies then serialise with the host).  The host buffers must stay
 *    valid until `stream` has passed the call.
 *  - Device: initial_state, final_state (device pointers or NULL), a_log,
 *    dt_bias and the workspace (kda_chunk_fwd_host_workspace_size bytes,
 *    256-byte aligned).
 *  - Stream order: nothing starts before earlier work on `stream`; when
 *    `stream` passes the call, out (host) and final_state are complete.  The
 *    internal streams are created on the first call per device and shared by
 *    all calls on it.
 *  - Errors as kda_chunk_fwd, plus KDA_ERR_UNSUPPORTED for cu_seqlens,
 *    h_out, v_new_out or KDA_REUSE_PREP.
 */
kda_status kda_chunk_fwd_host(const kda_fwd_args *args, kda_stream_t stream);

/* Bytes of workspace kda_segment_summary needs. */
size_t kda_segment_summary_workspace_size(const kda_fwd_args *args, int32_t num_segments);

/*
 * Segment affine summary ("Hyper-Parallel Chunk KDA current implementation
 * design", section 5.1, PreProcessFwd: H_out = M @ H_in + E; "KDA Context
 * Parallelism (KCP)", "Les notations").  Segment s covers the tokens
 * [seg_bounds[s], seg_bounds[s+1]) of the token axis (b*T + t for BSND, the
 * packed index for TND); each segment must lie inside one sequence (caller
 * precondition).  For each segment and head:
 *   M[s,h]       = M_b ... M_{a+1}, M_t = (I - beta_t k_t k_t^T) Diag(alpha_t),
 *                  later tokens on the left              [S, H, dk, dk] fp32
 *   S_tilde[s,h] = the state after the segment started from zero
 *                                                        [S, H, dk, dv] fp32
 * so that the state leaving a segment is M S_in + S_tilde.  Uses q, k, v, g,
 * a_log, dt_bias, beta, flags, sizes and workspace of args (q is not needed
 * by the math but is validated); ignores initial_state, cu_seqlens,
 * num_seqs, out, final_state, h_out, v_new_out.  Arithmetic as
 * kda_chunk_fwd (bf16 heads of 64 channels: M and S_tilde are the windows of
 * the 128-wide ones, whose M is blockdiag(M, I)).
 * seg_bounds: device int32 [num_segments+1], strictly increasing, within
 * [0, tokens].  Errors as kda_chunk_fwd, plus KDA_ERR_INVALID_ARG for
 * num_segments < 1 or a null M / S_tilde / seg_bounds. */
kda_status kda_segment_summary(const kda_fwd_args *args, const int32_t *seg_bounds,
                               int32_t num_segments, float *M, float *S_tilde,
                               kda_stream_t stream);

/*
 * Ordered prefix scan of segment summaries ("KDA Context Parallelism (KCP)",
 * "L'algorithme"; "Hyper-Parallel Chunk KDA current implementation design",
 * sections 5.3 and 6.3: forward summaries compose in time order).
 * For every chain c and head h, with S = S0[c,h] (zeros when S0 is NULL):
 *   for j in 0..num_segments-1:  S_in[c,j,h] = S;  S = M[c,j,h] S + S_tilde[c,j,h]
 *   S_final[c,h] = S   (when S_final is not NULL)
 * M: [C, S, H, dk, dk]; S_tilde, S_in: [C, S, H, dk, dv]; S0, S_final:
 * [C, H, dk, dv]; all fp32.  Computed in fp32 on CUDA cores (no tensor-core
 * rounding).  S_in must not alias the inputs.
 * Errors: KDA_ERR_INVALID_ARG (null M / S_tilde / S_in, sizes < 1),
 * KDA_ERR_UNSUPPORTED (dk, dv not 64/128), KDA_ERR_ALIGNMENT, KDA_ERR_CUDA. */
kda_status kda_state_prefix_scan(const float *M, const float *S_tilde, const float *S0,
                                 int32_t num_chains, int32_t num_segments, int32_t H,
                                 int32_t dk, int32_t dv, float *S_in, float *S_final,
                                 kda_stream_t stream);

/*
 * State gather, cache pool -> packed rows (vllm-ascend KDA prefill state copy
 * article, section "数值契约", numerical contract).
 * The cache holds num_rows rows, row_stride_elems elements apart; the first
 * payload_elems elements of each row are the state, the rest of the row is a
 * gap that is never read or written.  For i in [0, n_sel):
 *   packed[i, :] = cache_row[idx[i]]  if 0 <= idx[i] < num_rows and (flags is
 *                                      NULL or flags[i])
 *                = 0                  otherwise.
 * Duplicate indices are legal.  Every packed row is written.  Addresses are
 * computed in 64 bits (rows may lie more than 4 GiB apart).  n_sel == 0
 * returns KDA_OK and launches nothing.
 * cache: [num_rows, row_stride_elems] of cache_dtype; idx: [n_sel] int32 or
 * int64; flags: [n_sel] bool (one byte each) or NULL; packed: [n_sel,
 * payload_elems] of cache_dtype.
 * Errors: KDA_ERR_INVALID_ARG (null pointers with n_sel > 0, num_rows < 1,
 * payload_elems < 1, row_stride_elems < payload_elems, n_sel < 0),
 * KDA_ERR_CUDA. */
kda_status kda_state_gather(const void *cache, kda_dtype cache_dtype, int64_t num_rows,
                            int64_t row_stride_elems, int64_t payload_elems, const void *idx,
                            kda_index_dtype idx_dtype, const bool *flags, int64_t n_sel,
                            void *packed, kda_stream_t stream);

/*
 * State scatter, packed rows -> cache pool (same contract).  For i in
 * [0, n_sel) with 0 <= idx[i] < num_rows:
 *   cache_row[idx[i]] = convert(packed[i, :])    (fp32 -> bf16 rounds to
 *                                                 nearest even)
 * Out-of-range indices are skipped.  There are no flags: a flag describes
 * only an initial state and never suppresses a final write.  Valid targets
 * must be unique (caller precondition, not checked).  packed: [n_sel,
 * payload_elems] of packed_dtype.  The gap of each row is untouched.
 * n_sel == 0 returns KDA_OK and launches nothing.  Errors as gather. */
kda_status kda_state_scatter(void *cache, kda_dtype cache_dtype, int64_t num_rows,
                             int64_t row_stride_elems, int64_t payload_elems, const void *idx,
                             kda_index_dtype idx_dtype, const void *packed,
                             kda_dtype packed_dtype, int64_t n_sel, kda_stream_t stream);

/*
 * Recurrent decode step on states kept in a cache pool: the token-by-token
 * form of the recurrence ("KDA Chunk Backward - TPU/Pallas Kernel Design"
 * section 1) for the decode path named in the vllm-ascend KDA prefill state
 * copy article ("背景": decode goes through the recurrent kernel, prefill
 * through the chunked one), with the state read from and written back to the
 * pool in place.  For each sequence i in [0, N) and head h:
 *   S = cache_row[idx[i]][h]   if 0 <= idx[i] < num_rows and (init_flags is
 *                              NULL or init_flags[i]),   0 otherwise
 *   for t in [0, T):  S = Diag(alpha_t) S;  delta = v_t - S^T k^_t;
 *                     S = S + beta_t k^_t delta^T;  out_t = scale S^T q^_t
 *   cache_row[idx[i]][h] = S   if 0 <= idx[i] < num_rows (converted to the
 *                              cache dtype; bf16 rounds to nearest even)
 * alpha, k^, q^ and beta as in kda_chunk_fwd (flags KDA_L2NORM_QK,
 * KDA_BETA_SIGMOID, KDA_GATE_IN_KERNEL; the gate is a natural-log decay,
 * KDA_USE_EXP2 is accepted and changes nothing).  All arithmetic fp32.
 * Layouts: q, k [N, T, Hk, dk], v and out [N, T, H, dv] of qkv_dtype; g
 * [N, T, H, dk] and beta [N, T, H] fp32; the pool holds num_rows rows,
 * row_stride_elems apart, whose first H*dk*dv elements are the states
 * [H, dk, dv] (K-first, as final_state), the rest of a row untouched;
 * idx [N] int32/int64; init_flags [N] bool or NULL.  Valid rows must be
 * unique (caller precondition, not checked).  N == 0 launches nothing.
 * Pools whose base and row stride are 16-byte aligned move states with
 * vector accesses, others element by element (same results).
 * Errors: KDA_ERR_INVALID_ARG (null pointers with N > 0, N < 0, T < 1,
 * H < 1, Hk < 0 or not dividing H, num_rows < 1, row_stride_elems <
 * H*dk*dv, unknown flags, a_log
 * missing with KDA_GATE_IN_KERNEL), KDA_ERR_UNSUPPORTED (dk or dv not 64 /
 * 128, KDA_REUSE_PREP / KDA_SAFE_GATE / KDA_ALLOW_NEG_EIGVAL), KDA_ERR_CUDA.
 * With KDA_STATE_V_FIRST the pool states are [H, dv, dk] (element-wise
 * accesses).
 */
typedef struct {
  int32_t N, T, H, dk, dv;
  kda_dtype qkv_dtype;
  const void *q, *k, *v;
  const float *g;
  const float *a_log, *dt_bias;
  const float *beta;
  float scale, eps;
  uint32_t flags;
  void *out;
  void *cache;
  kda_dtype cache_dtype;
  int64_t num_rows, row_stride_elems;
  const void *idx;
  kda_index_dtype idx_dtype;
  const bool *init_flags;
  int32_t Hk;               /* key heads of q and k ([N, T, Hk, dk]): 0 (= H) or */
                            /* a divisor of H, value head h reads key head h/(H/Hk) */
} kda_decode_args;

kda_status kda_recurrent_step(const kda_decode_args *args, kda_stream_t stream);

/*
 * Arguments of the chunked backward ("KDA Chunk Backward - TPU/Pallas Kernel
 * Design", sections 1-2: the six stages recompute, dAv, reverse state
 * gradient, WY backward, intra-chunk backward, reverse cumsum, then gate and
 * L2-norm backward; "Hyper-Parallel Chunk KDA current implementation
 * design" section 5.2: the gradients bwd_finalize returns plus dh0).
 *
 * The gradients are those of L = <d_out, out> + <d_final_state, final_state>
 * of the forward described by `fwd`, with respect to its inputs as given:
 * q, k (raw, before the L2 norm), v, the gate input g (raw x with
 * KDA_GATE_IN_KERNEL, else the natural-log decay), beta (logits with
 * KDA_BETA_SIGMOID), a_log, dt_bias and initial_state.  With grouped key
 * heads the q/k gradients are summed over the value heads sharing a key head
 * (same design, section 4.2).  fwd.out, final_state, h_out, v_new_out and
 * fwd.workspace are ignored; every other field of fwd means what it means
 * for kda_chunk_fwd (KDA_REUSE_PREP is rejected).
 */
typedef struct {
  kda_fwd_args fwd;
  const void *d_out;           /* [.., H, dv] qkv_dtype, or NULL (= zeros)     */
  const float *d_final_state;  /* [N, H, dk, dv] fp32, or NULL (= zeros)       */
  void *dq, *dk;               /* [.., Hk, dk] qkv_dtype, written              */
  void *dv;                    /* [.., H, dv] qkv_dtype, written               */
  float *dg;                   /* [.., H, dk] fp32, written                    */
  float *dbeta;                /* [.., H] fp32, written                        */
  float *da_log;               /* [H] fp32 or NULL; zeros without              */
                               /* KDA_GATE_IN_KERNEL                           */
  float *ddt_bias;             /* [H, dk] fp32 or NULL; likewise               */
  float *d_initial_state;      /* [N, H, dk, dv] fp32 or NULL (not written)    */
  void *workspace;             /* device scratch, >= kda_chunk_bwd_workspace_size */
  size_t workspace_bytes;      /* and 256-byte aligned                         */
} kda_bwd_args;

/* Workspace bytes kda_chunk_bwd needs for these arguments; 0 when they fail
 * the argument checks.  It holds the recomputed forward intermediates, the
 * state entering and the state gradient leaving every chunk (fp32,
 * dk*dv*4 bytes per chunk and head each), and per-token fp32 scratch. */
size_t kda_chunk_bwd_workspace_size(const kda_bwd_args *args);

/* The chunked KDA backward.  bf16 inputs run on the tensor cores (bf16
 * operands, fp32 accumulation and state; chunks under strong gate decay are
 * recomputed on the CUDA cores in fp32), heads of 64 channels on zero-padded
 * 128-wide copies in the workspace (exact for the reason given at
 * kda_chunk_fwd; gradients cut back, dbeta and dA_log written directly);
 * fp32 inputs run in fp32 on the CUDA cores.
 * Deterministic: every sum runs in a fixed order.
 * Errors: those of kda_chunk_fwd for `fwd` (except that out may be NULL),
 * KDA_ERR_INVALID_ARG (null dq/dk/dv/dg/dbeta with tokens),
 * KDA_ERR_UNSUPPORTED (KDA_REUSE_PREP), KDA_ERR_ALIGNMENT,
 * KDA_ERR_WORKSPACE, KDA_ERR_CUDA. */
kda_status kda_chunk_bwd(const kda_bwd_args *args, kda_stream_t stream);

/*
 * Backward segment summary, the backward twin of kda_segment_summary
 * ("Hyper-Parallel Chunk KDA current implementation design" section 5.2,
 * npu_chunk_kda_pre_process_bwd: the local backward affine summary; "KDA
 * Chunk Backward - TPU/Pallas Kernel Design" section 2.4, dS_ext).  For
 * segment s = tokens [seg_bounds[s], seg_bounds[s+1]) and head h:
 *   E[s,h] = gradient of <d_out, o> over the segment's tokens with respect
 *            to the state entering the segment          [S, H, dk, dv] fp32
 * The segment's outputs are affine in that state, so E does not depend on
 * it; with the forward transition M of kda_segment_summary, the gradient of
 * the state entering the segment is M^T dS_out + E (the backward summary is
 * [E | M^T]; M is not recomputed here).  Uses q, k, v, g, a_log, dt_bias,
 * beta, flags, sizes, Hk and workspace of args (workspace of
 * kda_segment_bwd_summary_workspace_size); d_out [.., H, dv] qkv_dtype or
 * NULL (E = 0).  bf16: the tensor-core prep and reverse chain (heads of 64
 * channels on zero-padded copies); fp32: CUDA cores.  Errors as
 * kda_segment_summary, plus
 * KDA_ERR_UNSUPPORTED for KDA_REUSE_PREP. */
size_t kda_segment_bwd_summary_workspace_size(const kda_fwd_args *args, int32_t num_segments);
kda_status kda_segment_bwd_summary(const kda_fwd_args *args, const void *d_out,
                                   const int32_t *seg_bounds, int32_t num_segments, float *E,
                                   kda_stream_t stream);

/*
 * Reverse-order scan of the state gradient across segments (same sections:
 * the summaries are exchanged in reverse time order).  For every chain c and
 * head h, with g = dS_final[c,h] (zeros when NULL):
 *   for j = num_segments-1 .. 0:  dS_out[c,j,h] = g;  g = M[c,j,h]^T g + E[c,j,h]
 *   dS_initial[c,h] = g   (when not NULL)
 * dS_out[c,j] is the gradient of the state leaving segment j: the d_final
 * of that segment's kda_chunk_bwd.  M: [C, S, H, dk, dk]; E, dS_out:
 * [C, S, H, dk, dv]; dS_final, dS_initial: [C, H, dk, dv]; fp32, computed in
 * fp32 on CUDA cores.  dS_out must not alias the inputs.  Errors as
 * kda_state_prefix_scan. */
kda_status kda_state_grad_scan(const float *M, const float *E, const float *dS_final,
                               int32_t num_chains, int32_t num_segments, int32_t H, int32_t dk,
                               int32_t dv, float *dS_out, float *dS_initial, kda_stream_t stream);

/* Reads and clears the device error word kept at the start of a forward or
 * summary workspace: synchronises the stream, returns KDA_OK or
 * KDA_ERR_DEVICE_TIMEOUT when a bounded device-side wait gave up.  Every
 * kda_chunk_fwd / kda_segment_summary clears the word when it starts, so the
 * status describes the most recent such call on this workspace. */
kda_status kda_get_device_status(void *workspace, kda_stream_t stream);

/* A static, human-readable name for a status code. */
const char *kda_status_string(kda_status status);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
