// kda_static_scratch.cu - a forward entry point that allocates nothing.
//
// Some callers cannot allocate device memory for a workspace: a plugin whose
// host framework owns all device memory and exposes no allocator, or a
// latency-critical path where cudaMalloc (which may synchronise the device)
// is not allowed.  kda_chunk_fwd_static_scratch serves them: it runs the same
// forward as kda_chunk_fwd, with the scratch taken from a fixed array in the
// library's own device memory instead of a caller-provided workspace.
//
// The array lives for as long as the library is loaded, on every GPU the
// library is used on.  All calls share it, so calls that run at the same
// time on the GPU (for example on two streams) race; callers serialise them.
// The forward rewrites every scratch byte it later reads (the device error
// word and the strong-decay list count are cleared at the start of each
// call), so leftovers of an earlier call do not matter.  That is why
// KDA_REUSE_PREP, which reads an earlier call's chunk preparation back from
// the scratch, is refused here.  The device error word (a bounded wait that
// gave up) sits at the start of the array; kda_static_scratch_status reads
// and clears it, and the next forward clears it too.
#include <mutex>

#include "kda_internal.cuh"

// 32 MiB, 256-byte aligned: the upper bound on kda_chunk_fwd_workspace_size
// for problems this entry point accepts.
static __device__ __align__(256) unsigned char g_kda_static_scratch[KDA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (host code cannot take the address of a __device__ array directly).
kda_status scratch_for_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_static_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_static_scratch(const kda_fwd_args *args, kda_stream_t stream) {
  if (!args) return KDA_ERR_INVALID_ARG;
  const size_t need = kda_chunk_fwd_workspace_size(args);
  if (need == 0) return kda_chunk_fwd(args, stream);  // invalid arguments: same error as kda_chunk_fwd
  // the shared array holds whatever the last call left: nothing may be reused
  if (args->flags & KDA_REUSE_PREP) return KDA_ERR_UNSUPPORTED;
  if (need > (size_t)KDA_STATIC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
  void *ws = nullptr;
  const kda_status s = scratch_for_current_device(&ws);
  if (s != KDA_OK) return s;
  kda_fwd_args a = *args;
  a.workspace = ws;
  a.workspace_bytes = (size_t)KDA_STATIC_SCRATCH_BYTES;
  return kda_chunk_fwd(&a, stream);
}

extern "C" kda_status kda_static_scratch_status(kda_stream_t stream) {
  void *ws = nullptr;
  const kda_status s = scratch_for_current_device(&ws);
  if (s != KDA_OK) return s;
  return kda_get_device_status(ws, stream);
}
