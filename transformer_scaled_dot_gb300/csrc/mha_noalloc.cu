// mha_noalloc.cu -- mha_forward for callers that cannot allocate device memory.
//
// mha_forward needs a caller-provided workspace for the intermediate Q, K, V
// and merged heads. Some callers cannot obtain one: a plugin whose host
// application owns the whole device-memory budget and forbids allocation
// inside the plugin, a serving loop whose memory is planned up front and
// must not call cudaMalloc/cudaFree on the request path (both synchronise
// the device and stall the other streams), or a plain C caller with no access
// to the framework's caching allocator. For them this file keeps the
// workspace in a fixed file-scope device array and runs the unchanged
// mha_forward on it.
//
// The array is part of the library's device image: every GPU that loads the
// library holds these bytes until the process exits. All calls on a device
// share it and it keeps the last call's contents; calls that overlap on the
// GPU (different streams, or different host threads, without ordering
// between them) race on it. Nothing needs clearing between calls: every
// byte that a call reads from the scratch is written earlier in that same
// call (the projections write all of Q, K, V; attention writes every merged
// head row).
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "tsd_attention.h"

namespace {

static __device__ __align__(256) unsigned char g_mha_scratch[TSD_MHA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
struct ScratchEntry {
  unsigned long long ctx_id = 0;  // the context the address belongs to (0: none yet)
  void* ptr = nullptr;
};
ScratchEntry g_scratch[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Driver calls reached through the runtime (the library does not link libcuda).
template <typename F>
F driver_fn(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

// Unique id of the calling thread's current context (ids are never reused
// within a process, unlike context handles), or 0 if it has none.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_mha_scratch in the current context. The host-side
// symbol is only a stand-in, so the address is looked up with the device
// current and cached per device, keyed by the context's id: after a
// cudaDeviceReset, or with another context current, the lookup runs again.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long id = current_context_id();
  if (id == 0 || g_scratch[dev].ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_mha_scratch);  // binds the primary context if none is current
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    if (id == 0) id = current_context_id();
    g_scratch[dev].ctx_id = id;  // 0 if the id is unavailable: looked up on every call
    g_scratch[dev].ptr = p;
    *out = p;
    return cudaSuccess;
  }
  *out = g_scratch[dev].ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" attn_status mha_forward_noalloc(const void* x_q, const void* x_kv, const void* w_q,
                                           const void* w_k, const void* w_v, const void* w_o,
                                           void* out, int B, int n_q, int n_k, int d_model, int h,
                                           int d_k, int d_v, int mask_kind,
                                           const int32_t* kv_lens, float scale,
                                           tsd_stream_t stream) {
  // Sizes first: a request beyond the fixed scratch is refused before any
  // CUDA call. Invalid sizes (0 bytes) fall through to mha_forward's checks.
  const size_t need = mha_workspace_bytes(B, n_q, n_k, h, d_k, d_v);
  if (need > static_cast<size_t>(TSD_MHA_NOALLOC_SCRATCH_BYTES)) return ATTN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return mha_forward(x_q, x_kv, w_q, w_k, w_v, w_o, out, B, n_q, n_k, d_model, h, d_k, d_v,
                     mask_kind, kv_lens, scale, scratch,
                     static_cast<size_t>(TSD_MHA_NOALLOC_SCRATCH_BYTES), stream);
}
