// tq_score_noalloc: tq_score for callers that cannot allocate device memory.
//
// Some callers of this library are not free to call cudaMalloc.  A plugin
// hosted inside a larger runtime (an inference server, a framework that owns
// every byte of device memory through its own pool allocator) is usually
// forbidden to allocate behind its host's back: doing so can exceed the
// budget the host reserved and fragments memory it manages.  Latency-critical
// callers avoid cudaMalloc too, because it can synchronise the device.  Such
// callers still need the scratch that scoring uses (the rotated and projected
// queries, and the top-k candidates).  This entry point takes that scratch
// from one fixed array in device memory that is part of the library image, so
// the call itself allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library is loaded holds TQ_SCORE_NOALLOC_MAX_BYTES of it until the process
// exits.  Host code cannot use the array's name as a device address (on the
// host it names a stand-in object), so the first call on each device looks up
// the real address with cudaGetSymbolAddress while that device is current and
// keeps it.  That first call should therefore come before any stream capture.
// The address belongs to the CUDA context the library's module was loaded
// into: the kept address is tagged with that context's process-unique id
// (cuCtxGetId), and a call made under another context -- for example after
// cudaDeviceReset, which destroys the device's primary context and with it
// the array -- looks the address up again instead of reusing a stale one.
//
// All calls share the one array.  Calls whose work overlaps on the GPU (two
// streams, or two threads) race on it and must be serialised by the caller.
// The array keeps whatever the last call left in it; nothing in it needs to
// start at zero, because every byte the kernels read in a call was written
// earlier in the same call.
#include <cuda.h>

#include <mutex>

#include "tq_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_score_scratch[TQ_SCORE_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  unsigned long long ctx_id;  // cuCtxGetId of the context the address belongs to
  void* ptr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// The two driver calls used here, through the runtime's entry-point lookup
// (the library does not link the driver library directly, so that it loads on
// machines without one).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
template <typename Fn>
Fn driver_entry(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  return nullptr;
}

// Process-unique id of the current context (0 if there is none).
cudaError_t current_context_id(unsigned long long* id) {
  static const CtxGetCurrentFn get_current = driver_entry<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_entry<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  *id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (ctx == nullptr) return cudaSuccess;
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of g_score_scratch in the current device's current context
// (looked up once per context).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long id = 0;
  e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  if (id == 0) {
    // no context yet: the runtime's lookup makes the primary one current
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_score_scratch);
    if (e != cudaSuccess) return e;
    e = current_context_id(&id);
    if (e != cudaSuccess) return e;
    if (id == 0) return cudaErrorDeviceUninitialized;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& a = g_scratch_addr[dev];
  if (a.ptr == nullptr || a.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_score_scratch);
    if (e != cudaSuccess) return e;
    a.ctx_id = id;
    a.ptr = p;
  }
  *out = a.ptr;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" tq_status tq_score_noalloc(const tq_plan* p, const float* queries, int64_t G, int H, const void* packed,
                                      int64_t N, float* logits, int top_k, float* top_scores, int64_t* top_idx,
                                      void* stream) {
  if (!p || G < 0 || N < 0 || H < 1 || H > 256 || top_k < 0 || top_k > 64) return TQ_EINVAL;
  if (top_k > 0 && (top_k > N || !top_scores || !top_idx)) return TQ_EINVAL;
  if (G == 0 || N == 0) return TQ_OK;
  if (!queries || !packed || !logits) return TQ_EINVAL;
  if (!aligned16(queries) || !aligned16(packed) || !aligned16(logits)) return TQ_EALIGN;
  if (top_k > 0 && (!aligned16(top_scores) || !aligned16(top_idx))) return TQ_EALIGN;
  const size_t need = tq_score_workspace_bytes(p, G, H, N, top_k);
  if (need == 0 || need > (size_t)TQ_SCORE_NOALLOC_MAX_BYTES) return TQ_EUNSUPPORTED;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return TQ_ECUDA;
  // the same kernels and scratch layout as tq_score
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = tq::score_run(p, queries, G, H, static_cast<const uint8_t*>(packed), N, logits, top_k, top_scores,
                                top_idx, ws, s);
  return e == cudaSuccess ? TQ_OK : TQ_ECUDA;
}
