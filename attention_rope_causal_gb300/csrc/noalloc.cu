// Pre-rotate forward for callers that cannot allocate device memory.
//
// Some callers own all of the device memory they may touch: a framework whose caching allocator
// has reserved the GPU's memory up front (so a cudaMalloc from a library would fail or fragment its
// pool), or a host that forbids runtime allocations mid-step because an allocation can fail or
// stall.  The pre-rotate mode needs scratch space for the rotated Q and K; this entry point takes
// it from a fixed buffer compiled into the library instead of from the caller or from cudaMalloc.
//
// The buffer is a file-scope __device__ array of kNoAllocScratchBytes (64 MiB).  Every GPU that
// loads this library's code holds it until the process exits (or until its context is destroyed;
// the address is looked up again in a new context).  All calls share it and it keeps the
// last call's contents (every call overwrites the part it uses before reading it, so nothing needs
// clearing); calls that overlap on the GPU (different streams, or different host threads without
// ordering) race on it and must be serialised by the caller.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attnfuse.h"
#include "attnfuse_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = ATTNFUSE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Driver calls that name the current context and its unique id, fetched through the runtime (the
// library links no driver library).
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns& ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return fns;
}

// Unique id of the context current on this thread (0 if none is current yet or it cannot be named).
unsigned long long current_context_id() {
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return 0;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct Slot {
  unsigned long long ctx_id;  // context the address belongs to
  void* ptr;
};
Slot g_scratch[kMaxDevices] = {};

// The device address of the scratch array in the current device's context.  It is looked up with
// cudaGetSymbolAddress the first time a context asks, and again whenever the context changes (a
// cudaDeviceReset and a new primary context load the module again, possibly elsewhere).
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  const unsigned long long id = current_context_id();
  if (id != 0 && g_scratch[dev].ptr != nullptr && g_scratch[dev].ctx_id == id) {
    *out = g_scratch[dev].ptr;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the device's primary context current
  if (e != cudaSuccess) return e;
  g_scratch[dev] = Slot{current_context_id(), p};
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" attnfuse_status_t attnfuse_rope_causal_fwd_prerotate_noalloc(const void* q, const void* k, const void* v,
                                                                         void* out, float* lse, int B, int Hq,
                                                                         int Hkv, int N, int d, double rope_base,
                                                                         attnfuse_dtype_t dtype, void* stream) {
  // Every argument and the device are checked before anything touches the GPU, as in the other
  // entry points.
  attnfuse_status_t st =
      attnfuse::check_fwd_call(q, k, v, out, lse, B, Hq, Hkv, N, d, rope_base, ATTNFUSE_PREROTATE, dtype);
  if (st != ATTNFUSE_OK) return st;
  const size_t need = attnfuse_workspace_bytes(B, Hq, Hkv, N, d, ATTNFUSE_PREROTATE, dtype);
  if (need > kNoAllocScratchBytes) {
    attnfuse::set_last_error("rotated Q and K need %zu bytes; the no-allocation entry point has a fixed %zu-byte "
                             "buffer (use attnfuse_rope_causal_fwd with a workspace)",
                             need, kNoAllocScratchBytes);
    return ATTNFUSE_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();  // leave no sticky-looking error behind for the caller's own checks
    attnfuse::set_last_error("cudaGetSymbolAddress for the fixed scratch buffer: %s", cudaGetErrorString(e));
    return ATTNFUSE_ERR_CUDA;
  }
  // Same kernels as attnfuse_rope_causal_fwd in pre-rotate mode; the fixed buffer is its workspace,
  // so nothing is allocated.
  return attnfuse_rope_causal_fwd(q, k, v, out, lse, B, Hq, Hkv, N, d, rope_base, ATTNFUSE_PREROTATE, dtype, scratch,
                                  kNoAllocScratchBytes, stream);
}
