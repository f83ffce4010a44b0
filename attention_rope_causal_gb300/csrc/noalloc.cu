// Pre-rotate forward for callers that cannot allocate device memory.
//
// Some callers own all of the device memory they may touch: a framework whose caching allocator
// has reserved the GPU's memory up front (so a cudaMalloc from a library would fail or fragment its
// pool), or a host that forbids runtime allocations mid-step because an allocation can fail or
// stall.  The pre-rotate mode needs scratch space for the rotated Q and K; this entry point takes
// it from a fixed buffer compiled into the library instead of from the caller or from cudaMalloc.
//
// The buffer is a file-scope __device__ array of kNoAllocScratchBytes (64 MiB).  Every GPU that
// loads this library's code holds it until the process exits.  All calls share it and it keeps the
// last call's contents (every call overwrites the part it uses before reading it, so nothing needs
// clearing); calls that overlap on the GPU (different streams, or different host threads without
// ordering) race on it and must be serialised by the caller.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "attnfuse.h"
#include "attnfuse_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = ATTNFUSE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// The device address of the scratch array on the current device, looked up once per device.
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" attnfuse_status_t attnfuse_rope_causal_fwd_prerotate_noalloc(const void* q, const void* k, const void* v,
                                                                         void* out, float* lse, int B, int Hq,
                                                                         int Hkv, int N, int d, double rope_base,
                                                                         attnfuse_dtype_t dtype, void* stream) {
  const size_t need = attnfuse_workspace_bytes(B, Hq, Hkv, N, d, ATTNFUSE_PREROTATE, dtype);
  if (need == 0) {
    attnfuse::set_last_error("invalid sizes or dtype: B, Hq, Hkv, N >= 1, d in {64, 128}, dtype bf16 or fp16");
    return ATTNFUSE_ERR_INVALID_ARG;
  }
  if (need > kNoAllocScratchBytes) {
    attnfuse::set_last_error("rotated Q and K need %zu bytes; the no-allocation entry point has a fixed %zu-byte "
                             "buffer (use attnfuse_rope_causal_fwd with a workspace)",
                             need, kNoAllocScratchBytes);
    return ATTNFUSE_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    attnfuse::set_last_error("cudaGetSymbolAddress for the fixed scratch buffer: %s", cudaGetErrorString(e));
    return ATTNFUSE_ERR_CUDA;
  }
  // Same kernels as attnfuse_rope_causal_fwd in pre-rotate mode; the fixed buffer is its workspace,
  // so nothing is allocated.  The remaining argument checks happen there, before any launch.
  return attnfuse_rope_causal_fwd(q, k, v, out, lse, B, Hq, Hkv, N, d, rope_base, ATTNFUSE_PREROTATE, dtype, scratch,
                                  kNoAllocScratchBytes, stream);
}
