// usp_attention_fwd_noalloc: the materialised USP forward with its scratch
// memory taken from a fixed array compiled into the library, for callers that
// cannot allocate device memory themselves.
//
// Who needs this: code that runs under a host framework whose caching
// allocator owns the device memory (a raw cudaMalloc behind its back can fail
// once the pool has reserved the card, and breaks the framework's memory
// budget), and latency-critical callers that must not call cudaMalloc or
// cudaFree in their request path because those calls may synchronise the
// device.  Such callers still pass their inputs and outputs; only the
// intermediate buffers (head-sharded q/k/v, per-ring-step partial outputs and
// LSEs, merged head-sharded results) come from here.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes: every
// GPU that loads the library holds it until the process exits.  Host code may
// not use the array's name as a device address (on the host it names a
// stand-in object), so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the first
// call made on that device.  That first call should therefore come before any
// stream capture.  All calls share the one array and it keeps the previous
// call's contents; nothing in this path needs it zeroed (every byte is written
// before it is read).  Calls whose executions overlap on the GPU -- on
// different streams, or from different host threads -- race on the array and
// must be serialised by the caller.
#include <mutex>

#include "usp.h"
#include "usp_internal.cuh"

namespace usp {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDev] = {};

// Device address of the scratch array for the current device (looked up once).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return USP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDev) return USP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return USP_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return USP_OK;
}

}  // namespace
}  // namespace usp

extern "C" {

int usp_attention_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse, int64_t B,
                              int64_t H, int64_t N, int64_t D, int ulysses, int ring, float scale,
                              usp_dtype dtype, usp_stream_t stream) {
  const size_t need =
      usp_attention_workspace_bytes(B, H, N, D, ulysses, ring, dtype, USP_MATERIALISED, 0);
  if (need > usp::kNoAllocScratchBytes) return USP_ERR_WORKSPACE;  // problem too large for the fixed scratch
  void* scratch = nullptr;
  if (need > 0) {
    const int st = usp::scratch_address(&scratch);
    if (st != USP_OK) return st;
  }
  return usp_attention_fwd(q, k, v, out, lse, B, H, N, D, ulysses, ring, scale, dtype, USP_MATERIALISED,
                           scratch, usp::kNoAllocScratchBytes, stream);
}

}  // extern "C"
