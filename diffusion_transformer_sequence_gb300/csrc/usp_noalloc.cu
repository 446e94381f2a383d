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
// intermediate buffers (head-sharded q/k/v, and the per-ring-step partial
// outputs and LSEs -- or, with one ring step, the head-sharded chunk result)
// come from here.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes: every
// GPU that loads the library holds it until the process exits.  Host code may
// not use the array's name as a device address (on the host it names a
// stand-in object), so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the first
// call made on that device.  That first call should therefore come before any
// stream capture.  The address is cached with the id of the current context;
// after a cudaDeviceReset the next call sees a new context id and looks the
// address up again.  All calls share the one array and it keeps the previous
// call's contents; nothing in this path needs it zeroed (every byte is written
// before it is read).  Calls whose executions overlap on the GPU -- on
// different streams, or from different host threads -- race on the array and
// must be serialised by the caller.
#include <cuda.h>

#include <mutex>

#include "usp.h"
#include "usp_internal.cuh"

namespace usp {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
struct ScratchSlot {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;  // context the address belongs to (0: unknown)
};
ScratchSlot g_noalloc[kMaxDev];

// Id of the current context (driver cuCtxGetCurrent + cuCtxGetId, looked up
// through the runtime's entry-point query), or 0 when it cannot be read.
unsigned long long current_ctx_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<GetCurrent>(a);
      get_id = reinterpret_cast<GetId>(b);
    }
    (void)cudaGetLastError();  // a failed query leaves nothing behind for later calls
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array for the current device.  Looked up once
// per device and context (with the device current); a failed lookup clears
// the runtime's error state, so later launches do not report it again.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return record_cuda_error(e);
  }
  if (dev < 0 || dev >= kMaxDev) return USP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  ScratchSlot& slot = g_noalloc[dev];
  if (slot.ptr != nullptr) {
    const unsigned long long id = current_ctx_id();
    if (id != 0 && slot.ctx_id != 0 && id != slot.ctx_id) slot.ptr = nullptr;  // the context was reset
  }
  if (slot.ptr == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    }
    slot.ptr = p;
    slot.ctx_id = current_ctx_id();
  }
  *out = slot.ptr;
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
  if (need > usp::kNoAllocScratchBytes) {
    // Too large for the fixed scratch.  The workspace call runs the same
    // argument checks in the same order and, given no workspace, stops with
    // USP_ERR_WORKSPACE at its workspace check (before enqueueing anything),
    // so a problem with a bad argument gets the code the workspace call gives.
    return usp_attention_fwd(q, k, v, out, lse, B, H, N, D, ulysses, ring, scale, dtype, USP_MATERIALISED,
                             nullptr, 0, stream);
  }
  void* scratch = nullptr;
  if (need > 0) {
    const int st = usp::scratch_address(&scratch);
    if (st != USP_OK) return st;
  }
  return usp_attention_fwd(q, k, v, out, lse, B, H, N, D, ulysses, ring, scale, dtype, USP_MATERIALISED,
                           scratch, usp::kNoAllocScratchBytes, stream);
}

}  // extern "C"
