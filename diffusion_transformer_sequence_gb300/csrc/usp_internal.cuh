// Internal declarations shared by the libusp translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace usp {

// Error codes written into the per-device error word by kernels whose waits
// expired (the first code written wins; usp_device_status clears it).
enum DevError : unsigned int {
  kDevOk = 0,
  kDevTimeoutTmaProducer = 1,
  kDevTimeoutMma = 2,
  kDevTimeoutSoftmax = 3,
  kDevTimeoutEpilogue = 4,
};

// Per-launch guard: where to record an expired wait, and the wait limits.
struct Guard {
  unsigned int* err;        // per-device error word (device memory)
  long long spin_limit;     // polls before a wait gives up
  unsigned long long ns_limit;  // wall-clock bound per wait (globaltimer ns)
};

// Problem description for the attention kernels.  A "unit" is one
// (query head, KV head, output head) triple; the ring schedule maps
// unit -> heads for the materialised USP launch, the plain chunk call uses
// the identity.
struct RingSchedule {
  int ulysses;   // u  (1 for a plain chunk call)
  int ring;      // r  (1 for a plain chunk call)
  int steps;     // ring steps in this launch: units = steps * ring * ulysses * heads_per_rank
  int heads_per_rank;  // B * Hu (B * H for a plain chunk call)
};

// Launchers (return cudaError_t of the launch).
cudaError_t launch_relayout(const void* src, void* dst, int64_t runs_outer, int64_t B, int64_t H,
                            int64_t Ns, int64_t D, int ulysses, int ring, int elt, bool tok2head,
                            cudaStream_t stream);

// The same re-layout of up to three same-shape tensors in one launch.
cudaError_t launch_relayout_n(const void* const* srcs, void* const* dsts, int count, int64_t B, int64_t H,
                              int64_t Ns, int64_t D, int ulysses, int ring, int elt, bool tok2head,
                              cudaStream_t stream);

cudaError_t launch_lse_merge(const void* outs, const float* lses, int R, void* out, float* lse,
                             int64_t rows, int64_t D, int dtype, cudaStream_t stream);

// fp32 attention on the FP32 pipes.  q: [units_q][Nq][D]; k,v: [units_kv][Nk][D].
cudaError_t launch_attn_f32(const float* q, const float* k, const float* v, float* out, float* lse,
                            int64_t Nq, int64_t Nk, int D, float scale, RingSchedule sched,
                            int64_t out_step_stride_heads, cudaStream_t stream);

// fp32 fused USP forward over token-sharded stacks.
cudaError_t launch_attn_f32_fused(const float* q, const float* k, const float* v, float* out,
                                  float* lse, int64_t BH, int64_t sp, int64_t Ns, int D, float scale,
                                  cudaStream_t stream);

// bf16 tcgen05 attention forward (D = 128).
struct TcAttnArgs {
  const void* q; const void* k; const void* v;
  void* out; float* lse;
  // plain / materialised addressing: heads are contiguous [rows][D] blocks
  int64_t Nq, Nk;
  RingSchedule sched;
  int64_t out_step_stride_heads;   // heads between consecutive ring steps in out/lse
  // fused addressing: token-sharded stack [sp][BH][Ns][D]
  bool fused;
  int64_t BH, sp, Ns;
  float scale;
};
cudaError_t launch_attn_tc_fwd(const TcAttnArgs& a, const Guard& g, cudaStream_t stream);

// bf16 tcgen05 backward over token-sharded stacks (D = 128): prep (Delta,
// lse*log2e into workspace), dK/dV kernel, dQ kernel.
struct TcBwdArgs {
  const void *q, *k, *v, *out, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  float* delta;  // workspace [sp][BH][Ns]
  float* l2;     // workspace [sp][BH][Ns]
  int64_t BH, sp, Ns;
  float scale;
};
cudaError_t launch_attn_tc_bwd(const TcBwdArgs& a, const Guard& g, cudaStream_t stream);

// fp32 backward on the FP32 pipes over token-sharded stacks.
cudaError_t launch_attn_f32_bwd(const float* q, const float* k, const float* v, const float* out,
                                const float* lse, const float* dout, float* dq, float* dk, float* dv,
                                float* delta, int64_t BH, int64_t sp, int64_t Ns, int D, float scale,
                                cudaStream_t stream);

// Records the next phase event of the current call (no-op unless phase timing
// is enabled with usp_profile_phases).
void phase_mark(cudaStream_t s);

}  // namespace usp
