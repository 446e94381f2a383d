// Internal declarations shared by the libusp translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

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

// Raises a kernel's dynamic shared-memory limit once per device (bit d of
// `done` for device d < 64; devices beyond that set it on every launch).
// Concurrent first calls may both set it, which is harmless.
inline cudaError_t smem_limit_once(std::atomic<unsigned long long>& done, const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Launches `kernel` on `stream` with programmatic stream serialisation: its
// CTAs may start (prologue: barriers, TMEM, tensor-map prefetch) while the
// previous kernel of the stream drains its last wave.  Every kernel launched
// this way calls ptx::griddep_wait() before its first access to global
// memory, so it neither reads what that kernel writes nor overwrites what it
// reads before that kernel has completed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Per-launch guard: where to record an expired wait, and the wait limits.
struct Guard {
  unsigned int* err;        // per-device error word (device memory)
  long long spin_limit;     // polls before a wait gives up
  unsigned long long ns_limit;  // wall-clock bound per wait (globaltimer ns)
};

// Problem description for the attention kernels.  A "unit" is one
// (query head, KV head, output head) triple; the ring schedule maps
// unit -> heads for the materialised USP launch.
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

// The same re-layout of up to six tensors in one launch whose rows are
// row_bytes[i] bytes (D * element size); run alignment picks the vector width
// for the whole launch.
cudaError_t launch_relayout_rows(const void* const* srcs, void* const* dsts, const int64_t* row_bytes, int count,
                                 int64_t B, int64_t H, int64_t Ns, int ulysses, int ring, bool tok2head,
                                 cudaStream_t stream);
// The same re-layout of up to six same-shape tensors in one launch.
cudaError_t launch_relayout_n(const void* const* srcs, void* const* dsts, int count, int64_t B, int64_t H,
                              int64_t Ns, int64_t D, int ulysses, int ring, int elt, bool tok2head,
                              cudaStream_t stream);

// The merge of R head-sharded partial planes [r, u, B, Hu, Nr, D] written
// straight into the token-sharded stacks out [r, u, B, H, Ns, D] and lse
// [r, u, B, H, Ns]; 16-byte vectors when lse_merge_to_tokens_ok (D % 8,
// aligned pointers, R <= 8, 32-bit row indices), else one element per thread.
bool lse_merge_to_tokens_ok(const void* outs, const void* out, int R, int64_t B, int64_t Hu, int64_t Nr, int64_t D,
                            int u, int r);
cudaError_t launch_lse_merge_to_tokens(const void* outs, const float* lses, int R, void* out, float* lse, int64_t B,
                                       int64_t Hu, int64_t Nr, int64_t D, int u, int r, int dtype,
                                       cudaStream_t stream);
cudaError_t launch_lse_merge(const void* outs, const float* lses, int R, void* out, float* lse,
                             int64_t rows, int64_t D, int dtype, cudaStream_t stream);

// Unit -> heads mappings of the attention kernels.  Head-sharded stack head
// ((g*u + j)*B + b)*Hu + h' holds rank (g, j)'s slice of plain head
// b*H + j*Hu + h'.
enum UnitMode : int {
  kUnitPlain = 0,   // q head = kv head = unit, out head = out_base + unit
  kUnitRing = 1,    // materialised ring step t: KV chunk (g - t) mod ring, out plane t
  kUnitImgTxt = 2,  // unit = stack head: image queries against the text head of their group
  kUnitTxtImg = 3,  // unit = (c, j, b, h'): text queries of head group j against ring chunk c
};
struct UnitMap {
  int mode;
  RingSchedule sched;
  int64_t out_step_stride;  // heads between ring steps (output planes)
  int64_t out_base;         // head offset of the launch's first output head
  int64_t B, H, Hu;
};
struct UnitHeads {
  int64_t qh, kvh, kvh2, oh;  // kvh2: head of the second KV source
};
// Units, heads and ring indices all fit 32 bits (launch grids bound the
// unit count), so the index arithmetic divides in 32 bits; only the output
// head offset is formed in 64 bits.
__device__ __forceinline__ UnitHeads map_unit(const UnitMap& m, int64_t unit64) {
  UnitHeads r;
  const int unit = (int)unit64;
  r.kvh2 = unit;
  if (m.mode == kUnitPlain) {
    r.qh = r.kvh = unit;
    r.oh = m.out_base + unit;
    return r;
  }
  const RingSchedule& s = m.sched;
  if (m.mode == kUnitRing) {
    const int per_step = s.ring * s.ulysses * s.heads_per_rank;
    const int t = unit / per_step;
    const int qh = unit - t * per_step;
    const int group = s.heads_per_rank * s.ulysses;  // heads of one ring rank
    const int g = qh / group;
    const int c = ((g - t) % s.ring + s.ring) % s.ring;  // KV chunk at ring step t
    r.qh = qh;
    r.kvh = qh + (c - g) * group;
    r.oh = m.out_base + (int64_t)t * m.out_step_stride + qh;
    return r;
  }
  const int Hu = (int)m.Hu, B = (int)m.B;
  const int hp = unit % Hu, b = (unit / Hu) % B, j = (unit / (Hu * B)) % s.ulysses;
  const int th = b * (int)m.H + j * Hu + hp;  // plain (text) head of the same (j, b, h')
  if (m.mode == kUnitImgTxt) {
    r.qh = unit;
    r.kvh = th;
    r.oh = m.out_base + unit;
    return r;
  }
  const int c = unit / (Hu * B * s.ulysses);
  r.qh = th;
  r.kvh = ((c * s.ulysses + j) * B + b) * Hu + hp;
  r.oh = m.out_base + (int64_t)c * m.out_step_stride + th;
  return r;
}

// Operands of one attention launch.  A "stack" operand is the token-sharded
// stack [sp][BH][Ns][D] read as sp*Ns rows per head; a plain operand is
// [heads][rows][D].  The optional second KV source (plain) follows the first
// source's keys in the softmax, e.g. the text tokens of joint attention.
struct AttnArgs {
  const void* q; const void* k; const void* v;
  const void* k2; const void* v2;
  void* out; float* lse;
  bool q_stack, kv_stack, out_stack;
  int64_t Nq, Nk, Nk2;                 // rows per head of the plain operands
  int64_t q_heads, kv_heads, kv2_heads;  // heads of the plain operands
  int64_t BH, sp, Ns;                  // stack geometry
  UnitMap map;
  int64_t units;
  float scale;
};

// fp32 attention on the FP32 pipes (any D <= 128).
cudaError_t launch_attn_f32(const AttnArgs& a, int D, cudaStream_t stream);

// bf16 tcgen05 attention forward (D = 128): one launch serving one or two
// problems (same stack geometry and scale).
cudaError_t launch_attn_tc_fwd(const AttnArgs* sides, int nsides, const Guard& g, cudaStream_t stream);

// FP8 (E4M3) path: per-head quantisation of bf16 token stacks, then the fused
// FP8 attention forward.
int64_t fp8_vt_pitch(int64_t Ns);  // row pitch (bytes) of the transposed V codes: Ns rounded up to 16
cudaError_t launch_quantize_e4m3(const void* x, uint8_t* x8, float* scales, unsigned* amax, int64_t BH, int64_t sp,
                                 int64_t Ns, int64_t D, cudaStream_t stream);
cudaError_t launch_quantize_qkv_fp8(const void* q, const void* k, const void* v, uint8_t* q8, uint8_t* k8,
                                    uint8_t* vt8, unsigned* amax, int64_t BH, int64_t sp, int64_t Ns,
                                    cudaStream_t stream);
struct Fp8AttnArgs {
  const uint8_t *q8, *k8, *vt8;  // [sp][BH][Ns][128], [sp][BH][Ns][128], [sp][BH][128][Ns_pad]
  const unsigned* amax;          // [3][BH] float bits
  void* out;                     // bf16 [sp][BH][Ns][128]
  float* lse;                    // [sp][BH][Ns]
  int64_t BH, sp, Ns, Ns_pad;
  float scale;
};
cudaError_t launch_attn_fp8_fwd(const Fp8AttnArgs& a, const Guard& g, cudaStream_t stream);

// bf16 tcgen05 backward over token-sharded stacks (D = 128): prep (Delta,
// lse*log2e into workspace), dK/dV kernel, dQ kernel.
// All tensors are stacks [sp][BH][Ns][D] (lse, delta, l2 without D): the
// token-sharded stack (useg = 1: unit = head, over all sp segments) or the
// head-sharded stack of the materialised path viewed as [r*u][B*Hu][Nr][D]
// (useg = u: unit = (j, b, h'), over the segments g*u + j).
struct TcBwdArgs {
  const void *q, *k, *v, *out, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  float* delta;  // workspace [sp][BH][Ns_pad]
  float* l2;     // workspace [sp][BH][Ns_pad]
  int64_t BH, sp, Ns;
  int useg;
  float scale;
};
cudaError_t launch_attn_tc_bwd(const TcBwdArgs& a, const Guard& g, cudaStream_t stream);

// fp32 backward on the FP32 pipes over stacks (segment stride useg as in TcBwdArgs).
cudaError_t launch_attn_f32_bwd(const float* q, const float* k, const float* v, const float* out,
                                const float* lse, const float* dout, float* dq, float* dk, float* dv,
                                float* delta, int64_t BH, int64_t sp, int64_t Ns, int useg, int D, float scale,
                                cudaStream_t stream);

// Records the next phase event of the current call on stream `s` (no-op
// unless phase timing is enabled with usp_profile_phases).  The phase runs
// from event `from` (an earlier mark's return value; -1 = the previous mark)
// to this one.  Returns this mark's index, or -1.
int phase_mark(cudaStream_t s, int from = -1);
// Remembers `e` as this thread's last CUDA error (usp_last_cuda_error) and
// returns USP_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// Fork / join of the device's side stream: side_begin makes the side stream
// wait for the work enqueued so far on `main` and hands it out (holding the
// device's side-stream lock); side_end makes `main` wait for everything
// enqueued on the side stream and releases the lock.  Every successful
// side_begin must be followed by side_end on the same thread and device.
cudaError_t side_begin(cudaStream_t main, cudaStream_t* side);
cudaError_t side_end(cudaStream_t main);

}  // namespace usp
