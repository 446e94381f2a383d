// libusp C ABI: argument validation, workspace layout and the USP drivers.
//
// The driver composes the steps of USP attention in the order the USP PR
// page's Design gives them (the exchange within each Ulysses group, the ring
// steps on a kernel that also yields the log-sum-exp, the exchange back),
// with the virtual rank grid
// ulysses x ring laid out on one device:
//   * the all-to-all becomes the on-device re-layout (relayout.cu);
//   * the ring's peer-to-peer KV rotation becomes addressing: at ring step t
//     rank g reads KV chunk (g - t) mod ring in place, nothing is copied;
//   * the per-step results are merged by log-sum-exp (lse_merge.cu).
// Validation mirrors the PR page's Limitations table: every unsupported
// configuration fails loudly, before anything is enqueued.
#include <atomic>
#include <cmath>
#include <mutex>

#include "usp.h"
#include "usp_internal.cuh"

namespace usp {

__device__ unsigned int g_dev_error = 0;

namespace {

thread_local int t_last_cuda_error = 0;

// Phase timing (usp_profile_phases / usp_profile_read): events recorded at the
// kernel boundaries of the most recent attention call on this thread.
constexpr int kMaxPhases = 8;
struct PhaseState {
  bool enabled = false;
  bool created = false;
  int marks = 0;
  cudaEvent_t ev[kMaxPhases + 1];
  int from[kMaxPhases + 1];  // phase i runs from event from[i] to event i
};
thread_local PhaseState t_phase;

}  // namespace
int record_cuda_error(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return USP_ERR_CUDA;
}
int phase_mark(cudaStream_t s, int from) {
  if (!t_phase.enabled || t_phase.marks == 0 || t_phase.marks > kMaxPhases) return -1;
  const int i = t_phase.marks;
  if (cudaEventRecord(t_phase.ev[i], s) != cudaSuccess) return -1;
  t_phase.from[i] = (from >= 0 && from < i) ? from : i - 1;
  ++t_phase.marks;
  return i;
}
namespace {
void phase_begin(cudaStream_t s) {
  if (!t_phase.enabled) return;
  t_phase.marks = 0;
  if (cudaEventRecord(t_phase.ev[0], s) == cudaSuccess) t_phase.marks = 1;
}
std::atomic<long long> g_spin_limit{-1};
constexpr long long kDefaultSpinLimit = 1LL << 40;       // polls; the time bound below governs
constexpr unsigned long long kWaitNs = 2000000000ull;    // 2 s per wait

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices] = {};

int cuda_fail(cudaError_t e) { return record_cuda_error(e); }

int err_word(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return USP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dev_error);
    if (e != cudaSuccess) return cuda_fail(e);
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_err_ptr[dev];
  return USP_OK;
}

int guard(Guard* g) {
  unsigned int* p = nullptr;
  int st = err_word(&p);
  if (st != USP_OK) return st;
  long long lim = g_spin_limit.load();
  g->err = p;
  g->spin_limit = lim < 0 ? kDefaultSpinLimit : lim;
  g->ns_limit = kWaitNs;
  return USP_OK;
}

// Per-device side stream for a kernel that may overlap the caller's stream.
struct SideSlot {
  std::mutex mu;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideSlot g_side[kMaxDevices];

size_t elt_size(usp_dtype d) { return d == USP_BF16 ? 2 : 4; }
bool dtype_ok(usp_dtype d) { return d == USP_F32 || d == USP_BF16; }
bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }
size_t round_up(size_t x) { return (x + 255) & ~size_t(255); }

int check_dims(int64_t B, int64_t H, int64_t N, int64_t D, int u, int r) {
  if (B < 0 || H < 0 || N < 0 || D < 1 || u < 1 || r < 1) return USP_ERR_INVALID_ARG;
  if (H % u != 0) return USP_ERR_DIVISIBILITY;               // Ulysses degree must divide the heads
  if (N % ((int64_t)u * r) != 0) return USP_ERR_DIVISIBILITY;  // no padding: N % sp == 0
  return USP_OK;
}

// Kernel support for a (dtype, D) pair.
int check_kernel(usp_dtype dt, int64_t D) {
  if (!dtype_ok(dt)) return USP_ERR_UNSUPPORTED;
  if (dt == USP_BF16 && D != 128) return USP_ERR_UNSUPPORTED;
  if (dt == USP_F32 && D > 128) return USP_ERR_UNSUPPORTED;
  return USP_OK;
}

// Delta and lse*log2(e) per row, rows padded to a multiple of 4 per shard so
// each (shard, head) row block starts 16-byte aligned (tensor-map pitch).
size_t bwd_vec_bytes(int64_t B, int64_t H, int64_t N, int u, int r) {
  const int64_t sp = (int64_t)u * r, Ns = N / sp;
  return round_up((size_t)(sp * B * H * ((Ns + 3) / 4 * 4)) * 4);
}

// Materialised backward: head-sharded copies of q, k, v, O, dO, lse, the
// head-sharded gradients, and the Delta / lse*log2(e) vectors of the kernels
// over the head-sharded stack viewed as [r*u][B*Hu][Nr] (rows padded to 4).
struct BwdWorkspace {
  size_t xq, xk, xv, xo, xdo, xl, xdq, xdk, xdv, delta, l2, total;
};
BwdWorkspace bwd_layout(int64_t B, int64_t H, int64_t N, int64_t D, int u, int r, usp_dtype dt) {
  const size_t t = round_up((size_t)(B * H * N * D) * elt_size(dt));
  const size_t lb = round_up((size_t)(B * H * N) * 4);
  const int64_t Nr = N / r;
  const size_t vb = round_up((size_t)((int64_t)r * B * H * ((Nr + 3) / 4 * 4)) * 4);
  BwdWorkspace w{};
  size_t off = 0;
  w.xq = off; off += t;
  w.xk = off; off += t;
  w.xv = off; off += t;
  w.xo = off; off += t;
  w.xdo = off; off += t;
  w.xl = off; off += lb;
  w.xdq = off; off += t;
  w.xdk = off; off += t;
  w.xdv = off; off += t;
  w.delta = off; off += vb;
  w.l2 = off; off += vb;
  w.total = off;
  (void)u;
  return w;
}

struct FwdWorkspace {
  size_t xq, xk, xv, parts_o, parts_l, xo, xl, total;
};
FwdWorkspace fwd_layout(int64_t B, int64_t H, int64_t N, int64_t D, int r, usp_dtype dt) {
  const size_t t = round_up((size_t)(B * H * N * D) * elt_size(dt));
  const size_t lb = round_up((size_t)(B * H * N) * 4);
  FwdWorkspace w{};
  size_t off = 0;
  w.xq = off; off += t;
  w.xk = off; off += t;
  w.xv = off; off += t;
  if (r > 1) {  // the merge writes the token-sharded result directly
    w.parts_o = off; off += (size_t)r * t;
    w.parts_l = off; off += (size_t)r * lb;
  } else {       // the chunk result, re-laid out head -> token afterwards
    w.xo = off; off += t;
    w.xl = off; off += lb;
  }
  w.total = off;
  return w;
}

// Joint (text + image) materialised forward: the image part of fwd_layout
// with ring + 1 partial planes (the last against the text K/V), plus the
// text-query partials (ring chunk planes + one text plane) when requested.
struct JointWorkspace {
  size_t xq, xk, xv, parts_o, parts_l, tparts_o, tparts_l, total;
};
JointWorkspace joint_layout(int64_t B, int64_t H, int64_t N, int64_t Nt, int64_t D, int r, usp_dtype dt,
                            bool text_queries) {
  const size_t t = round_up((size_t)(B * H * N * D) * elt_size(dt));
  const size_t lb = round_up((size_t)(B * H * N) * 4);
  JointWorkspace w{};
  size_t off = 0;
  w.xq = off; off += t;
  w.xk = off; off += t;
  w.xv = off; off += t;
  w.parts_o = off; off += (size_t)(r + 1) * t;  // merged straight into the token-sharded out, lse
  w.parts_l = off; off += (size_t)(r + 1) * lb;
  if (text_queries) {
    w.tparts_o = off; off += (size_t)(r + 1) * round_up((size_t)(B * H * Nt * D) * elt_size(dt));
    w.tparts_l = off; off += (size_t)(r + 1) * round_up((size_t)(B * H * Nt) * 4);
  }
  w.total = off;
  return w;
}

int relayout(const void* src, void* dst, int64_t B, int64_t H, int64_t N, int64_t D, int u, int r,
             int elt, bool tok2head, cudaStream_t s) {
  const int64_t Ns = N / ((int64_t)u * r);
  cudaError_t e = launch_relayout(src, dst, 0, B, H, Ns, D, u, r, elt, tok2head, s);
  return e == cudaSuccess ? USP_OK : cuda_fail(e);
}

// A stack of rows of D elements and its fp32 LSE stack, re-laid out the same
// way: one launch when both move in 16-byte vectors (Ns a multiple of 4),
// else one launch each (the LSE's 4-byte runs would slow the big tensor).
int relayout_with_lse(const void* x, void* x_dst, const float* l, float* l_dst, int64_t B, int64_t H, int64_t N,
                      int64_t D, int u, int r, int elt, bool tok2head, cudaStream_t s) {
  const int64_t Ns = N / ((int64_t)u * r);
  const uintptr_t a = (uintptr_t)x | (uintptr_t)x_dst | (uintptr_t)l | (uintptr_t)l_dst |
                      (uintptr_t)(Ns * 4) | (uintptr_t)(Ns * D * elt);
  if ((a & 15) == 0) {
    const void* srcs[2] = {x, l};
    void* dsts[2] = {x_dst, l_dst};
    const int64_t rb[2] = {D * elt, 4};
    cudaError_t e = launch_relayout_rows(srcs, dsts, rb, 2, B, H, Ns, u, r, tok2head, s);
    return e == cudaSuccess ? USP_OK : cuda_fail(e);
  }
  int st = relayout(x, x_dst, B, H, N, D, u, r, elt, tok2head, s);
  if (st != USP_OK) return st;
  return relayout(l, l_dst, B, H, N, 1, u, r, 4, tok2head, s);
}

// Attention of one or two problems on the kernel for `dt`: bf16 runs both
// in one tcgen05 launch, fp32 (FP32 pipes) one launch per problem.
int run_attention(const AttnArgs* a, int n, usp_dtype dt, int64_t D, cudaStream_t s) {
  for (int i = 0; i < n; ++i)
    if (a[i].units > 65535) return USP_ERR_UNSUPPORTED;
  cudaError_t e = cudaSuccess;
  if (dt == USP_F32) {
    for (int i = 0; i < n && e == cudaSuccess; ++i) e = launch_attn_f32(a[i], (int)D, s);
  } else {
    Guard g;
    int st = guard(&g);
    if (st != USP_OK) return st;
    e = launch_attn_tc_fwd(a, n, g, s);
  }
  return e == cudaSuccess ? USP_OK : cuda_fail(e);
}
int run_attention(const AttnArgs& a, usp_dtype dt, int64_t D, cudaStream_t s) {
  return run_attention(&a, 1, dt, D, s);
}

// Plain-operand attention arguments: q [q_heads][Nq][D] against k, v [kv_heads][Nk][D].
AttnArgs plain_args(const void* q, const void* k, const void* v, void* out, float* lse, int64_t Nq,
                    int64_t q_heads, int64_t Nk, int64_t kv_heads, float scale) {
  AttnArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = out; a.lse = lse;
  a.Nq = Nq; a.Nk = Nk;
  a.q_heads = q_heads; a.kv_heads = kv_heads;
  a.map.mode = kUnitPlain;
  a.units = q_heads;
  a.scale = scale;
  return a;
}

// Stack-operand arguments of the fused forward: every (b, h) head attends
// over all sp shards of its keys (and over the optional text keys).
AttnArgs stack_args(const void* q, const void* k, const void* v, void* out, float* lse, int64_t BH, int64_t sp,
                    int64_t Ns, float scale) {
  AttnArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = out; a.lse = lse;
  a.q_stack = a.kv_stack = a.out_stack = true;
  a.BH = BH; a.sp = sp; a.Ns = Ns;
  a.map.mode = kUnitPlain;
  a.units = BH;
  a.scale = scale;
  return a;
}

// Per-(rank, ring step) chunk attention over the head-sharded stacks; ring
// step t writes output plane t (plane = r*B*H heads of Nr rows).
AttnArgs ring_args(const void* q, const void* k, const void* v, void* out, float* lse, int64_t B, int64_t Hu,
                   int64_t Nr, int u, int r, float scale) {
  const int64_t plane = (int64_t)r * u * B * Hu;
  AttnArgs a = plain_args(q, k, v, out, lse, Nr, plane, Nr, plane, scale);
  a.map.mode = kUnitRing;
  a.map.sched = RingSchedule{u, r, r, (int)(B * Hu)};
  a.map.out_step_stride = plane;
  a.units = (int64_t)r * plane;
  return a;
}
int chunk_attention(const void* q, const void* k, const void* v, void* out, float* lse, int64_t B,
                    int64_t Hu, int64_t Nr, int64_t D, int u, int r, float scale, usp_dtype dt,
                    cudaStream_t s) {
  return run_attention(ring_args(q, k, v, out, lse, B, Hu, Nr, u, r, scale), dt, D, s);
}

}  // namespace

cudaError_t side_begin(cudaStream_t main, cudaStream_t* side) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  SideSlot& sl = g_side[dev];
  sl.mu.lock();
  if (!sl.stream) {
    e = cudaStreamCreateWithFlags(&sl.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sl.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sl.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      sl.mu.unlock();
      return e;
    }
  }
  e = cudaEventRecord(sl.fork, main);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sl.stream, sl.fork, 0);
  if (e != cudaSuccess) {
    sl.mu.unlock();
    return e;
  }
  *side = sl.stream;
  return cudaSuccess;
}

cudaError_t side_end(cudaStream_t main) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;  // cannot happen after side_begin succeeded on this thread
  SideSlot& sl = g_side[dev];
  e = cudaEventRecord(sl.join, sl.stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(main, sl.join, 0);
  sl.mu.unlock();
  return e;
}

}  // namespace usp

using namespace usp;

extern "C" {

int usp_relayout_tok2head(const void* src, void* dst, int64_t B, int64_t H, int64_t N, int64_t D, int ulysses,
                          int ring, usp_dtype dtype, usp_stream_t stream) {
  int st = check_dims(B, H, N, D, ulysses, ring);
  if (st != USP_OK) return st;
  if (!dtype_ok(dtype)) return USP_ERR_UNSUPPORTED;
  if (B * H * N == 0) return USP_OK;
  if (!src || !dst) return USP_ERR_INVALID_ARG;
  return relayout(src, dst, B, H, N, D, ulysses, ring, (int)elt_size(dtype), true, (cudaStream_t)stream);
}

int usp_relayout_head2tok(const void* src, void* dst, int64_t B, int64_t H, int64_t N, int64_t D, int ulysses,
                          int ring, usp_dtype dtype, usp_stream_t stream) {
  int st = check_dims(B, H, N, D, ulysses, ring);
  if (st != USP_OK) return st;
  if (!dtype_ok(dtype)) return USP_ERR_UNSUPPORTED;
  if (B * H * N == 0) return USP_OK;
  if (!src || !dst) return USP_ERR_INVALID_ARG;
  return relayout(src, dst, B, H, N, D, ulysses, ring, (int)elt_size(dtype), false, (cudaStream_t)stream);
}

int usp_attn_chunk_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int64_t B, int64_t H,
                       int64_t Nq, int64_t Nk, int64_t D, float scale, usp_dtype dtype, usp_stream_t stream) {
  if (B < 0 || H < 0 || Nq < 0 || D < 1) return USP_ERR_INVALID_ARG;
  if (Nk < 1) return USP_ERR_INVALID_ARG;  // softmax over an empty key set is undefined
  if (!std::isfinite(scale)) return USP_ERR_INVALID_ARG;
  int st = check_kernel(dtype, D);
  if (st != USP_OK) return st;
  if (B * H * Nq == 0) return USP_OK;
  if (!q || !k || !v || !out || !lse) return USP_ERR_INVALID_ARG;
  if (B * H > 65535) return USP_ERR_UNSUPPORTED;
  if (dtype == USP_BF16 && !(aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(out, 16)))
    return USP_ERR_INVALID_ARG;
  if (!aligned(lse, 4)) return USP_ERR_INVALID_ARG;
  return run_attention(plain_args(q, k, v, out, lse, Nq, B * H, Nk, B * H, scale), dtype, D,
                       (cudaStream_t)stream);
}

int usp_lse_merge(const void* outs, const float* lses, int R, void* out, float* lse, int64_t B, int64_t H,
                  int64_t Nq, int64_t D, usp_dtype dtype, usp_stream_t stream) {
  if (B < 0 || H < 0 || Nq < 0 || D < 1 || R < 1) return USP_ERR_INVALID_ARG;
  if (!dtype_ok(dtype)) return USP_ERR_UNSUPPORTED;
  if (B * H * Nq == 0) return USP_OK;
  if (!outs || !lses || !out || !lse) return USP_ERR_INVALID_ARG;
  cudaError_t e = launch_lse_merge(outs, lses, R, out, lse, B * H * Nq, D, (int)dtype, (cudaStream_t)stream);
  return e == cudaSuccess ? USP_OK : cuda_fail(e);
}

size_t usp_attention_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t D, int ulysses, int ring,
                                     usp_dtype dtype, usp_mode mode, int backward) {
  if (check_dims(B, H, N, D, ulysses, ring) != USP_OK || check_kernel(dtype, D) != USP_OK) return 0;
  if (backward && mode == USP_MATERIALISED) return bwd_layout(B, H, N, D, ulysses, ring, dtype).total;
  if (backward) return 2 * bwd_vec_bytes(B, H, N, ulysses, ring);  // Delta and lse*log2(e)
  if (mode == USP_FUSED) return 0;
  return fwd_layout(B, H, N, D, ring, dtype).total;
}

int usp_attention_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int64_t B, int64_t H,
                      int64_t N, int64_t D, int ulysses, int ring, float scale, usp_dtype dtype, usp_mode mode,
                      void* workspace, size_t workspace_bytes, usp_stream_t stream) {
  int st = check_dims(B, H, N, D, ulysses, ring);
  if (st != USP_OK) return st;
  if (!std::isfinite(scale)) return USP_ERR_INVALID_ARG;
  if (mode != USP_MATERIALISED && mode != USP_FUSED) return USP_ERR_INVALID_ARG;
  st = check_kernel(dtype, D);
  if (st != USP_OK) return st;
  if (B * H * N == 0) return USP_OK;
  if (!q || !k || !v || !out || !lse) return USP_ERR_INVALID_ARG;
  if (dtype == USP_BF16 && !(aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(out, 16)))
    return USP_ERR_INVALID_ARG;
  if (!aligned(lse, 4)) return USP_ERR_INVALID_ARG;
  const int u = ulysses, r = ring;
  const int64_t sp = (int64_t)u * r, Ns = N / sp, Nr = N / r, Hu = H / u;
  cudaStream_t s = (cudaStream_t)stream;

  if (mode == USP_FUSED) {
    if (dtype == USP_BF16) phase_begin(s);
    st = run_attention(stack_args(q, k, v, out, lse, B * H, sp, Ns, scale), dtype, D, s);
    if (st == USP_OK && dtype == USP_BF16) phase_mark(s);
    return st;
  }

  // materialised
  if ((int64_t)r * r * u * B * Hu > 65535) return USP_ERR_UNSUPPORTED;
  const FwdWorkspace w = fwd_layout(B, H, N, D, r, dtype);
  if (!workspace || workspace_bytes < w.total) return USP_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return USP_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  const int elt = (int)elt_size(dtype);
  phase_begin(s);
  {  // q, k, v in one launch
    const void* srcs[3] = {q, k, v};
    void* dsts[3] = {ws + w.xq, ws + w.xk, ws + w.xv};
    cudaError_t e = launch_relayout_n(srcs, dsts, 3, B, H, Ns, D, u, r, elt, true, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  phase_mark(s);
  void* o_dst = r > 1 ? (void*)(ws + w.parts_o) : (void*)(ws + w.xo);
  float* l_dst = r > 1 ? (float*)(ws + w.parts_l) : (float*)(ws + w.xl);
  if ((st = chunk_attention(ws + w.xq, ws + w.xk, ws + w.xv, o_dst, l_dst, B, Hu, Nr, D, u, r, scale, dtype, s)) !=
      USP_OK)
    return st;
  phase_mark(s);
  if (r > 1) {  // ring merge and the Ulysses head -> token exchange in one pass
    cudaError_t e = launch_lse_merge_to_tokens(ws + w.parts_o, (const float*)(ws + w.parts_l), r, out, lse, B, Hu,
                                               Nr, D, u, r, (int)dtype, s);
    if (e != cudaSuccess) return cuda_fail(e);
  } else {
    st = relayout_with_lse(ws + w.xo, out, (const float*)(ws + w.xl), lse, B, H, N, D, u, r, elt, false, s);
  }
  phase_mark(s);
  return st;
}

size_t usp_attention_joint_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t Nt, int64_t D, int ulysses,
                                           int ring, usp_dtype dtype, usp_mode mode, int with_text_queries) {
  if (Nt < 0) return 0;
  if (Nt == 0) return usp_attention_workspace_bytes(B, H, N, D, ulysses, ring, dtype, mode, 0);
  if (check_dims(B, H, N, D, ulysses, ring) != USP_OK || check_kernel(dtype, D) != USP_OK) return 0;
  if (mode == USP_FUSED) return 0;
  return joint_layout(B, H, N, Nt, D, ring, dtype, with_text_queries != 0).total;
}

int usp_attention_fwd_joint(const void* q, const void* k, const void* v, const void* q_txt, const void* k_txt,
                            const void* v_txt, void* out, float* lse, void* out_txt, float* lse_txt, int64_t B,
                            int64_t H, int64_t N, int64_t Nt, int64_t D, int ulysses, int ring, float scale,
                            usp_dtype dtype, usp_mode mode, void* workspace, size_t workspace_bytes,
                            usp_stream_t stream) {
  if (Nt < 0) return USP_ERR_INVALID_ARG;
  if (Nt == 0)
    return usp_attention_fwd(q, k, v, out, lse, B, H, N, D, ulysses, ring, scale, dtype, mode, workspace,
                             workspace_bytes, stream);
  int st = check_dims(B, H, N, D, ulysses, ring);
  if (st != USP_OK) return st;
  if (!std::isfinite(scale)) return USP_ERR_INVALID_ARG;
  if (mode != USP_MATERIALISED && mode != USP_FUSED) return USP_ERR_INVALID_ARG;
  st = check_kernel(dtype, D);
  if (st != USP_OK) return st;
  if (B * H == 0) return USP_OK;
  const bool tq = q_txt != nullptr;
  if (!k_txt || !v_txt || (N > 0 && (!q || !k || !v || !out || !lse)) || (tq && (!out_txt || !lse_txt)))
    return USP_ERR_INVALID_ARG;
  if (dtype == USP_BF16) {
    const void* ptrs[8] = {q, k, v, out, q_txt, k_txt, v_txt, out_txt};
    for (const void* p : ptrs)
      if (p && !aligned(p, 16)) return USP_ERR_INVALID_ARG;
  }
  if (!aligned(lse, 4) || !aligned(lse_txt, 4)) return USP_ERR_INVALID_ARG;
  const int u = ulysses, r = ring;
  const int64_t sp = (int64_t)u * r, Ns = N / sp, Nr = N / r, Hu = H / u, BH = B * H;
  const int64_t plane = (int64_t)r * BH;  // heads of one partial plane of the head-sharded stack
  cudaStream_t s = (cudaStream_t)stream;
  const bool prof = dtype == USP_BF16;

  if (mode == USP_FUSED) {
    // image queries over the image stack then the text; text queries the same
    AttnArgs a[2];
    int n = 0;
    if (N > 0) {
      a[n] = stack_args(q, k, v, out, lse, BH, sp, Ns, scale);
      a[n].k2 = k_txt; a[n].v2 = v_txt; a[n].Nk2 = Nt; a[n].kv2_heads = BH;
      ++n;
    }
    if (tq) {
      AttnArgs& t = a[n++];
      t = stack_args(q_txt, k, v, out_txt, lse_txt, BH, sp, Ns, scale);
      t.q_stack = t.out_stack = false;
      t.Nq = Nt; t.q_heads = BH;
      t.k2 = k_txt; t.v2 = v_txt; t.Nk2 = Nt; t.kv2_heads = BH;
      if (N == 0) {  // text keys only
        t.k = k_txt; t.v = v_txt; t.kv_stack = false; t.Nk = Nt; t.kv_heads = BH;
        t.k2 = t.v2 = nullptr; t.Nk2 = 0;
      }
    }
    if (n == 0) return USP_OK;
    if (prof) phase_begin(s);
    if ((st = run_attention(a, n, dtype, D, s)) != USP_OK) return st;
    if (prof) phase_mark(s);
    return USP_OK;
  }

  // materialised
  const JointWorkspace w = joint_layout(B, H, N, Nt, D, r, dtype, tq);
  if (!workspace || workspace_bytes < w.total) return USP_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return USP_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  const int elt = (int)elt_size(dtype);
  UnitMap joint_map{};
  joint_map.sched = RingSchedule{u, r, r, (int)(B * Hu)};
  joint_map.B = B; joint_map.H = H; joint_map.Hu = Hu;
  float* tl = (float*)(ws + w.tparts_l);
  // Partial attention launches.  Each pairs the image queries with the text
  // queries that read the same K/V: (A) the head-sharded image chunks --
  // ring steps of the image queries (planes 0..r-1) and the text queries of
  // head group j against chunk c of that group (text planes 0..r-1); (B) the
  // text K/V -- image queries of rank (g, j) against the text of head group
  // j (plane r) and the text queries against the text (last text plane).
  AttnArgs img_img, txt_img, img_txt, txt_txt;
  if (N > 0) {
    img_img = ring_args(ws + w.xq, ws + w.xk, ws + w.xv, ws + w.parts_o, (float*)(ws + w.parts_l), B, Hu, Nr, u, r,
                        scale);
    txt_img = plain_args(q_txt, ws + w.xk, ws + w.xv, ws + w.tparts_o, tl, Nt, BH, Nr, plane, scale);
    txt_img.map = joint_map;
    txt_img.map.mode = kUnitTxtImg;
    txt_img.map.out_step_stride = BH;
    txt_img.units = plane;
    img_txt = plain_args(ws + w.xq, k_txt, v_txt, ws + w.parts_o, (float*)(ws + w.parts_l), Nr, plane, Nt, BH,
                         scale);
    img_txt.map = joint_map;
    img_txt.map.mode = kUnitImgTxt;
    img_txt.map.out_base = (int64_t)r * plane;
    img_txt.units = plane;
  }
  const int R_txt = N > 0 ? r + 1 : 1;
  txt_txt = plain_args(q_txt, k_txt, v_txt, ws + w.tparts_o, tl, Nt, BH, Nt, BH, scale);
  txt_txt.map.out_base = (int64_t)(R_txt - 1) * BH;

  if (prof) phase_begin(s);
  if (N > 0) {
    const void* srcs[3] = {q, k, v};
    void* dsts[3] = {ws + w.xq, ws + w.xk, ws + w.xv};
    cudaError_t e = launch_relayout_n(srcs, dsts, 3, B, H, Ns, D, u, r, elt, true, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (prof) phase_mark(s);
  }
  {
    // The two attention launches read the re-laid inputs and write disjoint
    // partial planes: the short second one (every query set against the
    // text) runs on the device's side stream, so its CTAs fill the first
    // one's last wave instead of waiting behind it.
    AttnArgs A[2] = {img_img, txt_img};
    AttnArgs Bt[2];
    int n = 0;
    if (N > 0) Bt[n++] = img_txt;
    if (tq) Bt[n++] = txt_txt;
    cudaStream_t side = s;
    const bool fork = N > 0 && n > 0;
    if (fork) {
      cudaError_t e = side_begin(s, &side);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    if (N > 0) st = run_attention(A, tq ? 2 : 1, dtype, D, s);
    if (st == USP_OK && n > 0) st = run_attention(Bt, n, dtype, D, side);
    if (fork) {
      const cudaError_t j = side_end(s);  // always join, also after a failed launch
      if (st == USP_OK && j != cudaSuccess) st = cuda_fail(j);
    }
    if (st != USP_OK) return st;
  }
  if (prof) phase_mark(s);
  if (N > 0) {  // ring + text merge and the Ulysses head -> token exchange in one pass
    cudaError_t e = launch_lse_merge_to_tokens(ws + w.parts_o, (const float*)(ws + w.parts_l), (int)(r + 1), out, lse,
                                               B, Hu, Nr, D, u, r, (int)dtype, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (prof) phase_mark(s);
  }
  if (tq) {
    cudaError_t e = launch_lse_merge(ws + w.tparts_o, tl, R_txt, out_txt, lse_txt, BH * Nt, D, (int)dtype, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (prof) phase_mark(s);
  }
  return USP_OK;
}

int usp_cross_attention_fwd(const void* q, const void* k_txt, const void* v_txt, void* out, float* lse, int64_t B,
                            int64_t H, int64_t N, int64_t Nt, int64_t D, int ulysses, int ring, float scale,
                            usp_dtype dtype, usp_stream_t stream) {
  if (B < 0 || H < 0 || N < 0 || D < 1 || ulysses < 1 || ring < 1) return USP_ERR_INVALID_ARG;
  if (Nt < 1) return USP_ERR_INVALID_ARG;  // softmax over an empty key set is undefined
  if (N % ((int64_t)ulysses * ring) != 0) return USP_ERR_DIVISIBILITY;
  if (!std::isfinite(scale)) return USP_ERR_INVALID_ARG;
  int st = check_kernel(dtype, D);
  if (st != USP_OK) return st;
  if (B * H * N == 0) return USP_OK;
  if (!q || !k_txt || !v_txt || !out || !lse) return USP_ERR_INVALID_ARG;
  if (dtype == USP_BF16 && !(aligned(q, 16) && aligned(k_txt, 16) && aligned(v_txt, 16) && aligned(out, 16)))
    return USP_ERR_INVALID_ARG;
  if (!aligned(lse, 4)) return USP_ERR_INVALID_ARG;
  const int64_t sp = (int64_t)ulysses * ring, BH = B * H;
  AttnArgs a = stack_args(q, k_txt, v_txt, out, lse, BH, sp, N / sp, scale);
  a.kv_stack = false;
  a.Nk = Nt;
  a.kv_heads = BH;
  return run_attention(a, dtype, D, (cudaStream_t)stream);
}

int usp_quantize_e4m3(const void* x, void* x8, float* scales, int64_t B, int64_t H, int64_t N, int64_t D,
                      int ulysses, int ring, usp_stream_t stream) {
  if (B < 0 || H < 0 || N < 0 || D < 1 || ulysses < 1 || ring < 1) return USP_ERR_INVALID_ARG;
  if (N % ((int64_t)ulysses * ring) != 0) return USP_ERR_DIVISIBILITY;
  if (D % 16 != 0) return USP_ERR_UNSUPPORTED;
  if (B * H == 0) return USP_OK;
  if (!scales || (N > 0 && (!x || !x8))) return USP_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(x8, 16) || !aligned(scales, 4)) return USP_ERR_INVALID_ARG;
  const int64_t sp = (int64_t)ulysses * ring, BH = B * H;
  if (sp * BH > 65535) return USP_ERR_UNSUPPORTED;
  // the scales buffer doubles as the amax scratch (converted in place)
  cudaError_t e = launch_quantize_e4m3(x, static_cast<uint8_t*>(x8), scales, reinterpret_cast<unsigned*>(scales),
                                       BH, sp, N / sp, D, (cudaStream_t)stream);
  return e == cudaSuccess ? USP_OK : cuda_fail(e);
}

size_t usp_attention_fp8_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t D, int ulysses, int ring) {
  if (check_dims(B, H, N, D, ulysses, ring) != USP_OK || D != 128) return 0;
  const int64_t sp = (int64_t)ulysses * ring, Ns = N / sp, BH = B * H;
  const size_t codes = round_up((size_t)(sp * BH * Ns * 128));
  return 2 * codes + round_up((size_t)(sp * BH * 128 * fp8_vt_pitch(Ns))) + round_up((size_t)(3 * BH) * 4);
}

int usp_attention_fwd_fp8(const void* q, const void* k, const void* v, void* out, float* lse, int64_t B, int64_t H,
                          int64_t N, int64_t D, int ulysses, int ring, float scale, void* workspace,
                          size_t workspace_bytes, usp_stream_t stream) {
  int st = check_dims(B, H, N, D, ulysses, ring);
  if (st != USP_OK) return st;
  if (!std::isfinite(scale)) return USP_ERR_INVALID_ARG;
  if (D != 128) return USP_ERR_UNSUPPORTED;
  if (B * H * N == 0) return USP_OK;
  if (!q || !k || !v || !out || !lse) return USP_ERR_INVALID_ARG;
  if (!(aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(out, 16) && aligned(lse, 4)))
    return USP_ERR_INVALID_ARG;
  const size_t need = usp_attention_fp8_workspace_bytes(B, H, N, D, ulysses, ring);
  if (!workspace || workspace_bytes < need) return USP_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return USP_ERR_INVALID_ARG;
  const int64_t sp = (int64_t)ulysses * ring, Ns = N / sp, BH = B * H, Ns_pad = fp8_vt_pitch(Ns);
  if (BH > 65535 || sp * BH > 65535) return USP_ERR_UNSUPPORTED;
  char* ws = static_cast<char*>(workspace);
  const size_t codes = round_up((size_t)(sp * BH * Ns * 128));
  uint8_t* q8 = reinterpret_cast<uint8_t*>(ws);
  uint8_t* k8 = q8 + codes;
  uint8_t* vt8 = k8 + codes;
  unsigned* amax = reinterpret_cast<unsigned*>(vt8 + round_up((size_t)(sp * BH * 128 * Ns_pad)));
  cudaStream_t s = (cudaStream_t)stream;
  Guard g;
  if ((st = guard(&g)) != USP_OK) return st;
  phase_begin(s);
  cudaError_t e = launch_quantize_qkv_fp8(q, k, v, q8, k8, vt8, amax, BH, sp, Ns, s);
  if (e != cudaSuccess) return cuda_fail(e);
  phase_mark(s);
  Fp8AttnArgs a{};
  a.q8 = q8; a.k8 = k8; a.vt8 = vt8; a.amax = amax;
  a.out = out; a.lse = lse;
  a.BH = BH; a.sp = sp; a.Ns = Ns; a.Ns_pad = Ns_pad;
  a.scale = scale;
  e = launch_attn_fp8_fwd(a, g, s);
  if (e != cudaSuccess) return cuda_fail(e);
  phase_mark(s);
  return USP_OK;
}

int usp_attention_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t N, int64_t D,
                      int ulysses, int ring, float scale, usp_dtype dtype, void* workspace, size_t workspace_bytes,
                      usp_stream_t stream) {
  int st = check_dims(B, H, N, D, ulysses, ring);
  if (st != USP_OK) return st;
  if (!std::isfinite(scale)) return USP_ERR_INVALID_ARG;
  st = check_kernel(dtype, D);
  if (st != USP_OK) return st;
  if (B * H * N == 0) return USP_OK;
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return USP_ERR_INVALID_ARG;
  if (dtype == USP_BF16 && !(aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(out, 16) &&
                             aligned(dout, 16) && aligned(dq, 16) && aligned(dk, 16) && aligned(dv, 16)))
    return USP_ERR_INVALID_ARG;
  if (!aligned(lse, 4)) return USP_ERR_INVALID_ARG;
  const size_t lb = bwd_vec_bytes(B, H, N, ulysses, ring);
  if (!workspace || workspace_bytes < 2 * lb) return USP_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return USP_ERR_INVALID_ARG;
  const int64_t sp = (int64_t)ulysses * ring, Ns = N / sp;
  if (B * H > 65535 || (Ns + 127) / 128 * sp > 2147483647LL) return USP_ERR_UNSUPPORTED;
  float* delta = static_cast<float*>(workspace);
  float* l2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + lb);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (dtype == USP_F32) {
    e = launch_attn_f32_bwd((const float*)q, (const float*)k, (const float*)v, (const float*)out, lse,
                            (const float*)dout, (float*)dq, (float*)dk, (float*)dv, delta, B * H, sp, Ns, 1, (int)D,
                            scale, s);
  } else {
    Guard g;
    st = guard(&g);
    if (st != USP_OK) return st;
    TcBwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.out = out; a.dout = dout; a.lse = lse;
    a.dq = dq; a.dk = dk; a.dv = dv;
    a.delta = delta; a.l2 = l2;
    a.BH = B * H; a.sp = sp; a.Ns = Ns; a.useg = 1;
    a.scale = scale;
    phase_begin(s);
    e = launch_attn_tc_bwd(a, g, s);  // marks a phase after each of its three kernels
  }
  return e == cudaSuccess ? USP_OK : cuda_fail(e);
}

int usp_attention_bwd_materialised(const void* q, const void* k, const void* v, const void* out, const float* lse,
                                   const void* dout, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t N,
                                   int64_t D, int ulysses, int ring, float scale, usp_dtype dtype, void* workspace,
                                   size_t workspace_bytes, usp_stream_t stream) {
  int st = check_dims(B, H, N, D, ulysses, ring);
  if (st != USP_OK) return st;
  if (!std::isfinite(scale)) return USP_ERR_INVALID_ARG;
  st = check_kernel(dtype, D);
  if (st != USP_OK) return st;
  if (B * H * N == 0) return USP_OK;
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return USP_ERR_INVALID_ARG;
  if (dtype == USP_BF16 && !(aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(out, 16) &&
                             aligned(dout, 16) && aligned(dq, 16) && aligned(dk, 16) && aligned(dv, 16)))
    return USP_ERR_INVALID_ARG;
  if (!aligned(lse, 4)) return USP_ERR_INVALID_ARG;
  const int u = ulysses, r = ring;
  const BwdWorkspace w = bwd_layout(B, H, N, D, u, r, dtype);
  if (!workspace || workspace_bytes < w.total) return USP_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return USP_ERR_INVALID_ARG;
  const int64_t sp = (int64_t)u * r, Ns = N / sp, Nr = N / r, Hu = H / u;
  if (B * H > 65535 || (Nr + 127) / 128 * r > 2147483647LL) return USP_ERR_UNSUPPORTED;
  char* ws = static_cast<char*>(workspace);
  const int elt = (int)elt_size(dtype);
  cudaStream_t s = (cudaStream_t)stream;
  Guard g;
  if (dtype == USP_BF16 && (st = guard(&g)) != USP_OK) return st;
  phase_begin(s);
  {  // Ulysses token -> head of q, k, v, O, dO and the lse: one launch when the
     // lse runs are 16-byte multiples (Ns % 4 == 0), else the lse separately
    const void* srcs[6] = {q, k, v, out, dout, lse};
    void* dsts[6] = {ws + w.xq, ws + w.xk, ws + w.xv, ws + w.xo, ws + w.xdo, ws + w.xl};
    const int64_t rb[6] = {D * elt, D * elt, D * elt, D * elt, D * elt, 4};
    const bool with_lse = ((Ns * 4) & 15) == 0 && aligned(lse, 16);
    cudaError_t e = launch_relayout_rows(srcs, dsts, rb, with_lse ? 6 : 5, B, H, Ns, u, r, true, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (!with_lse && (st = relayout(lse, ws + w.xl, B, H, N, 1, u, r, 4, true, s)) != USP_OK) return st;
  }
  phase_mark(s);
  // Every (ring rank g, Ulysses rank j) unit over all ring chunks of its
  // heads, with the merged lse: the head-sharded stack viewed as
  // [r*u][B*Hu][Nr][D], whose unit (j, b, h') owns the segments g*u + j.
  float* delta = reinterpret_cast<float*>(ws + w.delta);
  cudaError_t e;
  if (dtype == USP_F32) {
    e = launch_attn_f32_bwd((const float*)(ws + w.xq), (const float*)(ws + w.xk), (const float*)(ws + w.xv),
                            (const float*)(ws + w.xo), (const float*)(ws + w.xl), (const float*)(ws + w.xdo),
                            (float*)(ws + w.xdq), (float*)(ws + w.xdk), (float*)(ws + w.xdv), delta, B * Hu, sp, Nr,
                            u, (int)D, scale, s);
    if (e == cudaSuccess) phase_mark(s);
  } else {
    TcBwdArgs a{};
    a.q = ws + w.xq; a.k = ws + w.xk; a.v = ws + w.xv; a.out = ws + w.xo; a.dout = ws + w.xdo;
    a.lse = reinterpret_cast<const float*>(ws + w.xl);
    a.dq = ws + w.xdq; a.dk = ws + w.xdk; a.dv = ws + w.xdv;
    a.delta = delta; a.l2 = reinterpret_cast<float*>(ws + w.l2);
    a.BH = B * Hu; a.sp = sp; a.Ns = Nr; a.useg = u;
    a.scale = scale;
    e = launch_attn_tc_bwd(a, g, s);  // marks a phase after each of its three kernels
    if (e == cudaSuccess) phase_mark(s);  // both kernels joined back on `s`
  }
  if (e != cudaSuccess) return cuda_fail(e);
  {  // the gradients head -> token in one launch
    const void* srcs[3] = {ws + w.xdq, ws + w.xdk, ws + w.xdv};
    void* dsts[3] = {dq, dk, dv};
    e = launch_relayout_n(srcs, dsts, 3, B, H, Ns, D, u, r, elt, false, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  phase_mark(s);
  return USP_OK;
}

int usp_device_status(usp_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int* p = nullptr;
  int st = err_word(&p);
  if (st != USP_OK) return st;
  unsigned int v = 0;
  e = cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e);
    return USP_ERR_TIMEOUT;
  }
  return USP_OK;
}

const char* usp_status_string(int status) {
  switch (status) {
    case USP_OK: return "USP_OK";
    case USP_ERR_INVALID_ARG: return "USP_ERR_INVALID_ARG";
    case USP_ERR_DIVISIBILITY: return "USP_ERR_DIVISIBILITY";
    case USP_ERR_UNSUPPORTED: return "USP_ERR_UNSUPPORTED";
    case USP_ERR_WORKSPACE: return "USP_ERR_WORKSPACE";
    case USP_ERR_CUDA: return "USP_ERR_CUDA";
    case USP_ERR_TIMEOUT: return "USP_ERR_TIMEOUT";
    default: return "USP_ERR_UNKNOWN";
  }
}

int usp_last_cuda_error(void) { return t_last_cuda_error; }

void usp_set_debug_spin_limit(long long polls) { g_spin_limit.store(polls < 0 ? -1 : polls); }

void usp_set_spin_limit(long long polls) { usp_set_debug_spin_limit(polls); }

int usp_profile_phases(int enable) {
  if (enable && !t_phase.created) {
    for (int i = 0; i <= kMaxPhases; ++i) {
      cudaError_t e = cudaEventCreate(&t_phase.ev[i]);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    t_phase.created = true;
  }
  t_phase.enabled = enable != 0;
  if (enable) t_phase.marks = 0;  // disabling keeps the last recorded call readable
  return USP_OK;
}

int usp_profile_read(float* ms, int max_phases) {
  if (!t_phase.created || t_phase.marks < 2) return 0;
  const int n = t_phase.marks - 1;
  for (int i = 1; i <= n; ++i) {  // phases may end on different streams
    cudaError_t e = cudaEventSynchronize(t_phase.ev[i]);
    if (e != cudaSuccess) return -cuda_fail(e);
  }
  for (int i = 0; i < n && i < max_phases; ++i) {
    cudaError_t e = cudaEventElapsedTime(&ms[i], t_phase.ev[t_phase.from[i + 1]], t_phase.ev[i + 1]);
    if (e != cudaSuccess) return -cuda_fail(e);
  }
  return n < max_phases ? n : max_phases;
}

}  // extern "C"
