// Ulysses all-to-all as an on-device re-layout (token-sharded <-> head-sharded).
//
// Both directions are a batched copy of contiguous runs of Ns*D elements:
//   tok2head: run (g, j, b, h', s) of the head-sharded stack
//             X[g, j, b, h', s*Ns : (s+1)*Ns, :]  <-  T[g, s, b, j*Hu + h', :, :]
//   head2tok: run (g, s, b, h) of the token-sharded stack
//             T[g, s, b, h, :, :]  <-  X[g, h / Hu, b, h % Hu, s*Ns : (s+1)*Ns, :]
// ("Multi-GPU parallelism: spreading one step over several cards", section
// "Sequence parallelism: Ulysses and Ring": all_to_all_heads / _tokens.)
// Every run is contiguous on both sides, so the kernel streams each run with
// the widest aligned vector (16 bytes on every workload) and several loads in
// flight per thread; staging through shared memory would add a copy without
// improving coalescing.  Run-level index arithmetic happens once per CTA.
#include "ptx.cuh"
#include "usp_internal.cuh"

namespace usp {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

template <typename Vec>
__device__ __forceinline__ Vec load_stream(const Vec* p) { return __ldg(p); }

// Up to six tensors per launch (blockIdx.z picks one), with the same run
// layout but each its own run length: q, k and v of the materialised forward
// (q, k, v, O, dO and the LSE of the materialised backward) go through one
// launch, and so do an output and its LSE.
constexpr int kMaxTensors = 6;
struct Tensors {
  const void* src[kMaxTensors];
  void* dst[kMaxTensors];
  int64_t run_vecs[kMaxTensors];
};

template <typename Vec, bool kTok2Head>
__global__ void __launch_bounds__(kThreads) relayout_kernel(const __grid_constant__ Tensors ts, int64_t nruns,
                                                            int64_t B, int64_t H, int64_t Hu, int64_t u) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int64_t run_vecs = ts.run_vecs[blockIdx.z];
  if ((int64_t)blockIdx.x * kThreads * kUnroll >= run_vecs) return;  // a shorter tensor of the launch
  const Vec* __restrict__ src = static_cast<const Vec*>(ts.src[blockIdx.z]);
  Vec* __restrict__ dst = static_cast<Vec*>(ts.dst[blockIdx.z]);
  for (int64_t run = blockIdx.y; run < nruns; run += gridDim.y) {
    int64_t src_run;
    if (kTok2Head) {
      // destination run order (g, j, b, h', s)
      int64_t t = run;
      const int64_t s = t % u; t /= u;
      const int64_t hp = t % Hu; t /= Hu;
      const int64_t b = t % B; t /= B;
      const int64_t j = t % u;
      const int64_t g = t / u;
      src_run = ((g * u + s) * B + b) * H + j * Hu + hp;
    } else {
      // destination run order (g, s, b, h)
      int64_t t = run;
      const int64_t h = t % H; t /= H;
      const int64_t b = t % B; t /= B;
      const int64_t s = t % u;
      const int64_t g = t / u;
      const int64_t j = h / Hu, hp = h % Hu;
      src_run = (((g * u + j) * B + b) * Hu + hp) * u + s;
    }
    const Vec* __restrict__ sp = src + src_run * run_vecs;
    Vec* __restrict__ dp = dst + run * run_vecs;
    const int64_t step = (int64_t)gridDim.x * kThreads * kUnroll;
    for (int64_t i0 = (int64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; i0 < run_vecs; i0 += step) {
      Vec tmp[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int64_t i = i0 + (int64_t)k * kThreads;
        if (i < run_vecs) tmp[k] = load_stream(sp + i);
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int64_t i = i0 + (int64_t)k * kThreads;
        if (i < run_vecs) dp[i] = tmp[k];
      }
    }
  }
}

template <typename Vec>
cudaError_t launch_vec(Tensors ts, int count, int64_t nruns, const int64_t* run_bytes, int64_t B, int64_t H,
                       int64_t Hu, int64_t u, bool tok2head, cudaStream_t stream) {
  int64_t run_vecs = 0;  // longest run of the launch, in vectors
  for (int i = 0; i < count; ++i) {
    ts.run_vecs[i] = run_bytes[i] / (int64_t)sizeof(Vec);
    if (ts.run_vecs[i] > run_vecs) run_vecs = ts.run_vecs[i];
  }
  const int64_t per_cta = (int64_t)kThreads * kUnroll;
  int64_t gx = (run_vecs + per_cta - 1) / per_cta;
  if (gx > 1024) gx = 1024;
  int64_t gy = nruns < 65535 ? nruns : 65535;
  dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)count);
  if (tok2head) return launch_pdl(relayout_kernel<Vec, true>, grid, dim3(kThreads), 0, stream, ts, nruns, B, H, Hu, u);
  return launch_pdl(relayout_kernel<Vec, false>, grid, dim3(kThreads), 0, stream, ts, nruns, B, H, Hu, u);
}

}  // namespace

cudaError_t launch_relayout_rows(const void* const* srcs, void* const* dsts, const int64_t* row_bytes, int count,
                                 int64_t B, int64_t H, int64_t Ns, int ulysses, int ring, bool tok2head,
                                 cudaStream_t stream) {
  if (count < 1 || count > kMaxTensors) return cudaErrorInvalidValue;
  const int64_t u = ulysses;
  const int64_t Hu = H / u;
  const int64_t nruns = (int64_t)ring * u * B * H;
  Tensors ts{};
  int64_t run_bytes[kMaxTensors];
  uintptr_t a = 0;
  for (int i = 0; i < count; ++i) {
    ts.src[i] = srcs[i];
    ts.dst[i] = dsts[i];
    run_bytes[i] = Ns * row_bytes[i];
    a |= (uintptr_t)srcs[i] | (uintptr_t)dsts[i] | (uintptr_t)run_bytes[i];
  }
  if ((a & 15) == 0) return launch_vec<uint4>(ts, count, nruns, run_bytes, B, H, Hu, u, tok2head, stream);
  if ((a & 7) == 0) return launch_vec<uint2>(ts, count, nruns, run_bytes, B, H, Hu, u, tok2head, stream);
  if ((a & 3) == 0) return launch_vec<uint32_t>(ts, count, nruns, run_bytes, B, H, Hu, u, tok2head, stream);
  if ((a & 1) == 0) return launch_vec<uint16_t>(ts, count, nruns, run_bytes, B, H, Hu, u, tok2head, stream);
  return launch_vec<uint8_t>(ts, count, nruns, run_bytes, B, H, Hu, u, tok2head, stream);
}

cudaError_t launch_relayout_n(const void* const* srcs, void* const* dsts, int count, int64_t B, int64_t H,
                              int64_t Ns, int64_t D, int ulysses, int ring, int elt, bool tok2head,
                              cudaStream_t stream) {
  if (count < 1 || count > kMaxTensors) return cudaErrorInvalidValue;
  int64_t rb[kMaxTensors];
  for (int i = 0; i < count; ++i) rb[i] = D * elt;
  return launch_relayout_rows(srcs, dsts, rb, count, B, H, Ns, ulysses, ring, tok2head, stream);
}

cudaError_t launch_relayout(const void* src, void* dst, int64_t /*runs_outer*/, int64_t B, int64_t H,
                            int64_t Ns, int64_t D, int ulysses, int ring, int elt, bool tok2head,
                            cudaStream_t stream) {
  return launch_relayout_n(&src, &dst, 1, B, H, Ns, D, ulysses, ring, elt, tok2head, stream);
}

}  // namespace usp
