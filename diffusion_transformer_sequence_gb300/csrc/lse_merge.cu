// The Ring step's log-sum-exp merge of R partial attention results.
//
// "Multi-GPU parallelism: spreading one step over several cards", section
// "Sequence parallelism: Ulysses and Ring": each KV block that arrives round
// the ring yields a local attention result; a log-sum-exp merge (the
// online-softmax rule) combines them.  Per row, in fp32:
//   m = max_t lse_t;  L = m + ln sum_t exp(lse_t - m);  out = sum_t exp(lse_t - L) out_t
// The merge is over the R ring steps of one row, not across D, so a row's D
// elements are split over threads in 16-byte vectors and no cross-thread
// reduction is needed.  HBM-bound: reads R rows of partials + R LSEs, writes
// one row + one LSE.  Inside the materialised USP forward the merge also
// performs the Ulysses head -> token re-layout (merge_tok_kernel).
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "usp_internal.cuh"

namespace usp {

bool lse_merge_to_tokens_ok(const void* outs, const void* out, int R, int64_t B, int64_t Hu, int64_t Nr, int64_t D,
                            int u, int r) {
  const uintptr_t a = (uintptr_t)outs | (uintptr_t)out;
  return (D == 128 || D == 64 || D == 32 || D == 16) && (a & 15) == 0 && R >= 1 && R <= 8 &&
         B * Hu <= 65535 && (int64_t)r * u <= 65535 && Nr * 16 + 255 < 2147483647LL;
}

namespace {

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float* f) {
  uint4 raw;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = raw;
}
__device__ __forceinline__ void store8(float* p, const float* f) {
  reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
// Eight elements held as loaded (packed bf16 stays 4 registers).
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 v;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ void get(float* f) const {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void get(float* f) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// 8 elements (16 or 32 bytes) per thread; D % 8 == 0, R <= kMaxR.
template <typename T, int kMaxR>
__global__ void __launch_bounds__(256) merge_vec_kernel(const T* __restrict__ outs,
                                                        const float* __restrict__ lses, int R,
                                                        T* __restrict__ out, float* __restrict__ lse,
                                                        int64_t rows, int64_t D) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int64_t tpr = D / 8;
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = gt / tpr;
  const int64_t c = (gt - row * tpr) * 8;
  if (row >= rows) return;
  // every load of the thread is issued before any arithmetic (the partials
  // and the LSEs are independent, so their memory latencies overlap); the
  // row statistics use the hardware exp2 / log2 approximations (relative
  // error ~1e-7, far inside the merge's fp32 and bf16 tolerances)
  const int64_t plane = rows * D;
  Raw8<T> x[kMaxR];
  float lv[kMaxR];
#pragma unroll
  for (int t = 0; t < kMaxR; ++t) {
    if (t < R) {
      x[t].load(outs + t * plane + row * D + c);
      lv[t] = __ldg(lses + t * rows + row);
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int t = 0; t < kMaxR; ++t)
    if (t < R) m = fmaxf(m, lv[t]);
  float s = 0.f;
#pragma unroll
  for (int t = 0; t < kMaxR; ++t)
    if (t < R) s += __expf(lv[t] - m);
  const float L = m + __logf(s);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
  for (int t = 0; t < kMaxR; ++t) {
    if (t < R) {
      const float wt = __expf(lv[t] - L);
      float f[8];
      x[t].get(f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wt, f[i], acc[i]);
    }
  }
  store8(out + row * D + c, acc);
  if (c == 0) lse[row] = L;
}

// Generic: one thread per output element (any D, any R).
template <typename T>
__global__ void __launch_bounds__(256) merge_scalar_kernel(const T* __restrict__ outs,
                                                           const float* __restrict__ lses, int R,
                                                           T* __restrict__ out, float* __restrict__ lse,
                                                           int64_t rows, int64_t D) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= rows * D) return;
  const int64_t row = gt / D;
  float m = -INFINITY;
  for (int t = 0; t < R; ++t) m = fmaxf(m, lses[t * rows + row]);
  float s = 0.f;
  for (int t = 0; t < R; ++t) s += expf(lses[t * rows + row] - m);
  const float L = m + logf(s);
  float acc = 0.f;
  for (int t = 0; t < R; ++t) acc = fmaf(expf(lses[t * rows + row] - L), to_f(outs[t * rows * D + gt]), acc);
  from_f(out + gt, acc);
  if (gt - row * D == 0) lse[row] = L;
}

// The merge fused with the Ulysses head -> token re-layout: the partials are
// planes of the head-sharded stack [r, u, B, Hu, Nr, D]; each merged row
// goes straight to its place in the token-sharded stack [r, u, B, H, Ns, D]
// (and its LSE to [r, u, B, H, Ns]), so the merged head-sharded result is
// never written.  Head-sharded row (g, j, b, h', n) is token-sharded row
// (g, n / Ns, b, j*Hu + h', n % Ns): the handbook's all_to_all_tokens as
// addressing.  grid.z = g*u + j, grid.y = b*Hu + h', grid.x = blocks of
// rows; a thread merges kVec 8-element vectors of one row (D / (8*kVec)
// threads per row), so the index arithmetic is paid once per 8*kVec elements.
template <typename T, int kMaxR, int kD, int kVec>
__global__ void __launch_bounds__(256) merge_tok_kernel(const T* __restrict__ outs, const float* __restrict__ lses,
                                                        int R, T* __restrict__ out, float* __restrict__ lse,
                                                        int64_t rows, int u, int B, int Hu, int Nr, int Ns) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  constexpr int kTpr = kD / (8 * kVec);  // threads per row
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int n = t / kTpr;
  if (n >= Nr) return;
  const int c0 = (t - n * kTpr) * 8;
  const int j = (int)blockIdx.z % u, g = (int)blockIdx.z / u;
  const int b = (int)blockIdx.y / Hu, hh = (int)blockIdx.y - b * Hu;
  const int s = n / Ns, n2 = n - s * Ns;
  const int64_t unit = ((int64_t)blockIdx.z * B + b) * Hu + hh;
  const int64_t row = unit * Nr + n;
  const int64_t orow = ((((int64_t)g * u + s) * B + b) * ((int64_t)u * Hu) + (int64_t)j * Hu + hh) * Ns + n2;
  const int64_t plane = rows * kD;
  Raw8<T> x[kMaxR][kVec];
  float lv[kMaxR];
#pragma unroll
  for (int q = 0; q < kMaxR; ++q) {
    if (q < R) {
#pragma unroll
      for (int v = 0; v < kVec; ++v) x[q][v].load(outs + q * plane + row * kD + c0 + v * 8 * kTpr);
      lv[q] = __ldg(lses + q * rows + row);
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int q = 0; q < kMaxR; ++q)
    if (q < R) m = fmaxf(m, lv[q]);
  float sum = 0.f;
#pragma unroll
  for (int q = 0; q < kMaxR; ++q)
    if (q < R) sum += __expf(lv[q] - m);
  const float L = m + __logf(sum);
  float wt[kMaxR];
#pragma unroll
  for (int q = 0; q < kMaxR; ++q) wt[q] = q < R ? __expf(lv[q] - L) : 0.f;
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxR; ++q) {
      if (q < R) {
        float f[8];
        x[q][v].get(f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wt[q], f[i], acc[i]);
      }
    }
    store8(out + orow * kD + c0 + v * 8 * kTpr, acc);
  }
  if (c0 == 0) lse[orow] = L;
}

// Generic form of merge_tok_kernel: one thread per output element.
template <typename T>
__global__ void __launch_bounds__(256) merge_tok_scalar_kernel(const T* __restrict__ outs,
                                                               const float* __restrict__ lses, int R,
                                                               T* __restrict__ out, float* __restrict__ lse,
                                                               int64_t rows, int64_t D, int64_t u, int64_t B,
                                                               int64_t Hu, int64_t Nr, int64_t Ns) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= rows * D) return;
  const int64_t row = gt / D, d = gt - row * D;
  const int64_t unit = row / Nr, n = row - unit * Nr;
  const int64_t hh = unit % Hu, b = (unit / Hu) % B, j = (unit / Hu / B) % u, g = unit / Hu / B / u;
  const int64_t s = n / Ns;
  const int64_t orow = (((g * u + s) * B + b) * (u * Hu) + j * Hu + hh) * Ns + (n - s * Ns);
  float m = -INFINITY;
  for (int q = 0; q < R; ++q) m = fmaxf(m, lses[q * rows + row]);
  float sum = 0.f;
  for (int q = 0; q < R; ++q) sum += expf(lses[q * rows + row] - m);
  const float L = m + logf(sum);
  float acc = 0.f;
  for (int q = 0; q < R; ++q) acc = fmaf(expf(lses[q * rows + row] - L), to_f(outs[q * rows * D + gt]), acc);
  from_f(out + orow * D + d, acc);
  if (d == 0) lse[orow] = L;
}

template <typename T, int kD, int kVec>
cudaError_t launch_tok_vec(const void* outs, const float* lses, int R, void* out, float* lse, int64_t rows, int u,
                           int B, int Hu, int Nr, int Ns, int r, cudaStream_t stream) {
  constexpr int kTpr = kD / (8 * kVec);
  const dim3 g((unsigned)(((int64_t)Nr * kTpr + 255) / 256), (unsigned)(B * Hu), (unsigned)(r * u)), b(256);
  if (R <= 2)
    return launch_pdl(merge_tok_kernel<T, 2, kD, kVec>, g, b, 0, stream, (const T*)outs, lses, R, (T*)out, lse, rows,
                      u, B, Hu, Nr, Ns);
  if (R <= 4)
    return launch_pdl(merge_tok_kernel<T, 4, kD, kVec>, g, b, 0, stream, (const T*)outs, lses, R, (T*)out, lse, rows,
                      u, B, Hu, Nr, Ns);
  return launch_pdl(merge_tok_kernel<T, 8, kD, kVec>, g, b, 0, stream, (const T*)outs, lses, R, (T*)out, lse, rows, u,
                    B, Hu, Nr, Ns);
}

template <typename T>
cudaError_t launch_typed_tok(const void* outs, const float* lses, int R, void* out, float* lse, int64_t B,
                             int64_t Hu, int64_t Nr, int64_t D, int u, int r, cudaStream_t stream) {
  const int64_t Ns = Nr / u;
  const int64_t rows = (int64_t)r * u * B * Hu * Nr;
  if (lse_merge_to_tokens_ok(outs, out, R, B, Hu, Nr, D, u, r)) {
    const int iu = u, iB = (int)B, iHu = (int)Hu, iNr = (int)Nr, iNs = (int)Ns;
    // four vectors per thread for bf16 (64 bytes of each partial), two for fp32
    if (D == 128 && sizeof(T) == 2)
      return launch_tok_vec<T, 128, 4>(outs, lses, R, out, lse, rows, iu, iB, iHu, iNr, iNs, r, stream);
    if (D == 128) return launch_tok_vec<T, 128, 2>(outs, lses, R, out, lse, rows, iu, iB, iHu, iNr, iNs, r, stream);
    if (D == 64) return launch_tok_vec<T, 64, 2>(outs, lses, R, out, lse, rows, iu, iB, iHu, iNr, iNs, r, stream);
    if (D == 32) return launch_tok_vec<T, 32, 2>(outs, lses, R, out, lse, rows, iu, iB, iHu, iNr, iNs, r, stream);
    if (D == 16) return launch_tok_vec<T, 16, 1>(outs, lses, R, out, lse, rows, iu, iB, iHu, iNr, iNs, r, stream);
  }
  return launch_pdl(merge_tok_scalar_kernel<T>, dim3((unsigned)((rows * D + 255) / 256)), dim3(256), 0, stream,
                    (const T*)outs, lses, R, (T*)out, lse, rows, D, (int64_t)u, B, Hu, Nr, Ns);
}

template <typename T>
cudaError_t launch_typed(const void* outs, const float* lses, int R, void* out, float* lse, int64_t rows,
                         int64_t D, cudaStream_t stream) {
  const uintptr_t a = (uintptr_t)outs | (uintptr_t)out;
  const bool vec = (D % 8 == 0) && ((a & 15) == 0) && R <= 8;
  if (vec) {
    const int64_t threads = rows * (D / 8);
    const int64_t blocks = (threads + 255) / 256;
    const dim3 g((unsigned)blocks), b(256);
    if (R <= 2) return launch_pdl(merge_vec_kernel<T, 2>, g, b, 0, stream, (const T*)outs, lses, R, (T*)out, lse, rows, D);
    if (R <= 4) return launch_pdl(merge_vec_kernel<T, 4>, g, b, 0, stream, (const T*)outs, lses, R, (T*)out, lse, rows, D);
    return launch_pdl(merge_vec_kernel<T, 8>, g, b, 0, stream, (const T*)outs, lses, R, (T*)out, lse, rows, D);
  }
  const int64_t blocks = (rows * D + 255) / 256;
  return launch_pdl(merge_scalar_kernel<T>, dim3((unsigned)blocks), dim3(256), 0, stream, (const T*)outs, lses, R,
                    (T*)out, lse, rows, D);
}

}  // namespace

cudaError_t launch_lse_merge_to_tokens(const void* outs, const float* lses, int R, void* out, float* lse, int64_t B,
                                       int64_t Hu, int64_t Nr, int64_t D, int u, int r, int dtype,
                                       cudaStream_t stream) {
  if (dtype == 1) return launch_typed_tok<__nv_bfloat16>(outs, lses, R, out, lse, B, Hu, Nr, D, u, r, stream);
  return launch_typed_tok<float>(outs, lses, R, out, lse, B, Hu, Nr, D, u, r, stream);
}

cudaError_t launch_lse_merge(const void* outs, const float* lses, int R, void* out, float* lse,
                             int64_t rows, int64_t D, int dtype, cudaStream_t stream) {
  if (dtype == 1) return launch_typed<__nv_bfloat16>(outs, lses, R, out, lse, rows, D, stream);
  return launch_typed<float>(outs, lses, R, out, lse, rows, D, stream);
}

}  // namespace usp
