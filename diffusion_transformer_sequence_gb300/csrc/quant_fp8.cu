// Per-head FP8 (OCP E4M3) quantisation of token-sharded stacks, the first
// step of the FP8 attention path ("Multi-GPU parallelism: spreading one step
// over several cards", Wan latency table: FP8 low precision as the last step).
//
// For each tensor and each (b, h) head, over every shard, token and
// dimension of the stack [sp][B*H][Ns][D]:
//   amax = max |x|;  inv = 448 / amax;  code = e4m3_rn_satfinite(x * inv)
// (amax = 0 gives inv = 1), both fp32 operations rounded to nearest, so the
// codes are reproducible bit for bit on the host.  The dequantisation scale
// amax / 448 is formed by the consumers.
//
// Kernels (all HBM-bound streaming):
//   amax_kernel    one CTA per 16 KB chunk of a (shard, head) block; block
//                  reduction, one atomicMax on the float bits per CTA
//                  (non-negative floats order like their bit patterns)
//   quant_kernel   16 elements per thread, codes in the input layout
//   quant_vt_kernel  V for the P V product: 128-key x 128-dim tiles staged
//                  through shared memory (4 keys per 32-bit word) and written
//                  transposed, [D][Ns_pad] per (shard, head) with zero
//                  padding, so V^T tiles are K-major operands (keys
//                  contiguous) for the tensor cores.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "usp_internal.cuh"

namespace usp {
namespace {

constexpr int kThreads = 256;
constexpr int64_t kChunk = 8192;  // elements per amax CTA

__device__ __forceinline__ float inv_scale(unsigned amax_bits) {
  const float a = __uint_as_float(amax_bits);
  return a > 0.f ? __fdiv_rn(448.f, a) : 1.f;
}

struct Srcs3 {
  const __nv_bfloat16* p[3];
  // constant-index selection keeps the parameter block out of local memory
  __device__ __forceinline__ const __nv_bfloat16* get(int i) const { return i == 0 ? p[0] : (i == 1 ? p[1] : p[2]); }
};

// amax[t][bh] over blocks (s, bh) of Ns*D contiguous elements.
__global__ void __launch_bounds__(kThreads) amax_kernel(Srcs3 srcs, unsigned* __restrict__ amax, int64_t BH,
                                                        int64_t block_elems) {
  const int t = blockIdx.z;
  const int64_t blk = blockIdx.y;                  // s * BH + bh
  const int64_t bh = blk % BH;
  const int64_t e0 = (int64_t)blockIdx.x * kChunk;
  const __nv_bfloat16* src = srcs.get(t) + blk * block_elems;
  const int64_t e1 = e0 + kChunk < block_elems ? e0 + kChunk : block_elems;
  float m = 0.f;
  for (int64_t e = e0 + 8 * (int64_t)threadIdx.x; e < e1; e += 8 * kThreads) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src + e));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m = fmaxf(m, __uint_as_float((w[i] & 0x7FFFu) << 16));          // |low half|
      m = fmaxf(m, __uint_as_float(w[i] & 0x7FFF0000u));              // |high half|
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  __shared__ float red[kThreads / 32];
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
    atomicMax(amax + (int64_t)t * BH + bh, __float_as_uint(m));
  }
}

struct Dsts3 {
  uint8_t* p[3];
  int tensor[3];  // which amax row each source uses
  __device__ __forceinline__ uint8_t* get(int i) const { return i == 0 ? p[0] : (i == 1 ? p[1] : p[2]); }
  __device__ __forceinline__ int row(int i) const { return i == 0 ? tensor[0] : (i == 1 ? tensor[1] : tensor[2]); }
};

// Codes in the input layout, 16 elements per thread.
__global__ void __launch_bounds__(kThreads) quant_kernel(Srcs3 srcs, Dsts3 dsts, const unsigned* __restrict__ amax,
                                                         int64_t BH, int64_t block_elems, int64_t total) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int z = blockIdx.y;
  const int64_t e = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * 16;
  if (e >= total) return;
  const int64_t bh = (e / block_elems) % BH;
  const float inv = inv_scale(__ldg(amax + (int64_t)dsts.row(z) * BH + bh));
  const uint4* s = reinterpret_cast<const uint4*>(srcs.get(z) + e);
  const uint4 a = __ldg(s), b = __ldg(s + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float x0 = __fmul_rn(__uint_as_float(w[2 * i] << 16), inv);
    const float x1 = __fmul_rn(__uint_as_float(w[2 * i] & 0xFFFF0000u), inv);
    const float x2 = __fmul_rn(__uint_as_float(w[2 * i + 1] << 16), inv);
    const float x3 = __fmul_rn(__uint_as_float(w[2 * i + 1] & 0xFFFF0000u), inv);
    out[i] = (uint32_t)ptx::e4m3x2(x0, x1) | ((uint32_t)ptx::e4m3x2(x2, x3) << 16);
  }
  *reinterpret_cast<uint4*>(dsts.get(z) + e) = make_uint4(out[0], out[1], out[2], out[3]);
}

// V^T: for each (s, bh) and 128-key tile, dst[s][bh][d][key] (row pitch Ns_pad).
// A thread reads 4 consecutive keys x 8 dims (16 lanes cover one 256-byte
// key row, so loads are coalesced) and packs, per dim, the 4 keys' codes into
// one 32-bit word of a shared [128 d][32 words] tile; word column kq of row d
// sits at kq ^ 4*((d/8) % 8), which limits the stores to 2-way bank conflicts
// and keeps each 16-byte group of 16 keys contiguous for the write-out.
__global__ void __launch_bounds__(kThreads) quant_vt_kernel(const __nv_bfloat16* __restrict__ v,
                                                            uint8_t* __restrict__ vt,
                                                            const unsigned* __restrict__ amax_v, int64_t BH,
                                                            int64_t Ns, int64_t Ns_pad) {
  __shared__ __align__(16) uint32_t tile[128 * 32];
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int64_t key0 = (int64_t)blockIdx.x * 128;
  const int64_t bh = blockIdx.y, s = blockIdx.z;
  const float inv = inv_scale(__ldg(amax_v + bh));
  const __nv_bfloat16* src = v + ((s * BH + bh) * Ns) * 128;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int dq = lane % 16, d0 = 8 * dq;
  const int sw = 4 * (dq & 7);
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int kq = pass * 16 + warp * 2 + lane / 16;  // keys 4kq .. 4kq+3 of the tile
    uint32_t w[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int64_t key = key0 + 4 * kq + r;
      if (key < Ns) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src + key * 128 + d0));
        w[r][0] = raw.x; w[r][1] = raw.y; w[r][2] = raw.z; w[r][3] = raw.w;
      } else {
        w[r][0] = w[r][1] = w[r][2] = w[r][3] = 0u;
      }
    }
#pragma unroll
    for (int dd = 0; dd < 8; ++dd) {
      float x[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t h = w[r][dd / 2];
        x[r] = __fmul_rn(__uint_as_float((dd & 1) ? (h & 0xFFFF0000u) : (h << 16)), inv);
      }
      tile[(d0 + dd) * 32 + (kq ^ sw)] = (uint32_t)ptx::e4m3x2(x[0], x[1]) | ((uint32_t)ptx::e4m3x2(x[2], x[3]) << 16);
    }
  }
  __syncthreads();
  uint8_t* dst = vt + ((s * BH + bh) * 128) * Ns_pad;
  for (int i = threadIdx.x; i < 128 * 8; i += kThreads) {
    const int d = i / 8, c = i % 8;                  // 16 keys [16c, 16c + 16) of dim row d
    const int64_t k = key0 + 16 * c;
    if (k < Ns_pad) {
      const uint4 val = *reinterpret_cast<const uint4*>(tile + d * 32 + 4 * (c ^ ((d >> 3) & 7)));
      *reinterpret_cast<uint4*>(dst + d * Ns_pad + k) = val;
    }
  }
}

// In place is allowed (amax and scales may be the same buffer): each thread
// reads and writes only its own element.
__global__ void scales_kernel(const unsigned* amax, float* scales, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float a = __uint_as_float(amax[i]);
  scales[i] = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
}

cudaError_t launch_amax(const void* const* srcs, int count, unsigned* amax, int64_t BH, int64_t sp, int64_t Ns,
                        int64_t D, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned) * BH * count, stream);
  if (e != cudaSuccess) return e;
  Srcs3 s{};
  for (int i = 0; i < count; ++i) s.p[i] = static_cast<const __nv_bfloat16*>(srcs[i]);
  const int64_t block_elems = Ns * D;
  dim3 grid((unsigned)((block_elems + kChunk - 1) / kChunk), (unsigned)(sp * BH), (unsigned)count);
  amax_kernel<<<grid, kThreads, 0, stream>>>(s, amax, BH, block_elems);
  return cudaGetLastError();
}

cudaError_t launch_quant(const void* const* srcs, uint8_t* const* dsts, const int* tensor, int count,
                         const unsigned* amax, int64_t BH, int64_t sp, int64_t Ns, int64_t D, cudaStream_t stream) {
  Srcs3 s{};
  Dsts3 d{};
  for (int i = 0; i < count; ++i) {
    s.p[i] = static_cast<const __nv_bfloat16*>(srcs[i]);
    d.p[i] = dsts[i];
    d.tensor[i] = tensor[i];
  }
  const int64_t total = sp * BH * Ns * D;
  dim3 grid((unsigned)((total / 16 + kThreads - 1) / kThreads), (unsigned)count, 1);
  return launch_pdl(quant_kernel, grid, dim3(kThreads), 0, stream, s, d, amax, BH, Ns * D, total);
}

}  // namespace

int64_t fp8_vt_pitch(int64_t Ns) { return (Ns + 15) / 16 * 16; }

cudaError_t launch_quantize_e4m3(const void* x, uint8_t* x8, float* scales, unsigned* amax, int64_t BH, int64_t sp,
                                 int64_t Ns, int64_t D, cudaStream_t stream) {
  cudaError_t e = launch_amax(&x, 1, amax, BH, sp, Ns, D, stream);
  if (e != cudaSuccess) return e;
  const int t0 = 0;
  e = launch_quant(&x, &x8, &t0, 1, amax, BH, sp, Ns, D, stream);
  if (e != cudaSuccess) return e;
  scales_kernel<<<(unsigned)((BH + 255) / 256), 256, 0, stream>>>(amax, scales, BH);
  return cudaGetLastError();
}

cudaError_t launch_quantize_qkv_fp8(const void* q, const void* k, const void* v, uint8_t* q8, uint8_t* k8,
                                    uint8_t* vt8, unsigned* amax, int64_t BH, int64_t sp, int64_t Ns,
                                    cudaStream_t stream) {
  const void* srcs[3] = {q, k, v};
  cudaError_t e = launch_amax(srcs, 3, amax, BH, sp, Ns, 128, stream);
  if (e != cudaSuccess) return e;
  uint8_t* dsts[2] = {q8, k8};
  const int tensor[2] = {0, 1};
  e = launch_quant(srcs, dsts, tensor, 2, amax, BH, sp, Ns, 128, stream);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((Ns + 127) / 128), (unsigned)BH, (unsigned)sp);
  return launch_pdl(quant_vt_kernel, grid, dim3(kThreads), 0, stream, static_cast<const __nv_bfloat16*>(v), vt8,
                    (const unsigned*)(amax + 2 * BH), BH, Ns, fp8_vt_pitch(Ns));
}

}  // namespace usp
