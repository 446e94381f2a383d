// fp32 attention with log-sum-exp on the FP32 pipes (no tensor cores: the
// 1e-5 bound of the handbook's fp32 demo rules out tf32).
//
// One warp owns one query row.  The block stages K and V tiles of 32 keys in
// shared memory; lane l scores key l of the tile, the row maximum and sum use
// warp-shuffle reductions (online softmax), and each lane accumulates the
// output dimensions d = lane + 32*i.  All arithmetic is IEEE fp32 with expf.
//
// Addressing: each operand is either plain [heads][rows][D] or the
// token-sharded stack [sp][BH][Ns][D] (sp*Ns rows per head); a unit (one
// query head against one KV head) is mapped to heads by the UnitMap (plain,
// materialised ring step, image-vs-text, text-vs-image chunk).  An optional
// second KV source (plain; the text tokens of joint attention) follows the
// first source's keys in the same online softmax.
#include "usp_internal.cuh"

namespace usp {
namespace {

constexpr int kWarps = 8;
constexpr int kTileK = 32;

// Stack addressing [segments][BH][Ns][D]: a unit ("head") h in [0, useg*BH)
// is (j, bh) = (h / BH, h % BH) and its k-th Ns-row segment is k*useg + j
// (the token-sharded stack: useg = 1; the materialised path's head-sharded
// stack [r*u][B*Hu][Nr][D]: useg = u).
struct F32Addr {
  bool fused;
  int64_t BH, Ns;
  int64_t useg = 1;
  __device__ __forceinline__ int64_t lse_off(int64_t head, int64_t row, int64_t nrows) const {
    if (!fused) return head * nrows + row;
    const int64_t j = head / BH, bh = head - j * BH;
    const int64_t s = row / Ns, n = row - s * Ns;
    return ((s * useg + j) * BH + bh) * Ns + n;
  }
  __device__ __forceinline__ int64_t row_off(int64_t head, int64_t row, int64_t nrows, int D) const {
    return lse_off(head, row, nrows) * (int64_t)D;
  }
};

// One operand of the forward: plain [heads][rows][D] or the token-sharded
// stack [sp][BH][Ns][D] read as sp*Ns rows per head.
struct F32Operand {
  const float* k;
  const float* v;
  bool stack;
  int64_t rows;  // rows per head
  __device__ __forceinline__ int64_t off(int64_t head, int64_t row, int D, const F32Addr& st) const {
    return stack ? st.row_off(head, row, 0, D) : (head * rows + row) * (int64_t)D;
  }
};

struct F32Fwd {
  const float* q;
  float* out;
  float* lse;
  bool q_stack;  // out follows q
  int64_t Nq;
  F32Operand kv, kv2;  // kv2.rows == 0: no second source
  F32Addr stack;
  UnitMap map;
  float scale;
};

template <int kDmax>
__global__ void __launch_bounds__(kWarps * 32) attn_f32_kernel(const F32Fwd p, int D) {
  __shared__ float Ks[kTileK][kDmax + 1];
  __shared__ float Vs[kTileK][kDmax];
  __shared__ float Qs[kWarps][kDmax];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const UnitHeads U = map_unit(p.map, blockIdx.y);
  const F32Operand qop{p.q, nullptr, p.q_stack, p.Nq};

  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  const bool active = row < p.Nq;
  if (active)
    for (int d = lane; d < D; d += 32) Qs[warp][d] = p.q[qop.off(U.qh, row, D, p.stack) + d];

  float m = -INFINITY, l = 0.f;
  float o[kDmax / 32];
#pragma unroll
  for (int i = 0; i < kDmax / 32; ++i) o[i] = 0.f;

  const int64_t n1 = p.kv.rows, Nk = n1 + p.kv2.rows;  // keys: first source, then second
  for (int64_t j0 = 0; j0 < Nk; j0 += kTileK) {
    __syncthreads();
    const int nk = (int)((Nk - j0) < kTileK ? (Nk - j0) : kTileK);
    for (int e = threadIdx.x; e < kTileK * D; e += blockDim.x) {
      const int jj = e / D, d = e - jj * D;
      float kv = 0.f, vv = 0.f;
      if (jj < nk) {
        const int64_t key = j0 + jj;
        const bool second = key >= n1;
        const F32Operand& src = second ? p.kv2 : p.kv;
        const int64_t off = src.off(second ? U.kvh2 : U.kvh, second ? key - n1 : key, D, p.stack) + d;
        kv = src.k[off];
        vv = src.v[off];
      }
      Ks[jj][d] = kv;
      Vs[jj][d] = vv;
    }
    __syncthreads();
    if (!active) continue;
    float s = -INFINITY;
    if (lane < nk) {
      float acc = 0.f;
      for (int d = 0; d < D; ++d) acc = fmaf(Qs[warp][d], Ks[lane][d], acc);
      s = acc * p.scale;
    }
    float mx = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(m, mx);
    const float pr = (lane < nk) ? expf(s - m_new) : 0.f;
    const float alpha = expf(m - m_new);  // m = -inf on the first tile -> 0
    float ps = pr;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
#pragma unroll
    for (int i = 0; i < kDmax / 32; ++i) o[i] *= alpha;
    for (int jj = 0; jj < nk; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, pr, jj);
#pragma unroll
      for (int i = 0; i < kDmax / 32; ++i) {
        const int d = lane + 32 * i;
        if (d < D) o[i] = fmaf(pj, Vs[jj][d], o[i]);
      }
    }
    m = m_new;
  }
  if (!active) return;
  const float inv = 1.f / l;
  const int64_t ooff = qop.off(U.oh, row, D, p.stack);
#pragma unroll
  for (int i = 0; i < kDmax / 32; ++i) {
    const int d = lane + 32 * i;
    if (d < D) p.out[ooff + d] = o[i] * inv;
  }
  if (lane == 0) p.lse[ooff / D] = m + logf(l);
}

// ---------------------------------------------------------------- backward
// Delta_i = sum_d dO_id O_id, one warp per row, shuffle reduction.
__global__ void __launch_bounds__(256) f32_bwd_delta_kernel(const float* __restrict__ out,
                                                            const float* __restrict__ dout, float* __restrict__ delta,
                                                            int64_t rows, int D) {
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  float acc = 0.f;
  for (int d = lane; d < D; d += 32) acc = fmaf(out[row * D + d], dout[row * D + d], acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) delta[row] = acc;
}

// One warp per "own" row (a query row for dQ, a key row for dK/dV); the other
// side streams through shared memory 32 rows at a time, lane l taking row l.
//   dQ_i  = scale sum_j P_ij (dP_ij - Delta_i) k_j
//   dV_j  = sum_i P_ij dO_i,   dK_j = scale sum_i P_ij (dP_ij - Delta_i) q_i
// with P_ij = exp(scale q_i.k_j - lse_i), dP_ij = dO_i . v_j.
template <int kDmax, bool kDQ>
__global__ void __launch_bounds__(kWarps * 32) f32_bwd_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ lse, const float* __restrict__ delta, const float* __restrict__ dout,
    float* __restrict__ g0, float* __restrict__ g1, int64_t N, int D, float scale, F32Addr addr) {
  __shared__ float A[kTileK][kDmax + 1];  // streamed: k (dQ) or q (dK/dV)
  __shared__ float Bs[kTileK][kDmax + 1]; // streamed: v (dQ) or dO (dK/dV)
  __shared__ float Ls[kTileK], Ds[kTileK];
  __shared__ float Own0[kWarps][kDmax], Own1[kWarps][kDmax];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t head = blockIdx.y;
  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  const bool active = row < N;
  float own_l = 0.f, own_d = 0.f;
  if (active) {
    const int64_t off = addr.row_off(head, row, N, D);
    for (int d = lane; d < D; d += 32) {
      Own0[warp][d] = kDQ ? q[off + d] : k[off + d];
      Own1[warp][d] = kDQ ? dout[off + d] : v[off + d];
    }
    if (kDQ) {
      own_l = lse[addr.lse_off(head, row, N)];
      own_d = delta[addr.lse_off(head, row, N)];
    }
  }
  float acc0[kDmax / 32], acc1[kDmax / 32];
#pragma unroll
  for (int i = 0; i < kDmax / 32; ++i) acc0[i] = acc1[i] = 0.f;
  for (int64_t j0 = 0; j0 < N; j0 += kTileK) {
    __syncthreads();
    const int nt = (int)((N - j0) < kTileK ? (N - j0) : kTileK);
    for (int e = threadIdx.x; e < kTileK * D; e += blockDim.x) {
      const int jj = e / D, d = e - jj * D;
      float a = 0.f, b = 0.f;
      if (jj < nt) {
        const int64_t off = addr.row_off(head, j0 + jj, N, D) + d;
        a = kDQ ? k[off] : q[off];
        b = kDQ ? v[off] : dout[off];
      }
      A[jj][d] = a;
      Bs[jj][d] = b;
    }
    if (!kDQ && threadIdx.x < kTileK) {
      const int jj = threadIdx.x;
      Ls[jj] = jj < nt ? lse[addr.lse_off(head, j0 + jj, N)] : 0.f;
      Ds[jj] = jj < nt ? delta[addr.lse_off(head, j0 + jj, N)] : 0.f;
    }
    __syncthreads();
    if (!active) continue;
    float p = 0.f, ds = 0.f;
    if (lane < nt) {
      float s = 0.f, dp = 0.f;
      for (int d = 0; d < D; ++d) {
        s = fmaf(Own0[warp][d], A[lane][d], s);
        dp = fmaf(kDQ ? Own1[warp][d] : Bs[lane][d], kDQ ? Bs[lane][d] : Own1[warp][d], dp);
      }
      const float l = kDQ ? own_l : Ls[lane];
      const float dl = kDQ ? own_d : Ds[lane];
      p = expf(s * scale - l);
      ds = p * (dp - dl);
    }
    for (int jj = 0; jj < nt; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
      for (int i = 0; i < kDmax / 32; ++i) {
        const int d = lane + 32 * i;
        if (d < D) {
          if (kDQ) {
            acc0[i] = fmaf(dsj, A[jj][d], acc0[i]);             // dQ += dS k
          } else {
            acc0[i] = fmaf(dsj, A[jj][d], acc0[i]);             // dK += dS q
            acc1[i] = fmaf(pj, Bs[jj][d], acc1[i]);             // dV += P dO
          }
        }
      }
    }
  }
  if (!active) return;
  const int64_t off = addr.row_off(head, row, N, D);
#pragma unroll
  for (int i = 0; i < kDmax / 32; ++i) {
    const int d = lane + 32 * i;
    if (d < D) {
      g0[off + d] = acc0[i] * scale;
      if (!kDQ) g1[off + d] = acc1[i];
    }
  }
}

template <int kDmax>
cudaError_t launch_bwd_dmax(const float* q, const float* k, const float* v, const float* out, const float* lse,
                            const float* dout, float* dq, float* dk, float* dv, float* delta, int64_t BH, int64_t N,
                            int D, float scale, F32Addr addr, cudaStream_t stream) {
  const int64_t rows = BH * N;
  f32_bwd_delta_kernel<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, stream>>>(out, dout, delta, rows, D);
  dim3 grid((unsigned)((N + kWarps - 1) / kWarps), (unsigned)BH, 1);
  f32_bwd_kernel<kDmax, true><<<grid, kWarps * 32, 0, stream>>>(q, k, v, lse, delta, dout, dq, nullptr, N, D, scale, addr);
  f32_bwd_kernel<kDmax, false><<<grid, kWarps * 32, 0, stream>>>(q, k, v, lse, delta, dout, dk, dv, N, D, scale, addr);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_f32_bwd(const float* q, const float* k, const float* v, const float* out,
                                const float* lse, const float* dout, float* dq, float* dk, float* dv,
                                float* delta, int64_t BH, int64_t sp, int64_t Ns, int useg, int D, float scale,
                                cudaStream_t stream) {
  F32Addr addr{true, BH, Ns, useg};
  const int64_t N = sp / useg * Ns, U = BH * useg;  // rows per unit, units
  if (D <= 32) return launch_bwd_dmax<32>(q, k, v, out, lse, dout, dq, dk, dv, delta, U, N, D, scale, addr, stream);
  if (D <= 64) return launch_bwd_dmax<64>(q, k, v, out, lse, dout, dq, dk, dv, delta, U, N, D, scale, addr, stream);
  return launch_bwd_dmax<128>(q, k, v, out, lse, dout, dq, dk, dv, delta, U, N, D, scale, addr, stream);
}

cudaError_t launch_attn_f32(const AttnArgs& a, int D, cudaStream_t stream) {
  if (a.out_stack != a.q_stack) return cudaErrorInvalidValue;  // out rows follow the query rows
  F32Fwd p{};
  p.q = static_cast<const float*>(a.q);
  p.out = static_cast<float*>(a.out);
  p.lse = a.lse;
  p.q_stack = a.q_stack;
  p.Nq = a.q_stack ? a.sp * a.Ns : a.Nq;
  p.kv = F32Operand{static_cast<const float*>(a.k), static_cast<const float*>(a.v), a.kv_stack,
                    a.kv_stack ? a.sp * a.Ns : a.Nk};
  p.kv2 = F32Operand{static_cast<const float*>(a.k2), static_cast<const float*>(a.v2), false,
                     a.k2 ? a.Nk2 : 0};
  p.stack = F32Addr{true, a.BH, a.Ns};
  p.map = a.map;
  p.scale = a.scale;
  dim3 grid((unsigned)((p.Nq + kWarps - 1) / kWarps), (unsigned)a.units, 1);
  if (D <= 32)
    attn_f32_kernel<32><<<grid, kWarps * 32, 0, stream>>>(p, D);
  else if (D <= 64)
    attn_f32_kernel<64><<<grid, kWarps * 32, 0, stream>>>(p, D);
  else
    attn_f32_kernel<128><<<grid, kWarps * 32, 0, stream>>>(p, D);
  return cudaGetLastError();
}

}  // namespace usp
