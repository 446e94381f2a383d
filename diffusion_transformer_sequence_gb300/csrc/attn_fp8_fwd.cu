// FP8 (OCP E4M3) fused USP attention forward on the tcgen05 tensor cores
// (D = 128), the low-precision step of "Multi-GPU parallelism: spreading one
// step over several cards" (Wan latency table: FP8 low precision).
//
// Inputs are the per-head quantised stacks of quant_fp8.cu: codes Q8, K8
// [sp][B*H][Ns][128] and V8^T [sp][B*H][128][Ns_pad], plus each tensor's
// per-head amax (dequantisation scale amax / 448).  Per (b, h) head and
// query row i, over every shard's keys (the ring merge happens inside the
// online softmax, as in the bf16 fused kernel):
//   S_ij = (q8_i . k8_j) * sq * sk * scale
//   P_ij = 2^(S_ij log2 e - m_i + 4)  rounded to E4M3 for the P V product
//   out_i = sv * sum_j P_ij v8_j / sum_j P_ij,  lse_i = ln sum_j exp(S_ij)
// with the row sum taken over the unrounded P in fp32.  The offset 4 (and a
// running maximum that only moves when it grows by more than 4) keeps every
// P in [0, 256], inside E4M3's range (448), and puts every P within 2^-10 of
// the row maximum in E4M3's normal range (3 mantissa bits) rather than
// among its subnormals.
//
// Structure as the bf16 kernel (one CTA per SM, 384 threads: TMA producer,
// MMA issuer, two softmax warpgroups in ping-pong over two 128-row query
// tiles; S and O accumulate in TMEM), with these differences:
//   * every GEMM is kind::f8f6f4 with both operands K-major in shared memory:
//     Q K^T from the Q and K tiles (128-byte rows = one 128B swizzle atom),
//     P V from P (written by the softmax warps into shared memory, swizzled)
//     and the V^T tile (keys contiguous, from the transposed V8^T);
//   * tiles are half the bytes, so the K/V ring has three stages.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "usp_internal.cuh"

namespace usp {
namespace {

constexpr int BM = 128;          // query rows per tile
constexpr int BN = 128;          // keys per tile
constexpr int HD = 128;          // head dim
constexpr int KV_STAGES = 3;
constexpr int TILE = BM * HD;    // one 128 x 128 E4M3 tile: 16 KB
constexpr int NUM_THREADS = 384;
constexpr float RESCALE_THRESHOLD = 4.0f;  // log2 units
constexpr float P_OFFSET = 4.0f;           // P = 2^(x - m + 4) <= 2^(4 + 4) = 256 < 448
constexpr int REGS_CTRL = 56;
constexpr int REGS_SOFTMAX = (NUM_THREADS * 168 - 128 * REGS_CTRL) / 256 / 8 * 8;
static_assert(128 * REGS_CTRL + 256 * REGS_SOFTMAX <= NUM_THREADS * 168, "register split exceeds the launch");

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + 2 * TILE;
constexpr int OFF_V = OFF_K + KV_STAGES * TILE;
constexpr int OFF_P = OFF_V + KV_STAGES * TILE;
constexpr int OFF_BAR = OFF_P + 2 * TILE;
constexpr int B_QFULL = 0;
constexpr int B_KFULL = 1;
constexpr int B_KEMPTY = B_KFULL + KV_STAGES;
constexpr int B_VFULL = B_KEMPTY + KV_STAGES;
constexpr int B_VEMPTY = B_VFULL + KV_STAGES;
constexpr int B_SFULL = B_VEMPTY + KV_STAGES;
constexpr int B_PFULL = B_SFULL + 2;
constexpr int B_ODONE = B_PFULL + 2;
constexpr int B_MMADONE = B_ODONE + 2;
constexpr int NUM_BARS = B_MMADONE + 1;
constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_SLOT + 8;
constexpr int SMEM_USED = OFF_ABORT + 8;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment of the base

struct Fp8Params {
  __nv_bfloat16* out;       // token-sharded stack [sp][BH][Ns][128]
  float* lse;               // [sp][BH][Ns]
  const unsigned* amax;     // [3][BH] float bits: q, k, v
  int64_t BH, Ns;
  int tps;                  // 128-row tiles per shard
  int tiles;                // tiles per head: tps * sp
  float scale_log2;         // scale * log2(e)
  Guard guard;
};

__device__ __forceinline__ float deq_scale(unsigned amax_bits) {
  const float a = __uint_as_float(amax_bits);
  return a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fp8_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_vt, const __grid_constant__ Fp8Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_SLOT);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int bh = blockIdx.y;
  const int qt0 = 2 * blockIdx.x;
  const int qt1 = (qt0 + 1 < p.tiles) ? qt0 + 1 : -1;  // -1: no second tile (compute on a copy)
  const int kv_total = p.tiles;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(B_QFULL), 1);
    for (int s = 0; s < KV_STAGES; ++s) {
      ptx::mbar_init(bar(B_KFULL + s), 1);
      ptx::mbar_init(bar(B_KEMPTY + s), 1);
      ptx::mbar_init(bar(B_VFULL + s), 1);
      ptx::mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(B_SFULL + i), 1);
      ptx::mbar_init(bar(B_PFULL + i), 128);
      ptx::mbar_init(bar(B_ODONE + i), 1);
    }
    ptx::mbar_init(bar(B_MMADONE), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + OFF_SLOT, 512);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_vt);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::griddep_wait();    // the prologue above overlapped the quantisation's tail
  ptx::griddep_launch();
  const uint32_t tmem = *tmem_slot;
  const Guard& G = p.guard;
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(REGS_CTRL) : "memory");
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      auto seg_row = [&](int t, int& seg, int& row0) {
        seg = t / p.tps;
        row0 = (t - seg * p.tps) * BM;
      };
      int seg, row0;
      ptx::mbar_arrive_expect_tx(bar(B_QFULL), 2 * TILE);
      seg_row(qt0, seg, row0);
      ptx::tma_load_4d(sbase + OFF_Q, &tm_q, bar(B_QFULL), 0, row0, bh, seg);
      seg_row(qt1 >= 0 ? qt1 : qt0, seg, row0);
      ptx::tma_load_4d(sbase + OFF_Q + TILE, &tm_q, bar(B_QFULL), 0, row0, bh, seg);
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < kv_total; ++j) {
        const int s = j % KV_STAGES;
        const uint32_t ph = (uint32_t)((j / KV_STAGES) & 1);
        seg_row(j, seg, row0);
        if (!ptx::mbar_wait(bar(B_KEMPTY + s), ph ^ 1u, G, abort_flag, kDevTimeoutTmaProducer)) break;
        ptx::mbar_arrive_expect_tx(bar(B_KFULL + s), TILE);
        ptx::tma_load_4d(sbase + OFF_K + s * TILE, &tm_k, bar(B_KFULL + s), 0, row0, bh, seg);
        issued_k = j + 1;
        if (!ptx::mbar_wait(bar(B_VEMPTY + s), ph ^ 1u, G, abort_flag, kDevTimeoutTmaProducer)) break;
        ptx::mbar_arrive_expect_tx(bar(B_VFULL + s), TILE);
        // V^T tile: keys [row0, row0 + 128) of shard seg, all 128 dims
        ptx::tma_load_4d(sbase + OFF_V + s * TILE, &tm_vt, bar(B_VFULL + s), row0, 0, bh, seg);
        issued_v = j + 1;
      }
      const uint64_t drain_ns = 200000000ull;
      ptx::mbar_drain(bar(B_QFULL), 0, drain_ns);
      for (int j = issued_k - KV_STAGES; j < issued_k; ++j)
        if (j >= 0) ptx::mbar_drain(bar(B_KFULL + j % KV_STAGES), (uint32_t)((j / KV_STAGES) & 1), drain_ns);
      for (int j = issued_v - KV_STAGES; j < issued_v; ++j)
        if (j >= 0) ptx::mbar_drain(bar(B_VFULL + j % KV_STAGES), (uint32_t)((j / KV_STAGES) & 1), drain_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = ptx::idesc_e4m3_f32(BM, BN);  // both GEMMs: M = N = 128, K-major operands
      const uint32_t tS[2] = {tmem, tmem + 128};
      const uint32_t tO[2] = {tmem + 256, tmem + 384};
      bool ok = ptx::mbar_wait(bar(B_QFULL), 0, G, abort_flag, kDevTimeoutMma);
      // K-major, 128-byte rows, 8-row groups 1024 B apart; a K = 32 step
      // advances the start address by 32 bytes inside the swizzle atom.
      const uint64_t dQ0 = ptx::smem_desc_sw128(sbase + OFF_Q, 16, 1024);
      const uint64_t dK0 = ptx::smem_desc_sw128(sbase + OFF_K, 16, 1024);
      const uint64_t dV0 = ptx::smem_desc_sw128(sbase + OFF_V, 16, 1024);
      const uint64_t dP0 = ptx::smem_desc_sw128(sbase + OFF_P, 16, 1024);
      auto issue_pv = [&](int i, int jv) {
        const uint64_t dv = ptx::launder(dV0 + (uint64_t)(((jv % KV_STAGES) * TILE) >> 4));
        const uint64_t dp = ptx::launder(dP0 + (uint64_t)((i * TILE) >> 4));
#pragma unroll
        for (int kk = 0; kk < BN / 32; ++kk)
          ptx::mma_ss_f8(tO[i], dp + (uint64_t)(kk * 2), dv + (uint64_t)(kk * 2), IDESC, (jv > 0 || kk > 0) ? 1u : 0u);
      };
      auto issue_s = [&](int i, int jk) {
        const uint64_t dk = ptx::launder(dK0 + (uint64_t)(((jk % KV_STAGES) * TILE) >> 4));
        const uint64_t dq = ptx::launder(dQ0 + (uint64_t)((i * TILE) >> 4));
#pragma unroll
        for (int kk = 0; kk < HD / 32; ++kk)
          ptx::mma_ss_f8(tS[i], dq + (uint64_t)(kk * 2), dk + (uint64_t)(kk * 2), IDESC, kk > 0 ? 1u : 0u);
      };
      for (int j = 0; ok && j < kv_total; ++j) {
        const int s = j % KV_STAGES;
        if (!(ok = ptx::mbar_wait(bar(B_KFULL + s), (uint32_t)((j / KV_STAGES) & 1), G, abort_flag, kDevTimeoutMma))) break;
        ptx::tc_fence_after();
        for (int i = 0; i < 2; ++i) {
          if (j > 0) {
            const int jv = j - 1;
            if (!(ok = ptx::mbar_wait(bar(B_PFULL + i), (uint32_t)(jv & 1), G, abort_flag, kDevTimeoutMma))) break;
            if (i == 0 && !(ok = ptx::mbar_wait(bar(B_VFULL + jv % KV_STAGES), (uint32_t)((jv / KV_STAGES) & 1), G,
                                                abort_flag, kDevTimeoutMma)))
              break;
            ptx::tc_fence_after();
            issue_pv(i, jv);
            if (i == 1) ptx::mma_commit(bar(B_VEMPTY + jv % KV_STAGES));
          }
          issue_s(i, j);
          ptx::mma_commit(bar(B_SFULL + i));
        }
        if (!ok) break;
        ptx::mma_commit(bar(B_KEMPTY + s));
      }
      if (ok) {
        const int jl = kv_total - 1;
        for (int i = 0; i < 2 && ok; ++i) {
          if (!(ok = ptx::mbar_wait(bar(B_PFULL + i), (uint32_t)(jl & 1), G, abort_flag, kDevTimeoutMma))) break;
          if (i == 0 && !(ok = ptx::mbar_wait(bar(B_VFULL + jl % KV_STAGES), (uint32_t)((jl / KV_STAGES) & 1), G,
                                              abort_flag, kDevTimeoutMma)))
            break;
          ptx::tc_fence_after();
          issue_pv(i, jl);
          ptx::mma_commit(bar(B_ODONE + i));
        }
        if (ok) ptx::mma_commit(bar(B_VEMPTY + jl % KV_STAGES));
      }
      ptx::mma_commit(bar(B_MMADONE));
      ptx::mbar_drain(bar(B_MMADONE), 0, 200000000ull);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(REGS_SOFTMAX) : "memory");
    // ------------------------------------------------------------ softmax
    const int wg = (warp - 4) / 4;     // query tile owned by this warpgroup
    const int quarter = warp % 4;      // TMEM lanes [32*quarter, 32*quarter + 32)
    const int row = quarter * 32 + lane;
    const uint32_t lane_bits = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_bits + wg * 128;
    const uint32_t tO = tmem + lane_bits + 256 + wg * 128;
    // this row of P in shared memory: 128 bytes, 16-byte chunks swizzled by row % 8
    uint8_t* prow = smem + OFF_P + wg * TILE + row * 128;
    const int sw = row & 7;
    const float sq = deq_scale(__ldg(p.amax + bh)), sk = deq_scale(__ldg(p.amax + p.BH + bh));
    const float sl2 = sq * sk * p.scale_log2;
    float m = -INFINITY;  // running reference maximum, log2 domain
    float l = 0.f;        // running row sum of P relative to m (offset included)
    bool ok = true;
    for (int j = 0; j < kv_total; ++j) {
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(B_SFULL + wg), (uint32_t)(j & 1), G, abort_flag,
                                                  kDevTimeoutSoftmax));
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t sr[BN];
      ptx::tmem_ld4x32(tS, sr);
      float* s = reinterpret_cast<float*>(sr);
      const int seg = j / p.tps;
      const int64_t rem = p.Ns - (int64_t)(j - seg * p.tps) * BN;
      const int valid = rem < BN ? (int)rem : BN;
      if (valid < BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= valid) s[c] = -INFINITY;
      }
      float mx[43];
#pragma unroll
      for (int c = 0; c < 42; ++c) mx[c] = ptx::max3(s[3 * c], s[3 * c + 1], s[3 * c + 2]);
      mx[42] = fmaxf(s[126], s[127]);
      mx[0] = ptx::MaxTree<43>::run(mx);
      const float m_tile = mx[0] * sl2;
      const bool need = m_tile > m + RESCALE_THRESHOLD;
      const float m_new = need ? m_tile : m;
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        const float alpha = need ? ptx::ex2(m - m_new) : 1.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + cc * 32, o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          ptx::tmem_st32(tO + cc * 32, o);
        }
        ptx::tmem_wait_st();
      }
      if (need) {
        l *= ptx::ex2(m - m_new);
        m = m_new;
      }
      // P = 2^(S*scale*log2e - m + 4): packed fp32 affine step, MUFU exponential,
      // E4M3 rounding, 16 keys per 16-byte shared-memory store.
      const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
      const uint64_t offm2 = ptx::f2_pack(P_OFFSET - m, P_OFFSET - m);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int c16 = 0; c16 < BN / 16; ++c16) {
        uint32_t pk[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int col = c16 * 16 + w * 4;
          float x0, x1, x2, x3;
          ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[col], s[col + 1]), sl2x2, offm2), x0, x1);
          ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[col + 2], s[col + 3]), sl2x2, offm2), x2, x3);
          const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1), p2 = ptx::ex2(x2), p3 = ptx::ex2(x3);
          acc[w] = ptx::f2_add(acc[w], ptx::f2_add(ptx::f2_pack(p0, p1), ptx::f2_pack(p2, p3)));
          pk[w] = (uint32_t)ptx::e4m3x2(p0, p1) | ((uint32_t)ptx::e4m3x2(p2, p3) << 16);
        }
        *reinterpret_cast<uint4*>(prow + ((c16 ^ sw) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      {
        float a0, a1;
        ptx::f2_unpack(ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3])), a0, a1);
        l += a0 + a1;
      }
      // generic-proxy stores of P -> visible to the tensor core (async proxy)
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(B_PFULL + wg));
    }
    // ------------------------------------------------------------ epilogue
    if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(B_ODONE + wg), 0, G, abort_flag, kDevTimeoutEpilogue));
    if (ok) {
      ptx::tc_fence_after();
      const int qt = wg == 0 ? qt0 : qt1;
      const int tq = qt >= 0 ? qt : qt0;
      const int seg = tq / p.tps;
      const int row0 = (tq - seg * p.tps) * BM;
      const bool store = qt >= 0 && (int64_t)row0 + row < p.Ns;
      const int64_t orow = ((int64_t)seg * p.BH + bh) * p.Ns + row0 + row;
      const float sv = deq_scale(__ldg(p.amax + 2 * p.BH + bh));
      const float f = sv / l;
      __nv_bfloat16* optr = p.out + orow * HD;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + cc * 32, o);
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = ptx::bf16x2(__uint_as_float(o[2 * c]) * f, __uint_as_float(o[2 * c + 1]) * f);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(optr + cc * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (store) p.lse[orow] = (m - P_OFFSET + log2f(l)) * 0.69314718055994531f;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 8-bit 4-D map (inner, rows, BH, sp) with 128 x 128 boxes and 128-byte swizzle.
bool make_map_u8(CUtensorMap* m, const void* base, int64_t inner, int64_t rows, int64_t BH, int64_t sp) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)BH, (cuuint64_t)sp};
  cuuint64_t strides[3] = {(cuuint64_t)inner, (cuuint64_t)(inner * rows), (cuuint64_t)(inner * rows * BH)};
  cuuint32_t box[4] = {128, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attn_fp8_fwd(const Fp8AttnArgs& a, const Guard& g, cudaStream_t stream) {
  static std::atomic<unsigned long long> attr{0};
  const cudaError_t ea = smem_limit_once(attr, (const void*)attn_fp8_fwd_kernel, SMEM_BYTES);
  if (ea != cudaSuccess) return ea;
  CUtensorMap mq, mk, mvt;
  if (!make_map_u8(&mq, a.q8, HD, a.Ns, a.BH, a.sp) || !make_map_u8(&mk, a.k8, HD, a.Ns, a.BH, a.sp) ||
      !make_map_u8(&mvt, a.vt8, a.Ns_pad, HD, a.BH, a.sp))
    return cudaErrorInvalidValue;
  Fp8Params p{};
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.amax = a.amax;
  p.BH = a.BH;
  p.Ns = a.Ns;
  p.tps = (int)((a.Ns + BM - 1) / BM);
  p.tiles = (int)(p.tps * a.sp);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.guard = g;
  dim3 grid((unsigned)((p.tiles + 1) / 2), (unsigned)a.BH, 1);
  return launch_pdl(attn_fp8_fwd_kernel, grid, dim3(NUM_THREADS), SMEM_BYTES, stream, mq, mk, mvt, p);
}

}  // namespace usp
