// bf16 attention forward with log-sum-exp on the tcgen05 tensor cores (D = 128).
//
// What it computes (per (b, h), query row i; no mask, not causal):
//   S_ij = scale q_i.k_j;  lse_i = ln sum_j exp(S_ij);  out_i = sum_j exp(S_ij - lse_i) v_j
// -- the per-card attention of "Multi-GPU parallelism: spreading one step over
// several cards" (section "Sequence parallelism: Ulysses and Ring") with the
// LSE that the USP PR page ("Ring kernel selection") requires of a ring kernel.
// In fused mode the KV loop runs over every shard of the token-sharded stack,
// so the Ring step's log-sum-exp merge happens inside the online softmax.
//
// CTA organisation (one CTA per SM: ~193 KB shared memory, 512 TMEM columns):
//   warp 0        TMA producer: Q0, Q1 once, then K_j / V_j through a 2-stage ring
//   warp 1        TMEM allocator and single-thread tcgen05.mma issuer
//   warps 4..7    softmax for query tile 0 (thread = one query row = one TMEM lane)
//   warps 8..11   softmax for query tile 1
// TMEM columns: S0 [0,128)  S1 [128,256)  O0 [256,384)  O1 [384,512).  P_i is
// written as packed bf16 over the first 64 columns of S_i and consumed from
// TMEM as the A operand of O_i += P_i V_j.
// MMA issue order per KV tile j: PV0(j-1), S0(j), PV1(j-1), S1(j), so while one
// softmax warpgroup works on its S tile the tensor core runs the other tile's
// GEMMs (two query tiles in ping-pong).
// Online softmax in the log2 domain with ex2.approx; the running maximum is
// only moved (and O rescaled) when it grows by more than 8 (a factor 256), which
// is exact because O and the row sum always share the same reference maximum.
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
constexpr int KV_STAGES = 2;
constexpr int TILE_BYTES = BM * HD * 2;   // one 128 x 128 bf16 tile
constexpr int HALF_BYTES = TILE_BYTES / 2;  // 64-column half (128-byte rows, 128B swizzle)
constexpr int NUM_THREADS = 384;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
#ifndef USP_REGS_CTRL
#define USP_REGS_CTRL 56
#endif
constexpr int REGS_CTRL = USP_REGS_CTRL;
constexpr int REGS_SOFTMAX = (NUM_THREADS * 168 - 128 * REGS_CTRL) / 256 / 8 * 8;
static_assert(128 * REGS_CTRL + 256 * REGS_SOFTMAX <= NUM_THREADS * 168, "register split exceeds the launch");

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
constexpr int OFF_V = OFF_K + KV_STAGES * TILE_BYTES;
constexpr int OFF_BAR = OFF_V + KV_STAGES * TILE_BYTES;
// barrier slots (8 bytes each)
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

struct TcParams {
  void* out;
  float* lse;
  int64_t Nq, Nk;           // rows per head (plain addressing)
  RingSchedule sched;
  int64_t out_step_stride;  // heads between ring steps in out / lse
  int fused;
  int64_t BH, Ns;           // fused addressing
  int q_tiles;              // query tiles per unit
  int kv_tiles;             // KV tiles per unit
  int tiles_per_seg;        // fused: tiles per shard
  float scale_log2;         // scale * log2(e)
  Guard guard;
};

struct Unit {
  int64_t qh, kvh, oh;
};

__device__ __forceinline__ Unit unit_heads(const TcParams& p, int64_t unit) {
  Unit u;
  if (p.fused) {
    u.qh = u.kvh = u.oh = unit;
    return u;
  }
  const RingSchedule& s = p.sched;
  const int64_t per_step = (int64_t)s.ring * s.ulysses * s.heads_per_rank;
  const int64_t t = unit / per_step;
  const int64_t qh = unit - t * per_step;
  const int64_t rank_heads = (int64_t)s.heads_per_rank * s.ulysses;  // heads per ring group
  const int64_t g = qh / rank_heads;
  const int64_t c = ((g - t) % s.ring + s.ring) % s.ring;             // KV chunk at ring step t
  u.qh = qh;
  u.kvh = qh + (c - g) * rank_heads;
  u.oh = t * p.out_step_stride + qh;
  return u;
}

// A tile of a head: its first row inside its shard (or head), the shard, and
// how many of its 128 rows exist.
struct TileRef {
  int row0;
  int seg;
  int valid;
};
__device__ __forceinline__ TileRef tile_ref(const TcParams& p, int tile, bool is_q) {
  TileRef t;
  if (p.fused) {
    t.seg = tile / p.tiles_per_seg;
    t.row0 = (tile - t.seg * p.tiles_per_seg) * BM;
    const int64_t rem = p.Ns - t.row0;
    t.valid = rem < BM ? (int)rem : BM;
  } else {
    t.seg = 0;
    t.row0 = tile * BM;
    const int64_t rem = (is_q ? p.Nq : p.Nk) - t.row0;
    t.valid = rem < BM ? (int)rem : BM;
  }
  return t;
}

__device__ __forceinline__ void load_tile(const CUtensorMap* map, const TcParams& p, uint32_t dst,
                                          uint32_t bar, int64_t head, const TileRef& t) {
  if (p.fused) {
    ptx::tma_load_4d(dst, map, bar, 0, t.row0, (int)head, t.seg);
    ptx::tma_load_4d(dst + HALF_BYTES, map, bar, 64, t.row0, (int)head, t.seg);
  } else {
    ptx::tma_load_3d(dst, map, bar, 0, t.row0, (int)head);
    ptx::tma_load_3d(dst + HALF_BYTES, map, bar, 64, t.row0, (int)head);
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_SLOT);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int64_t unit = blockIdx.y;
  const Unit U = unit_heads(p, unit);
  const int qt0 = 2 * blockIdx.x;
  const int qt1 = (qt0 + 1 < p.q_tiles) ? qt0 + 1 : -1;  // -1: no second tile (compute on a copy)

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
    ptx::prefetch_tmap(&tm_v);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Guard& G = p.guard;
  // Register split: the producer/MMA warpgroup hands registers to the two
  // softmax warpgroups (128*REGS_CTRL + 256*REGS_SOFTMAX = 384*168, the
  // allocation the CTA was launched with).
  // Each role's code sits inside the branch that set its register budget, so
  // the compiler allocates every region against the right limit.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(REGS_CTRL) : "memory");
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const TileRef q0 = tile_ref(p, qt0, true);
      const TileRef q1 = tile_ref(p, qt1 >= 0 ? qt1 : qt0, true);
      ptx::mbar_arrive_expect_tx(bar(B_QFULL), 2 * TILE_BYTES);
      load_tile(&tm_q, p, sbase + OFF_Q, bar(B_QFULL), U.qh, q0);
      load_tile(&tm_q, p, sbase + OFF_Q + TILE_BYTES, bar(B_QFULL), U.qh, q1);
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < p.kv_tiles; ++j) {
        const int s = j % KV_STAGES;
        const uint32_t ph = (uint32_t)((j / KV_STAGES) & 1);
        const TileRef kt = tile_ref(p, j, false);
        if (!ptx::mbar_wait(bar(B_KEMPTY + s), ph ^ 1u, G, abort_flag, kDevTimeoutTmaProducer)) break;
        ptx::mbar_arrive_expect_tx(bar(B_KFULL + s), TILE_BYTES);
        load_tile(&tm_k, p, sbase + OFF_K + s * TILE_BYTES, bar(B_KFULL + s), U.kvh, kt);
        issued_k = j + 1;
        if (!ptx::mbar_wait(bar(B_VEMPTY + s), ph ^ 1u, G, abort_flag, kDevTimeoutTmaProducer)) break;
        ptx::mbar_arrive_expect_tx(bar(B_VFULL + s), TILE_BYTES);
        load_tile(&tm_v, p, sbase + OFF_V + s * TILE_BYTES, bar(B_VFULL + s), U.kvh, kt);
        issued_v = j + 1;
      }
      // Drain: every copy this thread issued must land before shared memory is released.
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
      constexpr uint32_t IDESC_QK = ptx::idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(BM, HD, 0, 1);  // P from TMEM, V MN-major
      const uint32_t tS[2] = {tmem, tmem + 128};
      const uint32_t tO[2] = {tmem + 256, tmem + 384};
      const uint32_t sQ[2] = {sbase + OFF_Q, sbase + OFF_Q + TILE_BYTES};
      bool ok = ptx::mbar_wait(bar(B_QFULL), 0, G, abort_flag, kDevTimeoutMma);
      // Descriptors are built once; per-MMA start addresses are added to the
      // low (address >> 4) field, which cannot carry out of its 14 bits since
      // shared memory ends below 256 KB.
      const uint64_t dV0 = ptx::smem_desc_sw128(sbase + OFF_V, HALF_BYTES, 1024);
      const uint64_t dK0 = ptx::smem_desc_sw128(sbase + OFF_K, 16, 1024);
      const uint64_t dQ0 = ptx::smem_desc_sw128(sQ[0], 16, 1024);
      auto issue_pv = [&](int i, int jv) {
        const uint64_t dv = ptx::launder(dV0 + (uint64_t)(((jv % KV_STAGES) * TILE_BYTES) >> 4));
        const uint32_t ts = ptx::launder(tS[i]);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // B = V tile viewed as [K = keys][N = D]: N-contiguous 128-byte rows,
          // 8-row groups 1024 B apart (SBO), the two 64-column halves 16 KB apart (LBO).
          ptx::mma_ts(tO[i], ts + kk * 8, dv + (uint64_t)((kk * 16 * 128) >> 4), IDESC_PV,
                      (jv > 0 || kk > 0) ? 1u : 0u);
        }
      };
      auto issue_s = [&](int i, int jk) {
        const uint64_t dk = ptx::launder(dK0 + (uint64_t)(((jk % KV_STAGES) * TILE_BYTES) >> 4));
        const uint64_t dq = ptx::launder(dQ0 + (uint64_t)((i * TILE_BYTES) >> 4));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t off = (uint64_t)((((kk / 4) * HALF_BYTES) + (kk % 4) * 32) >> 4);
          ptx::mma_ss(tS[i], dq + off, dk + off, IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      for (int j = 0; ok && j < p.kv_tiles; ++j) {
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
        const int jl = p.kv_tiles - 1;
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
      // Drain: all MMAs this thread issued complete before TMEM is released.
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
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running reference maximum, log2 domain
    float l = 0.f;        // running row sum relative to m
    bool ok = true;
    for (int j = 0; j < p.kv_tiles; ++j) {
      // every lane waits; the decision is made warp-uniform before the
      // warp-collective TMEM accesses below
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(B_SFULL + wg), (uint32_t)(j & 1), G, abort_flag,
                                                  kDevTimeoutSoftmax));
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t sr[BN];
      ptx::tmem_ld4x32(tS, sr);
      float* s = reinterpret_cast<float*>(sr);
      const int valid = tile_ref(p, j, false).valid;
      if (valid < BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= valid) s[c] = -INFINITY;
      }
      // row maximum: a tree of 3-input max (64 instructions, depth 5)
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
      // P = exp2(S*scale*log2e - m): the affine step on packed fp32 pairs, the
      // exponential on the MUFU, bf16 packing, 32 columns per TMEM store.
      const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
      const uint64_t negm2 = ptx::f2_pack(-m, -m);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int col = q4 * 32 + 2 * c;
          float x0, x1;
          ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[col], s[col + 1]), sl2x2, negm2), x0, x1);
          const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
          acc[c & 3] = ptx::f2_add(acc[c & 3], ptx::f2_pack(p0, p1));
          pk[c] = ptx::bf16x2(p0, p1);
        }
        ptx::tmem_st16(tS + q4 * 16, pk);
      }
      {
        float a0, a1;
        ptx::f2_unpack(ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3])), a0, a1);
        l += a0 + a1;
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(B_PFULL + wg));
    }
    // ------------------------------------------------------------ epilogue
    if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(B_ODONE + wg), 0, G, abort_flag, kDevTimeoutEpilogue));
    if (ok) {
      ptx::tc_fence_after();
      const int qt = wg == 0 ? qt0 : qt1;
      const TileRef t = tile_ref(p, qt >= 0 ? qt : qt0, true);
      const bool store = qt >= 0 && row < t.valid;
      int64_t orow;
      if (p.fused)
        orow = ((int64_t)t.seg * p.BH + U.oh) * p.Ns + t.row0 + row;
      else
        orow = U.oh * p.Nq + t.row0 + row;
      const float inv_l = 1.f / l;
      __nv_bfloat16* optr = reinterpret_cast<__nv_bfloat16*>(p.out) + orow * HD;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + cc * 32, o);
        ptx::tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack_bf16(__uint_as_float(o[2 * c]) * inv_l, __uint_as_float(o[2 * c + 1]) * inv_l);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(optr + cc * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (store) p.lse[orow] = (m + log2f(l)) * 0.69314718055994531f;
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

// bf16 [heads][rows][128] with boxes of 64 columns x 128 rows, 128-byte swizzle.
bool make_map_3d(CUtensorMap* m, const void* base, int64_t rows, int64_t heads) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)rows, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)rows * HD * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)BM, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// bf16 token-sharded stack [sp][BH][Ns][128].
bool make_map_4d(CUtensorMap* m, const void* base, int64_t Ns, int64_t BH, int64_t sp) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)HD, (cuuint64_t)Ns, (cuuint64_t)BH, (cuuint64_t)sp};
  cuuint64_t strides[3] = {(cuuint64_t)HD * 2, (cuuint64_t)Ns * HD * 2, (cuuint64_t)BH * Ns * HD * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)BM, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attn_tc_fwd(const TcAttnArgs& a, const Guard& g, cudaStream_t stream) {
  static bool attr_set = false;  // per process; the attribute is per function, not per device
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  TcParams p{};
  p.out = a.out;
  p.lse = a.lse;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.guard = g;
  CUtensorMap mq, mk, mv;
  int64_t units;
  if (a.fused) {
    const int tps = (int)((a.Ns + BM - 1) / BM);
    p.fused = 1;
    p.BH = a.BH;
    p.Ns = a.Ns;
    p.tiles_per_seg = tps;
    p.q_tiles = (int)(tps * a.sp);
    p.kv_tiles = (int)(tps * a.sp);
    p.Nq = p.Nk = a.sp * a.Ns;
    units = a.BH;
    if (!make_map_4d(&mq, a.q, a.Ns, a.BH, a.sp) || !make_map_4d(&mk, a.k, a.Ns, a.BH, a.sp) ||
        !make_map_4d(&mv, a.v, a.Ns, a.BH, a.sp))
      return cudaErrorInvalidValue;
  } else {
    p.fused = 0;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.sched = a.sched;
    p.out_step_stride = a.out_step_stride_heads;
    p.tiles_per_seg = 0;
    p.q_tiles = (int)((a.Nq + BM - 1) / BM);
    p.kv_tiles = (int)((a.Nk + BN - 1) / BN);
    const int64_t per_step = (int64_t)a.sched.ring * a.sched.ulysses * a.sched.heads_per_rank;
    units = (int64_t)a.sched.steps * per_step;
    const int64_t kv_heads = per_step;  // the KV stack holds one step's worth of heads
    if (!make_map_3d(&mq, a.q, a.Nq, per_step) || !make_map_3d(&mk, a.k, a.Nk, kv_heads) ||
        !make_map_3d(&mv, a.v, a.Nk, kv_heads))
      return cudaErrorInvalidValue;
  }
  dim3 grid((unsigned)((p.q_tiles + 1) / 2), (unsigned)units, 1);
  attn_tc_fwd_kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace usp
