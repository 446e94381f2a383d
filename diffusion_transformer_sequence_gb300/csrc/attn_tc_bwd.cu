// bf16 USP attention backward on the tcgen05 tensor cores (D = 128).
//
// What it computes ("Feat: USP sequence parallelism (Ulysses x Ring) via
// SequenceParallelPlan; Wan enabled", Numerics and "Ring kernel selection":
// the forward returns the LSE and pairs with a real backward; every ring step
// uses its own KV chunk and the MERGED LSE).  With P = exp(scale q k^T - lse):
//   Delta_i = sum_d dO_id O_id,  dP = dO V^T,  dS = P * (dP - Delta),
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K.
// The kernels read the token-sharded stacks [sp][B*H][Ns][D] in place through
// 4-D tensor maps (the same addressing as the fused forward), so the Ulysses
// re-layout and the ring rotation are addressing, and each KV chunk's dK/dV
// accumulates over every query shard -- every (rank, ring step) pair -- inside
// one CTA, in a fixed order.  No atomics: the gradients are bitwise
// reproducible run to run.
//
//   usp_bwd_prep_kernel   Delta = rowsum(dO * O) and L2 = lse * log2(e), fp32
//   usp_bwd_dkdv_kernel   one CTA per (head, 128-key tile); loops over every
//                         128-query tile: S^T = K Q^T, dP^T = V dO^T (TMEM),
//                         P^T, dS^T in registers -> bf16 back into TMEM,
//                         dV += P^T dO, dK += dS^T Q (TMEM accumulators)
//   usp_bwd_dq_kernel     one CTA per (head, 128-query tile); loops over every
//                         128-key tile: S = Q K^T, dP = dO V^T, dS -> TMEM,
//                         dQ += dS K
// Roles (384 threads): warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer,
// warps 4..11 two elementwise warpgroups splitting the columns of each tile.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "usp_internal.cuh"

namespace usp {
namespace {

constexpr int BM = 128;
constexpr int HD = 128;
constexpr int TILE_BYTES = BM * HD * 2;
constexpr int HALF_BYTES = TILE_BYTES / 2;
constexpr int VEC_BYTES = BM * 4;  // 128 fp32 (L2 or Delta of one tile)
constexpr int NUM_THREADS = 384;
constexpr int REGS_CTRL = 56;
constexpr int REGS_ELEM = (NUM_THREADS * 168 - 128 * REGS_CTRL) / 256 / 8 * 8;
constexpr float LOG2E = 1.4426950408889634f;

struct BwdParams {
  void* dst0;          // dkdv: dK   | dq: dQ
  void* dst1;          // dkdv: dV   | dq: unused
  const float* l2;     // lse * log2(e), [sp][BH][Ns]
  const float* delta;  // rowsum(dO * O), [sp][BH][Ns]
  int64_t BH, Ns;      // heads and rows per segment of the tensor maps
  int64_t Ns_pad;      // row pitch of l2 / delta (Ns rounded up to 4: 16-byte rows for TMA)
  int tiles_per_seg;
  int tiles;           // tiles per unit (segments of the unit * tiles_per_seg)
  int useg;            // segment stride: the unit's k-th segment is k * useg + j (j = unit / BH)
  float scale, scale_log2;
  Guard guard;
};

struct TileRef {
  int row0, seg, valid;
};
// Tile `tile` of the unit whose segment offset is j: the token-sharded stack
// (useg = 1, j = 0) has every segment (virtual rank) of head bh; the
// head-sharded stack of the materialised path (segments g*u + j, u = useg)
// has the ring chunks g of Ulysses group j.
__device__ __forceinline__ TileRef tile_ref(const BwdParams& p, int tile, int j) {
  TileRef t;
  const int k = tile / p.tiles_per_seg;
  t.seg = k * p.useg + j;
  t.row0 = (tile - k * p.tiles_per_seg) * BM;
  const int64_t rem = p.Ns - t.row0;
  t.valid = rem < BM ? (int)rem : BM;
  return t;
}
__device__ __forceinline__ void load_tile(const CUtensorMap* map, uint32_t dst, uint32_t bar, int64_t bh,
                                          const TileRef& t) {
  ptx::tma_load_4d(dst, map, bar, 0, t.row0, (int)bh, t.seg);
  ptx::tma_load_4d(dst + HALF_BYTES, map, bar, 64, t.row0, (int)bh, t.seg);
}
__device__ __forceinline__ int64_t row_index(const BwdParams& p, int64_t bh, const TileRef& t, int r) {
  return ((int64_t)t.seg * p.BH + bh) * p.Ns + t.row0 + r;
}
__device__ __forceinline__ int64_t vec_index(const BwdParams& p, int64_t bh, const TileRef& t, int r) {
  return ((int64_t)t.seg * p.BH + bh) * p.Ns_pad + t.row0 + r;
}

// Shared memory: two resident 128-row tiles A0, A1 (K and V for dK/dV, Q and
// dO for dQ); then the dK/dV kernel's STAGES x (two streamed 128-row tiles +
// two fp32 vectors) and barriers (the dQ kernel's K and V rings are laid out
// with it, below).  Every GEMM is a 128 x 128 (x 128 or 64)
// tcgen05.mma: a narrower N costs nearly the same time per 16-deep step
// (69 against 65 clocks measured at N = 64 and 128), so it halves the rate.
constexpr int STAGES = 2;
constexpr int OFF_A0 = 0;
constexpr int OFF_A1 = TILE_BYTES;
constexpr int OFF_STAGE = 2 * TILE_BYTES;
constexpr int STAGE_BYTES = 2 * TILE_BYTES + 2 * VEC_BYTES;
constexpr int OFF_BAR = OFF_STAGE + STAGES * STAGE_BYTES;
enum Bar : int {  // the dK/dV kernel's barriers
  B_RES = 0,                    // resident K and V landed
  B_FULL = 1,                   // + stage: a query tile's Q, dO, L2, Delta landed
  B_EMPTY = B_FULL + STAGES,    // + stage: the tile's last GEMM (dK) done, stage free
  B_SFULL = B_EMPTY + STAGES,   // S^T GEMM done
  B_DPFULL,                     // dP^T GEMM done
  B_PREADY,                     // first half of P^T written to TMEM (256 arrivals)
  B_PREADY2,                    // second half of P^T written (256)
  B_DSREADY,                    // dS^T written to TMEM (256)
  B_ODONE,                      // the last dV and dK GEMMs done
  B_MMADONE,                    // every MMA of the CTA done (drain before TMEM is released)
  NUM_BARS
};
constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_SLOT + 8;
constexpr int SMEM_BYTES = OFF_ABORT + 8 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t stage_addr(uint32_t sbase, int s) { return sbase + OFF_STAGE + s * STAGE_BYTES; }

// dK/dV prologue: barriers and TMEM.  Returns the TMEM base.
__device__ __forceinline__ uint32_t prologue(uint8_t* smem, uint32_t sbase, int warp) {
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8 * i; };
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(B_RES), 1);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar(B_FULL + s), 1);
      ptx::mbar_init(bar(B_EMPTY + s), 1);
    }
    ptx::mbar_init(bar(B_SFULL), 1);
    ptx::mbar_init(bar(B_DPFULL), 1);
    ptx::mbar_init(bar(B_PREADY), 256);
    ptx::mbar_init(bar(B_PREADY2), 256);
    ptx::mbar_init(bar(B_DSREADY), 256);
    ptx::mbar_init(bar(B_ODONE), 1);
    ptx::mbar_init(bar(B_MMADONE), 1);
    *reinterpret_cast<volatile int*>(smem + OFF_ABORT) = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + OFF_SLOT, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  return *reinterpret_cast<uint32_t*>(smem + OFF_SLOT);
}

__device__ __forceinline__ void teardown(uint32_t tmem, int warp) {
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Store 64 fp32 columns of one row (times `mul`) as bf16 to global.  Every
// lane of the warp runs the (warp-collective) TMEM loads; only lanes with
// `store` set write.
__device__ __forceinline__ void store_row64(__nv_bfloat16* dst, uint32_t taddr, float mul, bool store) {
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t o[32];
    ptx::tmem_ld32(taddr + cc * 32, o);
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) pk[c] = ptx::bf16x2(__uint_as_float(o[2 * c]) * mul, __uint_as_float(o[2 * c + 1]) * mul);
    if (store) {
      uint4* d = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v) d[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
  }
}

// K-major operand descriptor of k-step kk (16 of the 128 head-dim columns).
__device__ __forceinline__ uint64_t kmajor_step(uint64_t d0, int kk) {
  return d0 + (uint64_t)((((kk / 4) * HALF_BYTES) + (kk % 4) * 32) >> 4);
}
// A-operand (packed bf16) column of k-step kk when warpgroup 0 wrote rows
// [0,64) at columns [0,32) and warpgroup 1 wrote [64,128) at [64,96).
__device__ __forceinline__ uint32_t packed_col(int kk) { return kk < 4 ? kk * 8 : 64 + (kk - 4) * 8; }

// Elementwise warps split every phase in two so the tensor core always has an
// independent 128-wide GEMM queued behind the one the warps are waiting for:
//   dK/dV per query tile i:  S^T(i) dP^T(i) | dV(i) S^T(i+1) | dK(i) dP^T(i+1) ...
//     the warps compute P^T(i) while dP^T(i) runs, dS^T(i) while dV(i) and
//     S^T(i+1) run.  S^T(i+1) overwrites the columns dV(i) reads P^T(i)
//     from, so it follows dV(i); the warps hand P^T over in two halves (the
//     first 32 query columns of each warpgroup, then the rest) and the first
//     half of dV(i) runs while they compute the second (1-2% faster than one
//     hand-over; quarters were slower);
//   dQ per key tile j:  S(j+1) dP(j+1) dQ(j) ...  the warps release S(j) and
//     dP(j) as soon as they have read them, write dS(j) into TMEM once dQ(j-1)
//     has read dS(j-1), and release the K and V slots (the tensor core's
//     completion of dQ(j-1) and dP(j) is what they have just waited for), so
//     the MMA issuer commits only to barriers someone waits on.
// (a thread owns one TMEM lane = one row; warpgroup w owns columns
// [64w, 64w+64) and writes its packed bf16 results inside columns it has read)

// =====================================================================
// dK, dV: one CTA per (head, 128-key tile); resident K (A0), V (A1);
// streamed Q, dO, L2, Delta per 128-query tile.
// TMEM: S^T [0,128)  dP^T [128,256)  dV [256,384)  dK [384,512).
// =====================================================================
__global__ void __launch_bounds__(NUM_THREADS, 1)
    usp_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                        const __grid_constant__ CUtensorMap tm_l2, const __grid_constant__ CUtensorMap tm_dl,
                        const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int jseg = (int)(blockIdx.y / p.BH);
  const int64_t bh = blockIdx.y - (int64_t)jseg * p.BH;
  const TileRef kt = tile_ref(p, blockIdx.x, jseg);
  const Guard& G = p.guard;
  const uint32_t tmem = prologue(smem, sbase, warp);
  ptx::griddep_wait();    // the prologue above overlapped the previous kernel's tail
  ptx::griddep_launch();
  const uint32_t tSt = tmem, tdPt = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
  const int T = p.tiles;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(REGS_CTRL) : "memory");
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      ptx::mbar_arrive_expect_tx(bar(B_RES), 2 * TILE_BYTES);
      load_tile(&tm_k, sbase + OFF_A0, bar(B_RES), bh, kt);
      load_tile(&tm_v, sbase + OFF_A1, bar(B_RES), bh, kt);
      int issued = 0;
      for (int i = 0; i < T; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (uint32_t)((i / STAGES) & 1);
        if (!ptx::mbar_wait(bar(B_EMPTY + s), ph ^ 1u, G, abort_flag, kDevTimeoutTmaProducer)) break;
        const TileRef qt = tile_ref(p, i, jseg);
        const uint32_t st = stage_addr(sbase, s);
        ptx::mbar_arrive_expect_tx(bar(B_FULL + s), 2 * TILE_BYTES + 2 * VEC_BYTES);
        load_tile(&tm_q, st, bar(B_FULL + s), bh, qt);
        load_tile(&tm_do, st + TILE_BYTES, bar(B_FULL + s), bh, qt);
        ptx::tma_load_3d(st + 2 * TILE_BYTES, &tm_l2, bar(B_FULL + s), qt.row0, (int)bh, qt.seg);
        ptx::tma_load_3d(st + 2 * TILE_BYTES + VEC_BYTES, &tm_dl, bar(B_FULL + s), qt.row0, (int)bh, qt.seg);
        issued = i + 1;
      }
      ptx::mbar_drain(bar(B_RES), 0, 200000000ull);
      for (int i = issued - STAGES; i < issued; ++i)
        if (i >= 0) ptx::mbar_drain(bar(B_FULL + i % STAGES), (uint32_t)((i / STAGES) & 1), 200000000ull);
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t ID_S = ptx::idesc_bf16_f32(BM, BM, 0, 0);  // S^T, dP^T
      constexpr uint32_t ID_G = ptx::idesc_bf16_f32(BM, HD, 0, 1);  // dV, dK (B = dO / Q, N-major)
      const uint64_t dK0 = ptx::smem_desc_sw128(sbase + OFF_A0, 16, 1024);
      const uint64_t dV0 = ptx::smem_desc_sw128(sbase + OFF_A1, 16, 1024);
      auto wait = [&](int b, uint32_t ph) { return ptx::mbar_wait(bar(b), ph, G, abort_flag, kDevTimeoutMma); };
      auto issue_st = [&](int i) -> bool {  // S^T(i) = K Q_i^T
        const int s = i % STAGES;
        if (!wait(B_FULL + s, (uint32_t)((i / STAGES) & 1))) return false;
        ptx::tc_fence_after();
        const uint64_t dq = ptx::launder(ptx::smem_desc_sw128(stage_addr(sbase, s), 16, 1024));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          ptx::mma_ss(tSt, kmajor_step(dK0, kk), kmajor_step(dq, kk), ID_S, kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar(B_SFULL));
        return true;
      };
      auto issue_dpt = [&](int i) {  // dP^T(i) = V dO_i^T (stage already waited for by S^T(i))
        const uint64_t ddo = ptx::launder(ptx::smem_desc_sw128(stage_addr(sbase, i % STAGES) + TILE_BYTES, 16, 1024));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          ptx::mma_ss(tdPt, kmajor_step(dV0, kk), kmajor_step(ddo, kk), ID_S, kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar(B_DPFULL));
      };
      bool ok = wait(B_RES, 0);
      if (ok) ok = issue_st(0);
      if (ok) issue_dpt(0);
      for (int i = 0; ok && i < T; ++i) {
        const uint32_t st = stage_addr(sbase, i % STAGES);
        const uint64_t bdo = ptx::launder(ptx::smem_desc_sw128(st + TILE_BYTES, HALF_BYTES, 1024));
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // dV += P^T dO (K = queries), in the halves the warps hand over
          if (!(ok = wait(h == 0 ? B_PREADY : B_PREADY2, (uint32_t)(i & 1)))) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // k-steps 2h, 2h+1 (warpgroup 0) and 4+2h, 5+2h (warpgroup 1)
            const int kk = (q & 1) + 2 * h + 4 * (q >> 1);
            ptx::mma_ts(tdV, tSt + packed_col(kk), bdo + (uint64_t)((kk * 2048) >> 4), ID_G,
                        (i > 0 || h > 0 || q > 0) ? 1u : 0u);
          }
        }
        if (!ok) break;
        if (i + 1 < T && !(ok = issue_st(i + 1))) break;
        if (!(ok = wait(B_DSREADY, (uint32_t)(i & 1)))) break;
        ptx::tc_fence_after();
        const uint64_t bq = ptx::launder(ptx::smem_desc_sw128(st, HALF_BYTES, 1024));
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)  // dK += dS^T Q
          ptx::mma_ts(tdK, tdPt + packed_col(kk), bq + (uint64_t)((kk * 2048) >> 4), ID_G, (i > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(bar(B_EMPTY + i % STAGES));
        if (i + 1 < T) issue_dpt(i + 1);
      }
      if (ok) ptx::mma_commit(bar(B_ODONE));
      ptx::mma_commit(bar(B_MMADONE));
      ptx::mbar_drain(bar(B_MMADONE), 0, 200000000ull);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(REGS_ELEM) : "memory");
    // ------------------------------------------------------------ elementwise
    const int wg = (warp - 4) / 4;
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;  // key row of this thread
    const uint32_t lane_bits = (uint32_t)(quarter * 32) << 16;
    const int c0 = wg * 64;               // query columns of this warpgroup
    const uint64_t sl2x2 = ptx::f2_pack(p.scale_log2, p.scale_log2);
    auto wait = [&](int b, uint32_t ph) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar(b), ph, G, abort_flag, kDevTimeoutSoftmax));
    };
    bool ok = true;
    for (int i = 0; i < T; ++i) {
      if (!(ok = wait(B_SFULL, (uint32_t)(i & 1)))) break;
      ptx::tc_fence_after();
      const uint32_t st = stage_addr(sbase, i % STAGES);
      const float* l2 = reinterpret_cast<const float*>(smem + (st - sbase) + 2 * TILE_BYTES) + c0;
      const float* dl = reinterpret_cast<const float*>(smem + (st - sbase) + 2 * TILE_BYTES + VEC_BYTES) + c0;
      uint32_t r[64];
      ptx::tmem_ld64(tSt + lane_bits + c0, r);
      float pv[64];
      uint32_t pk[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // P^T in two halves of 32 query columns (16 packed TMEM columns)
#pragma unroll
        for (int c = 16 * h; c < 16 * h + 16; ++c) {
          const float2 lv = *reinterpret_cast<const float2*>(l2 + 2 * c);
          float x0, x1;
          ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])), sl2x2,
                                     ptx::f2_pack(-lv.x, -lv.y)),
                         x0, x1);
          pv[2 * c] = ptx::ex2(x0);
          pv[2 * c + 1] = ptx::ex2(x1);
          pk[c] = ptx::bf16x2(pv[2 * c], pv[2 * c + 1]);
        }
        ptx::tmem_st16(tSt + lane_bits + c0 + 16 * h, pk + 16 * h);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(h == 0 ? B_PREADY : B_PREADY2));
      }
      if (!(ok = wait(B_DPFULL, (uint32_t)(i & 1)))) break;
      ptx::tc_fence_after();
      ptx::tmem_ld64(tdPt + lane_bits + c0, r);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float2 dv = *reinterpret_cast<const float2*>(dl + 2 * c);
        float y0, y1, d0, d1;
        ptx::f2_unpack(ptx::f2_add(ptx::f2_pack(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])),
                                   ptx::f2_pack(-dv.x, -dv.y)),
                       y0, y1);
        ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(pv[2 * c], pv[2 * c + 1]), ptx::f2_pack(y0, y1)), d0, d1);
        pk[c] = ptx::bf16x2(d0, d1);
      }
      ptx::tmem_st32(tdPt + lane_bits + c0, pk);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(B_DSREADY));
    }
    // ------------------------------------------------------------ epilogue
    if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(B_ODONE), 0, G, abort_flag, kDevTimeoutEpilogue));
    if (ok) {
      ptx::tc_fence_after();
      const bool store = row < kt.valid;
      const int64_t rr = row_index(p, bh, kt, store ? row : 0);
      store_row64(reinterpret_cast<__nv_bfloat16*>(p.dst1) + rr * HD + c0, tdV + lane_bits + c0, 1.f, store);
      store_row64(reinterpret_cast<__nv_bfloat16*>(p.dst0) + rr * HD + c0, tdK + lane_bits + c0, p.scale, store);
    }
  }
  teardown(tmem, warp);
}

// =====================================================================
// dQ: one CTA per (head, 128-query tile); resident Q (A0), dO (A1);
// streamed K through a 3-slot ring and V through a 2-slot ring (a K tile is
// read by S(j) and, late, by dQ(j); a V tile only by dP(j), so the two are
// released at different times and K needs the deeper ring to keep the next
// loads in flight).  Q is also copied once into TMEM (bf16 pairs), so
// S = Q K^T reads only K from shared memory (one shared-memory operand fewer
// per tile; the backward measured 2.4-2.6% faster with it).
// TMEM: S [0,128)  dP [128,256)  dQ [256,384)  dS [384,448)  Q [448,512).
// =====================================================================
constexpr int KSLOTS = 3, VSLOTS = 2;
constexpr int DQ_OFF_K = 2 * TILE_BYTES;
constexpr int DQ_OFF_V = DQ_OFF_K + KSLOTS * TILE_BYTES;
constexpr int DQ_OFF_BAR = DQ_OFF_V + VSLOTS * TILE_BYTES;
enum DqBar : int {
  Q_RES = 0,                // resident Q and dO landed
  Q_KFULL = 1,              // + slot: a K tile landed
  Q_KEMPTY = Q_KFULL + KSLOTS,  // + slot: free (one elementwise thread, after it saw dQ(j) done)
  Q_VFULL = Q_KEMPTY + KSLOTS,  // + slot: a V tile landed
  Q_VEMPTY = Q_VFULL + VSLOTS,  // + slot: free (one elementwise thread, after it saw dP(j) done)
  Q_SFULL = Q_VEMPTY + VSLOTS,  // S GEMM done
  Q_DPFULL,                 // dP GEMM done
  Q_SFREE,                  // S(j) read by the warps (256 arrivals)
  Q_DPFREE,                 // dP(j) read (256)
  Q_DSREADY,                // dS(j) written (256)
  Q_DQDONE,                 // dQ GEMM of tile j (which read dS(j)) done
  Q_QTMEM,                  // Q copied into TMEM (256)
  Q_ODONE,
  Q_MMADONE,
  Q_NUM_BARS
};
constexpr int DQ_OFF_SLOT = DQ_OFF_BAR + Q_NUM_BARS * 8;
constexpr int DQ_OFF_ABORT = DQ_OFF_SLOT + 8;
constexpr int DQ_SMEM_BYTES = DQ_OFF_ABORT + 8 + 1024;
static_assert(DQ_SMEM_BYTES <= 232448, "shared memory budget");

__global__ void __launch_bounds__(NUM_THREADS, 1)
    usp_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + DQ_OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + DQ_OFF_ABORT);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int jseg = (int)(blockIdx.y / p.BH);
  const int64_t bh = blockIdx.y - (int64_t)jseg * p.BH;
  const TileRef qt = tile_ref(p, blockIdx.x, jseg);
  const Guard& G = p.guard;
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(Q_RES), 1);
    for (int s = 0; s < KSLOTS; ++s) {
      ptx::mbar_init(bar(Q_KFULL + s), 1);
      ptx::mbar_init(bar(Q_KEMPTY + s), 1);
    }
    for (int s = 0; s < VSLOTS; ++s) {
      ptx::mbar_init(bar(Q_VFULL + s), 1);
      ptx::mbar_init(bar(Q_VEMPTY + s), 1);
    }
    ptx::mbar_init(bar(Q_SFULL), 1);
    ptx::mbar_init(bar(Q_DPFULL), 1);
    ptx::mbar_init(bar(Q_SFREE), 256);
    ptx::mbar_init(bar(Q_DPFREE), 256);
    ptx::mbar_init(bar(Q_DSREADY), 256);
    ptx::mbar_init(bar(Q_DQDONE), 1);
    ptx::mbar_init(bar(Q_QTMEM), 256);
    ptx::mbar_init(bar(Q_ODONE), 1);
    ptx::mbar_init(bar(Q_MMADONE), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + DQ_OFF_SLOT, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<uint32_t*>(smem + DQ_OFF_SLOT);
  const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256, tdS = tmem + 384, tQ = tmem + 448;
  const int T = p.tiles;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(REGS_CTRL) : "memory");
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      ptx::mbar_arrive_expect_tx(bar(Q_RES), 2 * TILE_BYTES);
      load_tile(&tm_q, sbase + OFF_A0, bar(Q_RES), bh, qt);
      load_tile(&tm_do, sbase + OFF_A1, bar(Q_RES), bh, qt);
      int issued_k = 0, issued_v = 0;
      // K runs ahead of V by up to one slot: issue in the order the MMAs consume
      for (int j = 0; j < T; ++j) {
        const TileRef kt = tile_ref(p, j, jseg);
        const int sk = j % KSLOTS, sv = j % VSLOTS;
        if (!ptx::mbar_wait(bar(Q_KEMPTY + sk), (uint32_t)(((j / KSLOTS) & 1) ^ 1), G, abort_flag,
                            kDevTimeoutTmaProducer))
          break;
        ptx::mbar_arrive_expect_tx(bar(Q_KFULL + sk), TILE_BYTES);
        load_tile(&tm_k, sbase + DQ_OFF_K + sk * TILE_BYTES, bar(Q_KFULL + sk), bh, kt);
        issued_k = j + 1;
        if (!ptx::mbar_wait(bar(Q_VEMPTY + sv), (uint32_t)(((j / VSLOTS) & 1) ^ 1), G, abort_flag,
                            kDevTimeoutTmaProducer))
          break;
        ptx::mbar_arrive_expect_tx(bar(Q_VFULL + sv), TILE_BYTES);
        load_tile(&tm_v, sbase + DQ_OFF_V + sv * TILE_BYTES, bar(Q_VFULL + sv), bh, kt);
        issued_v = j + 1;
      }
      ptx::mbar_drain(bar(Q_RES), 0, 200000000ull);
      for (int j = issued_k - KSLOTS; j < issued_k; ++j)
        if (j >= 0) ptx::mbar_drain(bar(Q_KFULL + j % KSLOTS), (uint32_t)((j / KSLOTS) & 1), 200000000ull);
      for (int j = issued_v - VSLOTS; j < issued_v; ++j)
        if (j >= 0) ptx::mbar_drain(bar(Q_VFULL + j % VSLOTS), (uint32_t)((j / VSLOTS) & 1), 200000000ull);
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t ID_S = ptx::idesc_bf16_f32(BM, BM, 0, 0);  // S, dP
      constexpr uint32_t ID_G = ptx::idesc_bf16_f32(BM, HD, 0, 1);  // dQ (B = K, N-major)
      const uint64_t dO0 = ptx::smem_desc_sw128(sbase + OFF_A1, 16, 1024);
      auto wait = [&](int b, uint32_t ph) { return ptx::mbar_wait(bar(b), ph, G, abort_flag, kDevTimeoutMma); };
      auto issue_s = [&](int j) -> bool {  // S(j) = Q K_j^T (A = Q in TMEM)
        const int sk = j % KSLOTS;
        if (!wait(Q_KFULL + sk, (uint32_t)((j / KSLOTS) & 1))) return false;
        ptx::tc_fence_after();
        const uint64_t dk = ptx::launder(ptx::smem_desc_sw128(sbase + DQ_OFF_K + sk * TILE_BYTES, 16, 1024));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          ptx::mma_ts(tS, tQ + kk * 8, kmajor_step(dk, kk), ID_S, kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar(Q_SFULL));
        return true;
      };
      auto issue_dp = [&](int j) -> bool {  // dP(j) = dO V_j^T
        const int sv = j % VSLOTS;
        if (!wait(Q_VFULL + sv, (uint32_t)((j / VSLOTS) & 1))) return false;
        ptx::tc_fence_after();
        const uint64_t dv = ptx::launder(ptx::smem_desc_sw128(sbase + DQ_OFF_V + sv * TILE_BYTES, 16, 1024));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          ptx::mma_ss(tdP, kmajor_step(dO0, kk), kmajor_step(dv, kk), ID_S, kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar(Q_DPFULL));  // the warps release the V slot once they see it
        return true;
      };
      bool ok = wait(Q_RES, 0);
      if (ok) ok = wait(Q_QTMEM, 0);
      if (ok) ok = issue_s(0);
      if (ok) ok = issue_dp(0);
      for (int j = 0; ok && j < T; ++j) {
        if (j + 1 < T) {
          if (!(ok = wait(Q_SFREE, (uint32_t)(j & 1)))) break;    // S(j) read by the warps
          if (!(ok = issue_s(j + 1))) break;
          if (!(ok = wait(Q_DPFREE, (uint32_t)(j & 1)))) break;   // dP(j) read by the warps
          if (!(ok = issue_dp(j + 1))) break;
        }
        if (!(ok = wait(Q_DSREADY, (uint32_t)(j & 1)))) break;
        ptx::tc_fence_after();
        const int sk = j % KSLOTS;
        const uint64_t bk = ptx::launder(ptx::smem_desc_sw128(sbase + DQ_OFF_K + sk * TILE_BYTES, HALF_BYTES, 1024));
        const uint32_t ds = ptx::launder(tdS);
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)  // dQ += dS K (K = keys)
          ptx::mma_ts(tdQ, ds + kk * 8, bk + (uint64_t)((kk * 2048) >> 4), ID_G, (j > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(bar(Q_DQDONE));  // the warps release the K slot once they see it
      }
      if (ok) ptx::mma_commit(bar(Q_ODONE));
      ptx::mma_commit(bar(Q_MMADONE));
      ptx::mbar_drain(bar(Q_MMADONE), 0, 200000000ull);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(REGS_ELEM) : "memory");
    const int wg = (warp - 4) / 4;
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;  // query row of this thread
    const uint32_t lane_bits = (uint32_t)(quarter * 32) << 16;
    const int c0 = wg * 64;               // key columns of this warpgroup
    const int64_t grow = row_index(p, bh, qt, row < qt.valid ? row : 0);
    const int64_t vrow = vec_index(p, bh, qt, row < qt.valid ? row : 0);
    const float l2 = row < qt.valid ? p.l2[vrow] : 0.f;
    const float dlt = row < qt.valid ? p.delta[vrow] : 0.f;
    const uint64_t sl2x2 = ptx::f2_pack(p.scale_log2, p.scale_log2), nl2 = ptx::f2_pack(-l2, -l2),
                   ndl = ptx::f2_pack(-dlt, -dlt);
    auto wait = [&](int b, uint32_t ph) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar(b), ph, G, abort_flag, kDevTimeoutSoftmax));
    };
    bool ok = wait(Q_RES, 0);   // Q and dO resident in shared memory
    if (ok) {
      // this warpgroup's half of the thread's Q row (head-dim columns [64 wg, 64 wg + 64)) from
      // the 128-byte-swizzled tile into TMEM as bf16 pairs: Q columns [32 wg, 32 wg + 32), the
      // layout the S GEMM reads its A operand in (column c holds elements 2c and 2c + 1)
      const uint8_t* qrow = smem + OFF_A0 + wg * HALF_BYTES + row * 128;
      uint32_t qk[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + ((c ^ (row & 7)) * 16));
        qk[4 * c] = v.x;
        qk[4 * c + 1] = v.y;
        qk[4 * c + 2] = v.z;
        qk[4 * c + 3] = v.w;
      }
      ptx::tmem_st32(tQ + lane_bits + 32 * wg, qk);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(Q_QTMEM));
    }
    for (int j = 0; ok && j < T; ++j) {
      if (!(ok = wait(Q_SFULL, (uint32_t)(j & 1)))) break;
      ptx::tc_fence_after();
      uint32_t r[64];
      ptx::tmem_ld64(tS + lane_bits + c0, r);
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(Q_SFREE));      // S(j) may now be overwritten
      const int valid = tile_ref(p, j, jseg).valid - c0;  // key columns of this warpgroup that exist
      if (valid < 64) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= valid) r[c] = __float_as_uint(-INFINITY);
      }
      float pv[64];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float x0, x1;
        ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])), sl2x2, nl2),
                       x0, x1);
        pv[2 * c] = ptx::ex2(x0);
        pv[2 * c + 1] = ptx::ex2(x1);
      }
      if (!(ok = wait(Q_DPFULL, (uint32_t)(j & 1)))) break;
      if (threadIdx.x == 128) ptx::mbar_arrive(bar(Q_VEMPTY + j % VSLOTS));  // dP(j) has read V(j)
      ptx::tc_fence_after();
      ptx::tmem_ld64(tdP + lane_bits + c0, r);
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(Q_DPFREE));     // dP(j) may now be overwritten
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float y0, y1, d0, d1;
        ptx::f2_unpack(ptx::f2_add(ptx::f2_pack(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])), ndl), y0,
                       y1);
        ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(pv[2 * c], pv[2 * c + 1]), ptx::f2_pack(y0, y1)), d0, d1);
        pk[c] = ptx::bf16x2(d0, d1);
      }
      // dS(j) overwrites dS(j-1) once the dQ GEMM of tile j - 1 has read it
      if (j >= 1 && !(ok = wait(Q_DQDONE, (uint32_t)((j - 1) & 1)))) break;
      if (j >= 1 && threadIdx.x == 128) ptx::mbar_arrive(bar(Q_KEMPTY + (j - 1) % KSLOTS));  // dQ(j-1) read K(j-1)
      ptx::tc_fence_after();
      ptx::tmem_st32(tdS + lane_bits + 32 * wg, pk);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(Q_DSREADY));
    }
    if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(Q_ODONE), 0, G, abort_flag, kDevTimeoutEpilogue));
    if (ok) {
      ptx::tc_fence_after();
      store_row64(reinterpret_cast<__nv_bfloat16*>(p.dst0) + grow * HD + c0, tdQ + lane_bits + c0, p.scale,
                  row < qt.valid);
    }
  }
  teardown(tmem, warp);
}

// =====================================================================
// Delta = rowsum(dO * O) (fp32) and L2 = lse * log2(e): 16 threads per row
// of 128 bf16, 16-byte loads, shuffle reduction over the 16 lanes.
// =====================================================================
__global__ void __launch_bounds__(256) usp_bwd_prep_kernel(const __nv_bfloat16* __restrict__ out,
                                                           const __nv_bfloat16* __restrict__ dout,
                                                           const float* __restrict__ lse, float* __restrict__ delta,
                                                           float* __restrict__ l2, int64_t rows, int64_t Ns,
                                                           int64_t Ns_pad) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = gt / 16;
  const int part = (int)(gt % 16);
  float acc = 0.f;
  if (row < rows) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(out + row * HD) + part);
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + row * HD) + part);
    const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(ha[i]), y = __bfloat1622float2(hb[i]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) {
    const int64_t v = (row / Ns) * Ns_pad + row % Ns;  // padded pitch for the tensor map
    delta[v] = acc;
    l2[v] = lse[row] * LOG2E;
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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
bool map_stack_bf16(CUtensorMap* m, const void* base, int64_t Ns, int64_t BH, int64_t sp) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)HD, (cuuint64_t)Ns, (cuuint64_t)BH, (cuuint64_t)sp};
  cuuint64_t strides[3] = {(cuuint64_t)HD * 2, (cuuint64_t)Ns * HD * 2, (cuuint64_t)BH * Ns * HD * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)BM, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// fp32 per-row vector [sp][BH][Ns] with row pitch Ns_pad; 128-row boxes.
bool map_stack_f32(CUtensorMap* m, const void* base, int64_t Ns, int64_t Ns_pad, int64_t BH, int64_t sp) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)Ns, (cuuint64_t)BH, (cuuint64_t)sp};
  cuuint64_t strides[2] = {(cuuint64_t)Ns_pad * 4, (cuuint64_t)BH * Ns_pad * 4};
  cuuint32_t box[3] = {(cuuint32_t)BM, 1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attn_tc_bwd(const TcBwdArgs& a, const Guard& g, cudaStream_t stream) {
  static std::atomic<unsigned long long> attr0{0}, attr1{0};
  cudaError_t ea = smem_limit_once(attr0, (const void*)usp_bwd_dkdv_kernel, SMEM_BYTES);
  if (ea == cudaSuccess) ea = smem_limit_once(attr1, (const void*)usp_bwd_dq_kernel, DQ_SMEM_BYTES);
  if (ea != cudaSuccess) return ea;
  const int64_t rows = a.BH * a.sp * a.Ns;
  const int64_t Ns_pad = (a.Ns + 3) / 4 * 4;
  cudaError_t e = launch_pdl(usp_bwd_prep_kernel, dim3((unsigned)((rows * 16 + 255) / 256)), dim3(256), 0, stream,
                             (const __nv_bfloat16*)a.out, (const __nv_bfloat16*)a.dout, a.lse, a.delta, a.l2, rows,
                             a.Ns, Ns_pad);
  if (e != cudaSuccess) return e;
  const int prep_mark = phase_mark(stream);
  CUtensorMap mq, mk, mv, mdo, ml2, mdl;
  if (!map_stack_bf16(&mq, a.q, a.Ns, a.BH, a.sp) || !map_stack_bf16(&mk, a.k, a.Ns, a.BH, a.sp) ||
      !map_stack_bf16(&mv, a.v, a.Ns, a.BH, a.sp) || !map_stack_bf16(&mdo, a.dout, a.Ns, a.BH, a.sp) ||
      !map_stack_f32(&ml2, a.l2, a.Ns, Ns_pad, a.BH, a.sp) || !map_stack_f32(&mdl, a.delta, a.Ns, Ns_pad, a.BH, a.sp))
    return cudaErrorInvalidValue;
  BwdParams p{};
  p.l2 = a.l2;
  p.delta = a.delta;
  p.BH = a.BH;
  p.Ns = a.Ns;
  p.Ns_pad = Ns_pad;
  p.tiles_per_seg = (int)((a.Ns + BM - 1) / BM);
  p.useg = a.useg;
  p.tiles = (int)(p.tiles_per_seg * (a.sp / a.useg));
  p.scale = a.scale;
  p.scale_log2 = a.scale * LOG2E;
  p.guard = g;
  dim3 grid((unsigned)p.tiles, (unsigned)(a.BH * a.useg), 1);
  // The two kernels are independent (each writes its own gradients): dQ runs
  // on the device's side stream, so its CTAs fill the dK/dV kernel's last,
  // partial wave instead of waiting behind it.
  cudaStream_t side = nullptr;
  e = side_begin(stream, &side);
  if (e != cudaSuccess) return e;
  BwdParams pq = p;
  p.dst0 = a.dk;
  p.dst1 = a.dv;
  e = launch_pdl(usp_bwd_dkdv_kernel, grid, dim3(NUM_THREADS), SMEM_BYTES, stream, mq, mk, mv, mdo, ml2, mdl, p);
  phase_mark(stream, prep_mark);
  pq.dst0 = a.dq;
  pq.dst1 = nullptr;
  if (e == cudaSuccess) {
    usp_bwd_dq_kernel<<<grid, NUM_THREADS, DQ_SMEM_BYTES, side>>>(mq, mk, mv, mdo, pq);
    e = cudaGetLastError();
  }
  phase_mark(side, prep_mark);
  const cudaError_t j = side_end(stream);  // always join, also after a failed launch
  return e != cudaSuccess ? e : j;
}

}  // namespace usp
