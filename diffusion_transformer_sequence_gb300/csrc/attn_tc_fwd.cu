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
// CTA organisation (one CTA per SM: ~193 KB shared memory, 512 TMEM columns;
// a launch with one query set is persistent, each CTA walking several items):
//   warp 0        TMA producer: Q0, Q1 per item, then K_j / V_j through a 2-stage ring
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
constexpr int kPersistMaxKvTiles = 32;     // longest KV loop run on a persistent grid
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
constexpr int B_QEMPTY = B_MMADONE + 1;
constexpr int NUM_BARS = B_QEMPTY + 1;
constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_SLOT + 8;
constexpr int OFF_EPI = OFF_ABORT + 8;        // EpiInfo (one-CTA-per-item launches)
constexpr int SMEM_USED = OFF_EPI + 48;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment of the base

// How the 128-row tiles of one operand are addressed.
//   kind 0: 3-D tensor map (D, rows, heads), tiles 0.. of one head
//   kind 1: 4-D tensor map over the token-sharded stack (D, Ns, B*H, sp);
//           tile t is tile (t % tps) of shard (t / tps)
struct TileSrc {
  int kind;
  int64_t rows;  // kind 0: rows per head; kind 1: Ns
  int tps;       // tiles per head (kind 0) or per shard (kind 1)
  int tiles;     // tiles in total
};

// One query set of a launch and where its results go.
struct QSide {
  TileSrc q;
  void* out;
  float* lse;
  int out_kind;             // 0: out row = oh * out_rows + row;  1: token-sharded stack
  int64_t out_rows;
  UnitMap map;
  int pairs;                // CTAs per unit (pairs of query tiles)
  int64_t ctas;             // pairs * units
};

// A launch serves one or two query sets over the same KV sources: CTAs
// [0, qs[0].ctas) the first set, the rest the second (e.g. the image and the
// text queries of joint attention), so a short second set fills the first
// one's last wave instead of running as a launch of its own.
struct TcParams {
  QSide qs[2];
  TileSrc kv, kv2;          // kv2: optional second KV source (kind 0), e.g. text tokens
  int64_t BH, Ns;           // token-sharded stack geometry
  float scale_log2;         // scale * log2(e)
  Guard guard;
};

// Where the epilogue of each query tile of the CTA writes: its first output
// row, how many rows exist, and the out / lse base pointers.  In a launch
// with one CTA per item (possibly two query sets) warp 2, idle otherwise,
// fills it before the CTA's first barrier, so the softmax warps carry none of
// the query set's parameters through the KV loop; a persistent launch has one
// query set, whose parameters sit at fixed offsets, and its softmax warps
// compute each item's addressing after the item's KV loop.
struct EpiInfo {
  int64_t orow0[2];
  void* out;
  float* lse;
  int valid[2];
};
static_assert(sizeof(EpiInfo) <= 48, "EpiInfo slot");

// A tile of a head: its first row inside its shard (or head), the shard, and
// how many of its 128 rows exist.
struct TileRef {
  int row0;
  int seg;
  int valid;
};
__device__ __forceinline__ TileRef tile_of(const TileSrc& src, int tile) {
  TileRef t;
  t.seg = src.kind == 1 ? tile / src.tps : 0;
  t.row0 = (tile - t.seg * src.tps) * BM;
  const int64_t rem = src.rows - t.row0;
  t.valid = rem < BM ? (int)rem : BM;
  return t;
}
// KV tile j of a CTA: the first source's tiles, then the second source's.
template <bool kKv2>
__device__ __forceinline__ TileRef kv_tile(const TileSrc& kv, const TileSrc& kv2, int j, bool& second) {
  second = kKv2 && j >= kv.tiles;
  return second ? tile_of(kv2, j - kv.tiles) : tile_of(kv, j);
}

__device__ __forceinline__ void load_tile(const CUtensorMap* map, int kind, uint32_t dst, uint32_t bar,
                                          int64_t head, const TileRef& t) {
  if (kind == 1) {
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

// A work item: one unit (head, or (ring step, head)) and one pair of query
// tiles of one query set.
struct Item {
  int side;
  int unit;
  int qt0, qt1;  // qt1 = -1: no second tile (computed on a copy, not stored)
};
template <bool kPersist>
__device__ __forceinline__ Item item_of(const TcParams& p, int64_t item) {
  Item it;
  it.side = (!kPersist && item >= p.qs[0].ctas) ? 1 : 0;  // persistent launches carry one query set
  const int local = (int)item - (it.side ? (int)p.qs[0].ctas : 0);  // the grid has < 2^31 items
  const int pairs = it.side ? p.qs[1].pairs : p.qs[0].pairs;
  const int q_tiles = it.side ? p.qs[1].q.tiles : p.qs[0].q.tiles;
  it.unit = local / pairs;
  it.qt0 = 2 * (local - it.unit * pairs);
  it.qt1 = (it.qt0 + 1 < q_tiles) ? it.qt0 + 1 : -1;
  return it;
}
// First output row and valid rows of query tile wg of an item.
__device__ __forceinline__ void epi_rows(const TcParams& p, const QSide& S, const Item& it, int wg, int64_t& orow0,
                                         int& valid) {
  const int64_t oh = map_unit(S.map, it.unit).oh;
  const int qt = wg == 0 ? it.qt0 : it.qt1;
  const TileRef t = tile_of(S.q, qt >= 0 ? qt : it.qt0);
  orow0 = S.out_kind == 1 ? ((int64_t)t.seg * p.BH + oh) * p.Ns + t.row0 : oh * S.out_rows + t.row0;
  valid = qt >= 0 ? t.valid : 0;
}

// kKv2: a second KV source follows the first (compiled out when absent).
// kPersist: one query set, grid of at most one CTA per SM; CTA c takes items
// c, c + gridDim.x, ...  The next item's Q load and first S GEMMs then run
// under the previous item's last P V and epilogue, and the prologue (barrier
// set-up, TMEM allocation) is paid once per SM instead of once per item.
// Otherwise the grid has one CTA per item.
template <bool kKv2, bool kPersist>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_k2, const __grid_constant__ CUtensorMap tm_v2,
                       const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_SLOT);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int64_t item_end = kPersist ? p.qs[0].ctas : (int64_t)blockIdx.x + 1;
  const int64_t item_step = kPersist ? (int64_t)gridDim.x : 1;
  const int side0 = item_of<kPersist>(p, blockIdx.x).side;  // the query set of the CTA's first item
  const int kv_total = kKv2 ? p.kv.tiles + p.kv2.tiles : p.kv.tiles;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(B_QFULL), 1);
    ptx::mbar_init(bar(B_QEMPTY), 1);
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
  if (!kPersist && warp == 2 && lane == 0) {  // an otherwise idle warp fills the epilogue's addressing
    const Item it = item_of<false>(p, blockIdx.x);
    const QSide& S = p.qs[it.side];
    EpiInfo* epi = reinterpret_cast<EpiInfo*>(smem + OFF_EPI);
    for (int i = 0; i < 2; ++i) epi_rows(p, S, it, i, epi->orow0[i], epi->valid[i]);
    epi->out = S.out;
    epi->lse = S.lse;
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + OFF_SLOT, 512);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(side0 ? &tm_q1 : &tm_q0);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    if (kKv2) {
      ptx::prefetch_tmap(&tm_k2);
      ptx::prefetch_tmap(&tm_v2);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::griddep_wait();    // the prologue above overlapped the previous kernel's tail
  ptx::griddep_launch();
  const uint32_t tmem = *tmem_slot;
  const Guard& G = p.guard;
  // Barrier phases run on across the CTA's items: the KV ring, S and P by the
  // CTA's running KV tile count g = n * kv_total + j (item n, tile j), Q and
  // O by the item count n.
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
      int issued_q = 0, issued_k = 0, issued_v = 0;
      bool ok = true;
      int n = 0;
      for (int64_t item = blockIdx.x; ok && item < item_end; item += item_step, ++n) {
        const Item it = item_of<kPersist>(p, item);
        const QSide& S = p.qs[it.side];
        const UnitHeads U = map_unit(S.map, it.unit);
        const TileRef q0 = tile_of(S.q, it.qt0);
        const TileRef q1 = tile_of(S.q, it.qt1 >= 0 ? it.qt1 : it.qt0);
        // the previous item's S GEMMs have read both Q tiles
        if (n > 0 && !(ok = ptx::mbar_wait(bar(B_QEMPTY), (uint32_t)((n - 1) & 1), G, abort_flag,
                                           kDevTimeoutTmaProducer)))
          break;
        ptx::mbar_arrive_expect_tx(bar(B_QFULL), 2 * TILE_BYTES);
        const CUtensorMap* mq = it.side ? &tm_q1 : &tm_q0;
        load_tile(mq, S.q.kind, sbase + OFF_Q, bar(B_QFULL), U.qh, q0);
        load_tile(mq, S.q.kind, sbase + OFF_Q + TILE_BYTES, bar(B_QFULL), U.qh, q1);
        issued_q = n + 1;
        for (int j = 0; j < kv_total; ++j) {
          const int g = n * kv_total + j;
          const int s = g % KV_STAGES;
          const uint32_t ph = (uint32_t)((g / KV_STAGES) & 1);
          bool second;
          const TileRef kt = kv_tile<kKv2>(p.kv, p.kv2, j, second);
          const CUtensorMap* mk = second ? &tm_k2 : &tm_k;
          const CUtensorMap* mv = second ? &tm_v2 : &tm_v;
          const int kind = second ? 0 : p.kv.kind;
          const int64_t head = second ? U.kvh2 : U.kvh;
          if (!(ok = ptx::mbar_wait(bar(B_KEMPTY + s), ph ^ 1u, G, abort_flag, kDevTimeoutTmaProducer))) break;
          ptx::mbar_arrive_expect_tx(bar(B_KFULL + s), TILE_BYTES);
          load_tile(mk, kind, sbase + OFF_K + s * TILE_BYTES, bar(B_KFULL + s), head, kt);
          issued_k = g + 1;
          if (!(ok = ptx::mbar_wait(bar(B_VEMPTY + s), ph ^ 1u, G, abort_flag, kDevTimeoutTmaProducer))) break;
          ptx::mbar_arrive_expect_tx(bar(B_VFULL + s), TILE_BYTES);
          load_tile(mv, kind, sbase + OFF_V + s * TILE_BYTES, bar(B_VFULL + s), head, kt);
          issued_v = g + 1;
        }
      }
      // Drain: every copy this thread issued must land before shared memory is released.
      const uint64_t drain_ns = 200000000ull;
      if (issued_q > 0) ptx::mbar_drain(bar(B_QFULL), (uint32_t)((issued_q - 1) & 1), drain_ns);
      for (int g = issued_k - KV_STAGES; g < issued_k; ++g)
        if (g >= 0) ptx::mbar_drain(bar(B_KFULL + g % KV_STAGES), (uint32_t)((g / KV_STAGES) & 1), drain_ns);
      for (int g = issued_v - KV_STAGES; g < issued_v; ++g)
        if (g >= 0) ptx::mbar_drain(bar(B_VFULL + g % KV_STAGES), (uint32_t)((g / KV_STAGES) & 1), drain_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = ptx::idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(BM, HD, 0, 1);  // P from TMEM, V MN-major
      const uint32_t tS[2] = {tmem, tmem + 128};
      const uint32_t tO[2] = {tmem + 256, tmem + 384};
      const uint32_t sQ[2] = {sbase + OFF_Q, sbase + OFF_Q + TILE_BYTES};
      // Descriptors are built once; per-MMA start addresses are added to the
      // low (address >> 4) field, which cannot carry out of its 14 bits since
      // shared memory ends below 256 KB.
      const uint64_t dV0 = ptx::smem_desc_sw128(sbase + OFF_V, HALF_BYTES, 1024);
      const uint64_t dK0 = ptx::smem_desc_sw128(sbase + OFF_K, 16, 1024);
      const uint64_t dQ0 = ptx::smem_desc_sw128(sQ[0], 16, 1024);
      // O_i += P_i V for the V tile of running KV tile g; `first` (the item's
      // first KV tile) overwrites O_i instead.
      auto issue_pv = [&](int i, int g, bool first) {
        const uint64_t dv = ptx::launder(dV0 + (uint64_t)(((g % KV_STAGES) * TILE_BYTES) >> 4));
        const uint32_t ts = ptx::launder(tS[i]);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // B = V tile viewed as [K = keys][N = D]: N-contiguous 128-byte rows,
          // 8-row groups 1024 B apart (SBO), the two 64-column halves 16 KB apart (LBO).
          ptx::mma_ts(tO[i], ts + kk * 8, dv + (uint64_t)((kk * 16 * 128) >> 4), IDESC_PV,
                      (!first || kk > 0) ? 1u : 0u);
        }
      };
      auto issue_s = [&](int i, int g) {
        const uint64_t dk = ptx::launder(dK0 + (uint64_t)(((g % KV_STAGES) * TILE_BYTES) >> 4));
        const uint64_t dq = ptx::launder(dQ0 + (uint64_t)((i * TILE_BYTES) >> 4));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t off = (uint64_t)((((kk / 4) * HALF_BYTES) + (kk % 4) * 32) >> 4);
          ptx::mma_ss(tS[i], dq + off, dk + off, IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      bool ok = true;
      int n = 0;
      for (int64_t item = blockIdx.x; ok && item < item_end; item += item_step, ++n) {
        if (!(ok = ptx::mbar_wait(bar(B_QFULL), (uint32_t)(n & 1), G, abort_flag, kDevTimeoutMma))) break;
        const int g0 = n * kv_total;
        for (int j = 0; ok && j < kv_total; ++j) {
          const int g = g0 + j;
          const int s = g % KV_STAGES;
          if (!(ok = ptx::mbar_wait(bar(B_KFULL + s), (uint32_t)((g / KV_STAGES) & 1), G, abort_flag, kDevTimeoutMma)))
            break;
          ptx::tc_fence_after();
          for (int i = 0; i < 2; ++i) {
            if (j > 0) {
              const int gv = g - 1;
              if (!(ok = ptx::mbar_wait(bar(B_PFULL + i), (uint32_t)(gv & 1), G, abort_flag, kDevTimeoutMma))) break;
              if (i == 0 && !(ok = ptx::mbar_wait(bar(B_VFULL + gv % KV_STAGES), (uint32_t)((gv / KV_STAGES) & 1), G,
                                                  abort_flag, kDevTimeoutMma)))
                break;
              ptx::tc_fence_after();
              issue_pv(i, gv, j == 1);
              if (i == 1) ptx::mma_commit(bar(B_VEMPTY + gv % KV_STAGES));
            }
            issue_s(i, g);
            ptx::mma_commit(bar(B_SFULL + i));
          }
          if (!ok) break;
          ptx::mma_commit(bar(B_KEMPTY + s));
        }
        if (!ok) break;
        ptx::mma_commit(bar(B_QEMPTY));  // both Q tiles are free once this item's S GEMMs complete
        const int gl = g0 + kv_total - 1;
        for (int i = 0; i < 2 && ok; ++i) {
          if (!(ok = ptx::mbar_wait(bar(B_PFULL + i), (uint32_t)(gl & 1), G, abort_flag, kDevTimeoutMma))) break;
          if (i == 0 && !(ok = ptx::mbar_wait(bar(B_VFULL + gl % KV_STAGES), (uint32_t)((gl / KV_STAGES) & 1), G,
                                              abort_flag, kDevTimeoutMma)))
            break;
          ptx::tc_fence_after();
          issue_pv(i, gl, kv_total == 1);
          ptx::mma_commit(bar(B_ODONE + i));
        }
        if (ok) ptx::mma_commit(bar(B_VEMPTY + gl % KV_STAGES));
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
    bool ok = true;
    int n = 0;
    for (int64_t item = blockIdx.x; ok && item < item_end; item += item_step, ++n) {
      float m = -INFINITY;  // running reference maximum, log2 domain
      float l = 0.f;        // running row sum relative to m
      const int g0 = n * kv_total;
      for (int j = 0; j < kv_total; ++j) {
        // every lane waits; the decision is made warp-uniform before the
        // warp-collective TMEM accesses below
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(B_SFULL + wg), (uint32_t)((g0 + j) & 1), G, abort_flag,
                                                    kDevTimeoutSoftmax));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[BN];
        ptx::tmem_ld4x32(tS, sr);
        float* s = reinterpret_cast<float*>(sr);
        bool second;
        const int valid = kv_tile<kKv2>(p.kv, p.kv2, j, second).valid;
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
      // ---------------------------------------------------------- epilogue
      if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(B_ODONE + wg), (uint32_t)(n & 1), G, abort_flag,
                                                          kDevTimeoutEpilogue));
      if (!ok) break;
      ptx::tc_fence_after();
      int64_t orow0;
      int rows_valid;
      void* out_base;
      float* lse_base;
      if (kPersist) {  // one query set: its parameters sit at fixed offsets
        epi_rows(p, p.qs[0], item_of<true>(p, item), wg, orow0, rows_valid);
        out_base = p.qs[0].out;
        lse_base = p.qs[0].lse;
      } else {
        const EpiInfo* epi = reinterpret_cast<const EpiInfo*>(smem + OFF_EPI);
        orow0 = epi->orow0[wg];
        rows_valid = epi->valid[wg];
        out_base = epi->out;
        lse_base = epi->lse;
      }
      const bool store = row < rows_valid;
      const int64_t orow = orow0 + row;
      const float inv_l = 1.f / l;
      __nv_bfloat16* optr = reinterpret_cast<__nv_bfloat16*>(out_base) + orow * HD;
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
      if (store) lse_base[orow] = (m + log2f(l)) * 0.69314718055994531f;
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

namespace {

struct KvMaps {
  CUtensorMap k, v, k2, v2;
};

// Query-side description and tensor map of one AttnArgs.
bool make_qside(const AttnArgs& a, QSide* qs, CUtensorMap* mq) {
  auto tiles = [](int64_t rows) { return (int)((rows + BM - 1) / BM); };
  if (a.out_stack != a.q_stack) return false;  // out rows follow the query rows
  if (a.q_stack) {
    const int tps = tiles(a.Ns);
    qs->q = TileSrc{1, a.Ns, tps, (int)(tps * a.sp)};
    if (!make_map_4d(mq, a.q, a.Ns, a.BH, a.sp)) return false;
  } else {
    qs->q = TileSrc{0, a.Nq, tiles(a.Nq), tiles(a.Nq)};
    if (!make_map_3d(mq, a.q, a.Nq, a.q_heads)) return false;
  }
  qs->out = a.out;
  qs->lse = a.lse;
  qs->out_kind = a.out_stack ? 1 : 0;
  qs->out_rows = a.out_stack ? a.Ns : a.Nq;
  qs->map = a.map;
  qs->pairs = (qs->q.tiles + 1) / 2;
  qs->ctas = (int64_t)qs->pairs * a.units;
  return true;
}

// KV sources and their tensor maps.
bool make_kv(const AttnArgs& a, TcParams* p, KvMaps* m) {
  auto tiles = [](int64_t rows) { return (int)((rows + BM - 1) / BM); };
  if (a.kv_stack) {
    const int tps = tiles(a.Ns);
    p->kv = TileSrc{1, a.Ns, tps, (int)(tps * a.sp)};
    if (!make_map_4d(&m->k, a.k, a.Ns, a.BH, a.sp) || !make_map_4d(&m->v, a.v, a.Ns, a.BH, a.sp)) return false;
  } else {
    p->kv = TileSrc{0, a.Nk, tiles(a.Nk), tiles(a.Nk)};
    if (!make_map_3d(&m->k, a.k, a.Nk, a.kv_heads) || !make_map_3d(&m->v, a.v, a.Nk, a.kv_heads)) return false;
  }
  if (a.k2 && a.Nk2 > 0) {  // second KV source: plain [heads][Nk2][D]
    p->kv2 = TileSrc{0, a.Nk2, tiles(a.Nk2), tiles(a.Nk2)};
    if (!make_map_3d(&m->k2, a.k2, a.Nk2, a.kv2_heads) || !make_map_3d(&m->v2, a.v2, a.Nk2, a.kv2_heads))
      return false;
  } else {
    p->kv2 = TileSrc{0, 1, 1, 0};
    m->k2 = m->k;
    m->v2 = m->v;
  }
  return true;
}

}  // namespace

cudaError_t launch_attn_tc_fwd(const AttnArgs* sides, int nsides, const Guard& g, cudaStream_t stream) {
  static std::atomic<unsigned long long> attr[4];
  cudaError_t ea = smem_limit_once(attr[0], (const void*)attn_tc_fwd_kernel<false, false>, SMEM_BYTES);
  if (ea == cudaSuccess) ea = smem_limit_once(attr[1], (const void*)attn_tc_fwd_kernel<true, false>, SMEM_BYTES);
  if (ea == cudaSuccess) ea = smem_limit_once(attr[2], (const void*)attn_tc_fwd_kernel<false, true>, SMEM_BYTES);
  if (ea == cudaSuccess) ea = smem_limit_once(attr[3], (const void*)attn_tc_fwd_kernel<true, true>, SMEM_BYTES);
  if (ea != cudaSuccess) return ea;
  if (nsides < 1 || nsides > 2) return cudaErrorInvalidValue;
  const AttnArgs& a0 = sides[0];
  if (nsides == 2) {  // the two query sets share the KV sources, the stack geometry and the scale
    const AttnArgs& a1 = sides[1];
    if (a1.k != a0.k || a1.v != a0.v || a1.k2 != a0.k2 || a1.v2 != a0.v2 || a1.kv_stack != a0.kv_stack ||
        a1.Nk != a0.Nk || a1.Nk2 != a0.Nk2 || a1.kv_heads != a0.kv_heads || a1.kv2_heads != a0.kv2_heads ||
        a1.BH != a0.BH || a1.Ns != a0.Ns || a1.sp != a0.sp || a1.scale != a0.scale)
      return cudaErrorInvalidValue;
  }
  TcParams p{};
  CUtensorMap mq[2];
  KvMaps mkv;
  for (int i = 0; i < nsides; ++i)
    if (!make_qside(sides[i], &p.qs[i], &mq[i])) return cudaErrorInvalidValue;
  if (nsides == 1) {  // an empty second query set
    p.qs[1] = p.qs[0];
    p.qs[1].ctas = 0;
    mq[1] = mq[0];
  }
  if (!make_kv(a0, &p, &mkv)) return cudaErrorInvalidValue;
  p.BH = a0.BH;
  p.Ns = a0.Ns;
  p.scale_log2 = a0.scale * 1.4426950408889634f;
  p.guard = g;
  const int64_t items = p.qs[0].ctas + p.qs[1].ctas;
  if (items < 1 || items > 2147483647LL) return cudaErrorInvalidValue;
  // One query set with a short KV loop: a persistent grid of at most one CTA
  // per SM walks the items, hiding each item's Q load, first S GEMMs and
  // prologue under the previous item's epilogue (measured on GB300: cross-
  // attention over 4 text tiles 1.2-1.4x faster, 16-32 tiles 4-6%).  Long KV
  // loops keep one CTA per item: there the fixed costs are a small share and
  // the hardware's dynamic CTA placement balances the SMs better than a
  // static walk (64 tiles neutral, 128-256 tiles 1.5-2.5% slower persistent).
  // Two query sets also keep one CTA per item.
  const bool persist = nsides == 1 && p.kv.tiles + p.kv2.tiles <= kPersistMaxKvTiles;
  int64_t ctas = items;
  if (persist) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (sms > 0 && ctas > sms) ctas = sms;
  }
  const dim3 grid((unsigned)ctas, 1, 1), block(NUM_THREADS);
  const bool kv2 = p.kv2.tiles > 0;
  if (persist && kv2)
    return launch_pdl(attn_tc_fwd_kernel<true, true>, grid, block, SMEM_BYTES, stream, mq[0], mq[1], mkv.k, mkv.v,
                      mkv.k2, mkv.v2, p);
  if (persist)
    return launch_pdl(attn_tc_fwd_kernel<false, true>, grid, block, SMEM_BYTES, stream, mq[0], mq[1], mkv.k, mkv.v,
                      mkv.k2, mkv.v2, p);
  if (kv2)
    return launch_pdl(attn_tc_fwd_kernel<true, false>, grid, block, SMEM_BYTES, stream, mq[0], mq[1], mkv.k, mkv.v,
                      mkv.k2, mkv.v2, p);
  return launch_pdl(attn_tc_fwd_kernel<false, false>, grid, block, SMEM_BYTES, stream, mq[0], mq[1], mkv.k, mkv.v,
                    mkv.k2, mkv.v2, p);
}

}  // namespace usp
