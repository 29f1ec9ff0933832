// a3 / a5 / a6 -- CSA2 indexer scores on the tensor cores.
//
// s_j = sum_h w_h ReLU(q_h . K_j) (DeepSeek-V4.1 Flash, hn.213312.xyz
// sec. 2.3.1; 36kr "CSA2") for every visible indexer-K entry (Full) or for the
// entries of an HSI pool (Reindex, hn.213312.xyz sec. 2.3.4).  Per CTA: a
// range of 128-entry tiles of one group of up to QPC queries of one sequence
// (a multi-query decode block of up to 6 positions shares one group, so every
// indexer-K tile is read once for all of them).
//  - page mode (Full): the warp after the consumers (one elected lane)
//    streams whole cache pages, two per tile, into a shared-memory ring with
//    1-D bulk copies completing on mbarriers;
//  - gather mode (Reindex): each thread gathers its own entry of the pool
//    with cp.async into the same ring layout (block ids resolved to pages
//    once at set-up);
//  - the consumer warpgroups (two to four, see Shape) take tiles in turn;
//    thread t of a warpgroup owns entry t of the tile and TMEM lane t: it
//    decodes the entry (FP4 -> f16, exact; bf16 kept) into its warpgroup's
//    A buffer (TMEM, or shared memory for runs of 4 queries), and one thread
//    issues tcgen05.mma D[128 x 32*QPC] = K_tile . Q^T with Q_idx (f16 /
//    bf16) from shared memory;
//  - the epilogue reads D back (one row per thread), forms the ReLU-weighted
//    head sums, writes the scores, the 8-entry block maxima for HSI and folds
//    this CTA's key range per query (one slot each) for the top-k selection.
// The epilogue of a warpgroup's previous tile runs while its next MMA
// executes, and the warpgroups interleave on the tensor core.  Single-query
// FP4 page scans (every decode Full layer) replace the producer warp by one
// issuer warp per warpgroup, which copies that warpgroup's tiles and issues
// its MMAs, and lay the queries' tiles end to end over one wave of CTAs
// (one per SM).  When the grid is one wave, the first copying warp
// prefetches its first ring pass into L2 while the previous kernel (the
// compressor) still runs.  Every wait is bounded.
#include <algorithm>

#include "internal.h"
#include "score_common.cuh"
#include "tc.cuh"

namespace csa2 {
namespace {

// Consumer warpgroups: four on single-query FP4 tiles (latency-bound decode
// and epilogue, the decoded K tile in TMEM); four on FP4 runs of 4 queries
// with the decoded K tile in shared memory (TMEM then holds only the
// accumulators, 4 x 128 columns); two otherwise (TMEM and shared-memory
// budget).
template <int kDtype, int QPC, bool kGather>
struct Shape {
  static constexpr bool kSmemA = QPC == 4 && kDtype != CSA2_CACHE_BF16;
  static constexpr int kWG = ((QPC == 1 && kDtype != CSA2_CACHE_BF16) || kSmemA) ? 4 : 2;
  static constexpr int kConsumers = 128 * kWG;
  // single-query FP4 page scans: one issuer warp per consumer warpgroup
  // (copies of its tiles, its MMAs) instead of one producer warp
  static constexpr bool kIss = QPC == 1 && kDtype != CSA2_CACHE_BF16 && !kGather;
  static constexpr int kThreads = kConsumers + (kIss ? 32 * kWG : 32);
  static constexpr int kStages = kSmemA ? 6 : 2 * kWG;  // ring slots, used in tile order
};
constexpr int kABytes = 128 * kIdxDim * 2;  // a decoded K tile in shared memory (f16, K-major)
constexpr int kMaxTilesPerCta = 512;
constexpr int kMaxGatherTiles = 32;        // gather mode: resolved positions held in shared memory

template <int kDtype>
struct TileFmt {
  static constexpr int kPageData = (kDtype == CSA2_CACHE_BF16) ? kIdxBf16Data : kIdxFp4Data;
  static constexpr int kPageScales = (kDtype == CSA2_CACHE_FP4) ? kIdxFp4Scales
                                     : (kDtype == CSA2_CACHE_FP4_S32) ? kIdxS32Scales : 0;
  static constexpr int kSlotBytes = 2 * (kPageData + kPageScales);
};

struct ScoreArgs {
  int q0, Tq, r;
  int seg, gps;         // query groups: segments of `seg` queries from q0, `gps` groups of QPC each
  int q_fp4;            // score with FP4-encoded indexer queries
  int prefetch;         // page mode, one wave: warm L2 with the first ring pass before the wait
  const uint16_t* q_idx;
  const float* head_w;
  const int64_t* q_pos;
  CacheView ic;
  const int32_t* n_entries;
  int64_t max_entries;
  int tiles_per_cta;
  const int32_t* pool;  // gather mode: pool block ids [Q][n_blocks]
  int n_blocks;
  float* scores;        // [chunk][stride]
  int64_t stride;
  float* bmax;          // [chunk][ceil(max_entries/8)] or null
  uint32_t* krange;     // [chunk][kr_stride][2]: key range of each CTA's scores of each query
  int kr_stride;
  int32_t* status;
  // single-query page scans in one wave (flat != 0): CTA c takes tiles
  // [c total / G, (c + 1) total / G) of the flattened sequence of the chunk's
  // queries' tiles (tq per query, total = queries x tq), at most two queries
  int flat;
  int64_t tq, total;
  int kr_pad;  // flat mode: key-range slots read per query (unused ones are written empty)
};

// First flattened tile of CTA c, and the CTA holding flattened tile x (the
// largest c with flat_first(c) <= x).
__host__ __device__ inline int64_t flat_first(int64_t c, int64_t total, int64_t grid) { return c * total / grid; }
__host__ __device__ inline int64_t flat_cta_of(int64_t x, int64_t total, int64_t grid) {
  return ((x + 1) * grid - 1) / total;
}

using score::e2m1x8_to_f16x2;
using score::fadd2;
using score::ffma2;

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Barrier of one warpgroup (ids 1..4) or of all consumers (id 5).
__device__ __forceinline__ void wg_sync(int g) { asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory"); }
__device__ __forceinline__ void consumers_sync(int n) { asm volatile("bar.sync 5, %0;" ::"r"(n) : "memory"); }
// Page table hand-off in page mode: the consumers arrive once their share of
// the page table is written, the producer warp waits (barrier 6, all threads).
template <int kThreadsAll>
__device__ __forceinline__ void pages_arrive_n() { asm volatile("bar.arrive 6, %0;" ::"n"(kThreadsAll) : "memory"); }
template <int kThreadsAll>
__device__ __forceinline__ void pages_sync_n() { asm volatile("bar.sync 6, %0;" ::"n"(kThreadsAll) : "memory"); }
// End of a CTA with issuer warps (barrier 7, all threads).
template <int kThreadsAll>
__device__ __forceinline__ void all_sync_n() { asm volatile("bar.sync 7, %0;" ::"n"(kThreadsAll) : "memory"); }

template <int kDtype, int QPC, bool kGather>
__global__ void __launch_bounds__(Shape<kDtype, QPC, kGather>::kThreads, 1) score_tc_kernel(ScoreArgs a) {
  using F = TileFmt<kDtype>;
  using Sh = Shape<kDtype, QPC, kGather>;
  constexpr int kWG = Sh::kWG;
  constexpr int kConsumers = Sh::kConsumers;
  constexpr int kThreads = Sh::kThreads;
  constexpr int kStages = Sh::kStages;
  constexpr bool kIss = Sh::kIss;
  auto pages_arrive = [] { pages_arrive_n<kThreads>(); };
  auto pages_sync = [] { pages_sync_n<kThreads>(); };
  constexpr int kN = 32 * QPC;                    // MMA N: QPC queries x 32 heads
  constexpr int kAcols = 64;                      // 128 channels of f16 pairs
  constexpr bool kSmemA = Sh::kSmemA;
  // D double-buffered per warpgroup when tensor memory holds it (the MMA of
  // tile u runs while the epilogue of tile u-1 reads the other buffer)
  constexpr int kDBuf = (!kSmemA && kWG * kAcols + 2 * kWG * kN <= 512) ? 2 : 1;
  constexpr int kTmemCols = ((kSmemA ? 0 : kWG * kAcols) + kDBuf * kWG * kN) <= 256 ? 256 : 512;
  constexpr bool kBf16 = (kDtype == CSA2_CACHE_BF16);
  constexpr uint32_t kIdesc = tc::idesc_f16(128, kN, kBf16, kBf16, false, false);
  static_assert(!kGather || QPC == 1, "gather mode scores one query per CTA");
  // query slots of a CTA: the group's QPC queries, or in the flat mode the
  // (at most) two queries its tile range touches
  constexpr bool kFlatable = QPC == 1 && !kGather;
  constexpr int kQS = kFlatable ? 2 : QPC;
  const bool flat = kFlatable && a.flat;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int jg = blockIdx.y % a.gps;
  int qc0 = (blockIdx.y / a.gps) * a.seg + jg * QPC;  // chunk-local index of the first query
  int n_act = min(QPC, a.seg - jg * QPC);             // queries of the group; the rest are masked
  int64_t gt0 = 0, gt1 = 0;
  bool two = false;
  if (flat) {
    gt0 = flat_first(blockIdx.x, a.total, gridDim.x);
    gt1 = flat_first(blockIdx.x + 1, a.total, gridDim.x);
    qc0 = (int)(gt0 / a.tq);
    two = gt1 > (int64_t)(qc0 + 1) * a.tq;
    n_act = two ? 2 : 1;
  }
  const int g0 = a.q0 + qc0;                          // first query of the CTA
  const int b = g0 / a.Tq;
  if (!kGather && a.prefetch && warp == kConsumers / 32) {
    // While the previous kernel runs (the grid is one wave, so every CTA is
    // resident early): the producer warp brings the pages of this CTA's
    // first ring pass into L2.  Only hints are issued here: the block-table
    // entries read to aim them are read again after the wait, and every
    // prefetched page lies in the page pool.
    const int lane = tid & 31;
    const int64_t tb0 = flat ? gt0 - (int64_t)qc0 * a.tq : (int64_t)blockIdx.x * a.tiles_per_cta;
    const int64_t pp = 2 * tb0 + lane;  // logical page (of the CTA's first query)
    const int64_t qend = (int64_t)(qc0 + 1) * a.tq;
    const int64_t lim = flat ? 2 * ((gt1 < qend ? gt1 : qend) - gt0) : 2 * a.tiles_per_cta;
    if (lane < lim && lane < 2 * kStages && pp < a.ic.max_pages && pp * kPage < a.max_entries) {
      const int32_t pg = tc::ld_cg_s32(a.ic.block_table + (int64_t)b * a.ic.max_pages + pp);
      if (pg >= 0 && pg < a.ic.num_pages) {
        tc::bulk_prefetch_l2(a.ic.data + (int64_t)pg * F::kPageData, F::kPageData);
        if (F::kPageScales) tc::bulk_prefetch_l2(a.ic.scales + (int64_t)pg * F::kPageScales, F::kPageScales);
      }
    }
  }
  griddep_wait();  // before any other global read or tensor-memory allocation
  griddep_launch();

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* qtile = smem;                          // [kQS*32 rows][128] K-major: query slot j at j * 256 * 32
  uint8_t* ring = smem + 256 * 32 * kQS;          // kStages slots
  uint8_t* abuf = ring + kStages * TileFmt<kDtype>::kSlotBytes;  // kSmemA: one K tile per warpgroup
  __shared__ float hw[kQS][kIdxHeads];  // half the head weights (see the epilogue)
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], mma_bar[kWG];
  __shared__ __align__(8) uint64_t a_full[kWG];  // kIss: warpgroup g has stored its A tile
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ uint32_t rng_lo[kQS], rng_hi[kQS];  // this CTA's key range per query slot
  __shared__ int32_t ptab[kGather ? 1 : 2 * kMaxTilesPerCta];     // page mode: pages of this CTA's tiles
  __shared__ int32_t gtab[kGather ? kMaxGatherTiles * 128 : 1];   // gather mode: page*64+slot or -1

  int64_t nv[kQS];
  int64_t nv_max = 0;
#pragma unroll
  for (int q = 0; q < kQS; ++q) {
    const int bq = (g0 + q) / a.Tq;
    const int64_t ne = q < n_act ? (a.n_entries[bq] < a.max_entries ? a.n_entries[bq] : a.max_entries) : 0;
    nv[q] = q < n_act ? visible_entries(a.q_pos[g0 + q], a.r, ne) : 0;
    nv_max = nv[q] > nv_max ? nv[q] : nv_max;
  }
  const int64_t npos = kGather ? (int64_t)a.n_blocks * kHsiBlock : nv_max;
  const int64_t n_tiles = (npos + 127) / 128;
  int64_t t_begin = (int64_t)blockIdx.x * a.tiles_per_cta;
  int64_t t_end = t_begin + a.tiles_per_cta < n_tiles ? t_begin + a.tiles_per_cta : n_tiles;
  // flat mode: the active tiles are slot 0's tiles ta0 .. ta0 + ka - 1, then
  // slot 1's tiles 0 .. kb - 1 (tiles past a query's visible entries skipped)
  int64_t ta0 = 0;
  int ka = 0;
  if (flat) {
    ta0 = gt0 - (int64_t)qc0 * a.tq;
    const int64_t na = (two ? (int64_t)(qc0 + 1) * a.tq : gt1) - gt0;
    const int64_t nb = two ? gt1 - (int64_t)(qc0 + 1) * a.tq : 0;
    const int64_t ra = (nv[0] + 127) / 128 - ta0, rb = (nv[1] + 127) / 128;  // visible tiles left
    ka = (int)(ra < 0 ? 0 : (ra < na ? ra : na));
    const int kb = (int)(rb < nb ? rb : nb);
    t_begin = 0;
    t_end = ka + kb;
  }
  // query slot and tile (within its query) of CTA-local tile i
  auto tile_slot = [&](int64_t i) -> int { return flat ? (i < ka ? 0 : 1) : 0; };
  auto tile_of = [&](int64_t i) -> int64_t { return flat ? (i < ka ? ta0 + i : i - ka) : t_begin + i; };
  // key-range slot of query slot j: one per CTA of the query's tiles
  auto kr_slot = [&](int j) -> int64_t {
    return flat ? blockIdx.x - flat_cta_of((int64_t)(qc0 + j) * a.tq, a.total, gridDim.x) : (int64_t)blockIdx.x;
  };
  // this CTA's key range of query slot j; in the flat mode the CTA holding a
  // query's last tile also empties the query's slots past its own
  auto put_range = [&](int j, uint32_t lo, uint32_t hi) {
    uint32_t* kr = a.krange + (int64_t)(qc0 + j) * a.kr_stride * 2;
    const int64_t s = kr_slot(j);
    kr[2 * s] = lo;
    kr[2 * s + 1] = hi;
    if (flat && (int64_t)(qc0 + j + 1) * a.tq <= gt1)
      for (int64_t x = s + 1; x < a.kr_pad; ++x) {
        kr[2 * x] = 0xFFFFFFFFu;
        kr[2 * x + 1] = 0u;
      }
  };
  if (t_begin >= t_end) {  // uniform: the whole CTA leaves before any barrier, its slots empty
    if (tid < n_act) put_range(tid, 0xFFFFFFFFu, 0u);
    return;
  }
  const int n_my = (int)(t_end - t_begin);
  // logical page h of CTA-local tile i and the sequence it belongs to
  auto page_id = [&](int i, int h) -> int32_t {
    const int j = tile_slot(i);
    const int64_t p = 2 * tile_of(i) + h;
    const int64_t lim = flat ? nv[j] : nv_max;  // a group's tiles serve every query of the group
    return (p * kPage < lim) ? (int32_t)page_of(a.ic, (g0 + j) / a.Tq, p * kPage, a.status) : -1;
  };

  // ---- barriers and TMEM first: the producer starts copying pages while the
  // consumers build the Q tile
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 128);
    }
    for (int w = 0; w < kWG; ++w) {
      tc::mbar_init(&mma_bar[w], 1);
      tc::mbar_init(&a_full[w], 128);
    }
    abort_flag = 0;
    for (int q = 0; q < kQS; ++q) {
      rng_lo[q] = 0xFFFFFFFFu;
      rng_hi[q] = 0u;
    }
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = tmem_base;

  // the copy of CTA-local tile i into its ring slot (page mode)
  auto copy_tile = [&](int i) {
    const int s = i % kStages;
    uint8_t* slot = ring + (size_t)s * F::kSlotBytes;
    uint32_t bytes = 0;
    int64_t pages[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      pages[hh] = ptab[2 * i + hh];
      if (pages[hh] >= 0) bytes += F::kPageData + F::kPageScales;
    }
    tc::mbar_arrive_expect_tx(&full_bar[s], bytes);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      if (pages[hh] < 0) continue;
      tc::bulk_g2s(slot + hh * F::kPageData, a.ic.data + pages[hh] * F::kPageData, F::kPageData, &full_bar[s]);
      if (F::kPageScales)
        tc::bulk_g2s(slot + 2 * F::kPageData + hh * F::kPageScales, a.ic.scales + pages[hh] * F::kPageScales,
                     F::kPageScales, &full_bar[s]);
    }
  };

  if (kIss && warp >= kConsumers / 32) {
    // ------------------------------------------------------------- issuers
    // Issuer warp k serves warpgroup k, whose tiles k, k + kWG, ... use ring
    // slots k and k + kWG in turn: it copies the warpgroup's next tile into a
    // slot once the warpgroup has decoded the slot's tile and stored it as A
    // (a_full), and issues that tile's MMA.  The MMA issue, which holds its
    // thread for about a thousand cycles per tile, so stays off the
    // warpgroup's own path.
    const int k = warp - kConsumers / 32;
    const int lane = tid & 31;
    const int n_k = n_my > k ? (n_my - k + kWG - 1) / kWG : 0;
    const int first = n_k < 2 ? n_k : 2;
    if (lane < 2 * first) {
      const int i = k + kWG * (lane >> 1);
      ptab[2 * i + (lane & 1)] = page_id(i, lane & 1);
    }
    __syncwarp();
    if (lane < first) copy_tile(k + kWG * lane);
    __syncwarp();
    pages_sync();  // the consumers' share of the page table is written
    if (lane == 0) {
      const uint32_t acol_k = (uint32_t)(k * kAcols);
      const uint32_t dcol_k = (uint32_t)(kWG * kAcols + k * kDBuf * kN);
      int issued = -1, copied = first;
      for (int u = 0; u < n_k; ++u) {
        if (!tc::mbar_wait(&a_full[k], u & 1)) {
          report(a.status, CSA2_ERR_TIMEOUT);
          atomicExch(&abort_flag, 1);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
        tc::fence_after_sync();
        const int i = k + kWG * u;
        const uint32_t qaddr = tc::smem_u32(qtile) + tile_slot(i) * 256 * 32;
#pragma unroll
        for (int ks = 0; ks < kIdxDim / 16; ++ks)
          tc::mma_ts(tb + dcol_k + (uint32_t)((u % kDBuf) * kN), tb + acol_k + ks * 8,
                     tc::sdesc(qaddr + ks * 256, 128, kIdxDim * 16), kIdesc, ks > 0);
        tc::mma_commit(&mma_bar[k]);
        issued = u;
        if (u + 2 < n_k) {
          copy_tile(k + kWG * (u + 2));
          copied = u + 3;
        }
      }
      // no copy into this CTA's shared memory and no MMA in flight at its end
      for (int v = copied > 2 ? copied - 2 : 0; v < copied; ++v) {
        const int i = k + kWG * v;
        if (!tc::mbar_wait(&full_bar[i % kStages], (i / kStages) & 1)) report(a.status, CSA2_ERR_TIMEOUT);
      }
      if (issued >= 0 && !tc::mbar_wait(&mma_bar[k], issued & 1)) report(a.status, CSA2_ERR_TIMEOUT);
    }
    __syncwarp();
    tc::fence_before_sync();
    all_sync_n<kThreads>();  // then the consumers release tensor memory
    return;
  }

  if (warp == kConsumers / 32) {
    // ------------------------------------------------------------ producer
    if (!kGather) {
      const int lane = tid & 31;
      const int first = n_my < kStages ? n_my : kStages;
      if (lane < 2 * first) ptab[lane] = page_id(lane >> 1, lane & 1);  // the first pass; the consumers resolve the rest
      __syncwarp();
      auto issue = copy_tile;
      // the first pass over the ring (fresh slots) from one lane per tile, the
      // rest in order from lane 0 once the consumers release each slot
      if (lane < first) issue(lane);
      __syncwarp();
      pages_sync();  // the consumers' share of the page table is written
      if (lane == 0) {
        int issued = first;
        for (int i = first; i < n_my; ++i) {
          const int s = i % kStages;
          if (!tc::mbar_wait(&empty_bar[s], ((i / kStages) & 1) ^ 1)) {
            report(a.status, CSA2_ERR_TIMEOUT);
            atomicExch(&abort_flag, 1);
            break;
          }
          if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
          issue(i);
          ++issued;
        }
        // do not leave while copies into this CTA's shared memory are in flight
        for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
          if (!tc::mbar_wait(&full_bar[i % kStages], (i / kStages) & 1)) report(a.status, CSA2_ERR_TIMEOUT);
      }
    }
    return;
  }

  // ---- consumers' set-up: the pages after the producer's first pass (then
  // release the producer), Q_idx (f16 or bf16) into the B tile, head
  // weights, gather positions
  if (!kGather) {
    const int first = n_my < kStages ? n_my : kStages;
    for (int i = 2 * first + tid; i < 2 * n_my; i += kConsumers) ptab[i] = page_id(i >> 1, i & 1);
    pages_arrive();
  }
  for (int i = tid; i < kQS * 32 * kIdxDim / 8; i += kConsumers) {
    const int row = (8 * i) / kIdxDim, k = (8 * i) % kIdxDim;  // row = q*32 + h; 8 channels per load
    uint4 v = make_uint4(0u, 0u, 0u, 0u);  // masked queries: zero rows
    if (row / kIdxHeads < n_act)
      v = __ldg(reinterpret_cast<const uint4*>(a.q_idx + (int64_t)(g0 + row / kIdxHeads) * kIdxHeads * kIdxDim +
                                               (row % kIdxHeads) * kIdxDim + k));
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (score::q_operand8<kBf16>(w, a.q_fp4 != 0)) report(a.status, CSA2_ERR_RANGE);
    *reinterpret_cast<uint4*>(qtile + tc::kmajor_off(row, k, kIdxDim)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  for (int i = tid; i < kQS * kIdxHeads; i += kConsumers)
    hw[i / kIdxHeads][i % kIdxHeads] =
        (a.head_w && i / kIdxHeads < n_act) ? 0.5f * __ldg(a.head_w + (int64_t)g0 * kIdxHeads + i) : 0.5f;
  if (kGather) {
    // this thread's positions i = tid + kConsumers * u: every pool entry
    // loaded first, then every block-table entry, so that the loads of its
    // positions are in flight together rather than one pair after another
    constexpr int kIt = (kMaxGatherTiles * 128 + kConsumers - 1) / kConsumers;
    int32_t blkv[kIt];
#pragma unroll
    for (int u = 0; u < kIt; ++u) {
      const int i = tid + kConsumers * u;
      const int64_t p = t_begin * 128 + i;  // pool position
      blkv[u] = (i < n_my * 128 && p < npos) ? __ldg(a.pool + (int64_t)g0 * a.n_blocks + p / kHsiBlock) : -1;
    }
#pragma unroll
    for (int u = 0; u < kIt; ++u) {
      const int i = tid + kConsumers * u;
      const int64_t p = t_begin * 128 + i;
      const int32_t blk = blkv[u];
      int32_t e = -1;
      if (blk >= 0) {
        const int64_t j = (int64_t)blk * kHsiBlock + p % kHsiBlock;
        if ((int64_t)blk * kHsiBlock >= a.max_entries) {
          if (p % kHsiBlock == 0) report(a.status, CSA2_ERR_BAD_INDEX);
        } else if (j < nv[0]) {
          const int64_t page = page_of(a.ic, b, j, a.status);
          if (page >= 0) e = (int32_t)(page * kPage + j % kPage);
        }
      }
      if (i < n_my * 128) gtab[i] = e;
    }
  }
  tc::fence_async_smem();  // the Q tile is read by the tensor core
  consumers_sync(kConsumers);

  // -------------------------------------------------------------- consumers
  const int g = warp >> 2;               // warpgroup: tiles g, g + kWG, ...
  const int lt = tid & 127;              // entry of the tile, TMEM lane
  const uint32_t lane_base = 32 * (warp & 3);
  const uint32_t acol = (uint32_t)(g * kAcols);
  const uint32_t dcol0 = (uint32_t)((kSmemA ? 0 : kWG * kAcols) + g * kDBuf * kN);
  auto dcol_of = [&](int uu) { return dcol0 + (uint32_t)((uu % kDBuf) * kN); };
  uint8_t* atile = abuf + (size_t)g * kABytes;
  const int n_own = n_my > g ? (n_my - g + kWG - 1) / kWG : 0;
  uint32_t klo[kQS], khi[kQS];
#pragma unroll
  for (int q = 0; q < kQS; ++q) {
    klo[q] = 0xFFFFFFFFu;
    khi[q] = 0u;
  }
  const int h = lt >> 6, sl = lt & 63;  // where this entry sits in a tile's ring slot

  // gather mode: copy this thread's entry of own tile u into its slot
  auto gather = [&](int u) {
    if (kGather && u < n_own) {
      const int i = g + kWG * u;
      uint8_t* slot = ring + (size_t)(i % kStages) * F::kSlotBytes;
      const int32_t e = gtab[i * 128 + lt];
      if (e >= 0) {
        const int64_t page = e / kPage;
        const int es = e % kPage;
        if (kDtype != CSA2_CACHE_BF16) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            cp16(slot + h * kIdxFp4Data + (c * kPage + sl) * 16, a.ic.data + page * kIdxFp4Data + (c * kPage + es) * 16);
          if (kDtype == CSA2_CACHE_FP4)
            cp8(slot + 2 * kIdxFp4Data + h * kIdxFp4Scales + sl * 8, a.ic.scales + page * kIdxFp4Scales + es * 8);
          else
            cp4(slot + 2 * kIdxFp4Data + h * kIdxS32Scales + sl * 4, a.ic.scales + page * kIdxS32Scales + es * 4);
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            cp16(slot + h * kIdxBf16Data + (c * kPage + sl) * 16, a.ic.data + page * kIdxBf16Data + (c * kPage + es) * 16);
        }
      }
    }
    if (kGather) cp_commit();
  };
  gather(0);

  int last_issued = -1, waited = -1;  // own tile counters
  // each query slot's score and block-maximum rows, and its visible entries
  constexpr bool kRows = kQS <= 2;
  float* srow_q[kRows ? kQS : 1];
  float* brow_q[kRows ? kQS : 1];
  int nv32[kQS];
#pragma unroll
  for (int q = 0; q < kQS; ++q) {
    nv32[q] = (int)nv[q];
    if (kRows) {
      srow_q[q] = a.scores + (int64_t)(qc0 + q) * a.stride;
      brow_q[q] = a.bmax ? a.bmax + (int64_t)(qc0 + q) * ((a.max_entries + 7) / 8) : nullptr;
    }
  }

  // epilogue of own tile e (its MMA has completed): ReLU-weighted head sums,
  // scores, HSI block maxima, key ranges
  auto epilogue = [&](int e, bool ok) {
    const int ie = g + kWG * e;
    const int pos = (int)tile_of(ie) * 128 + lt;  // entry id (page mode) / pool position (gather mode)
    const int qs = tile_slot(ie);
#pragma unroll
    for (int q = 0; q < kQS; ++q) {
      if (q >= n_act) break;      // uniform over the CTA
      if (flat && q != qs) continue;  // flat mode: a tile scores one query slot, in D's first 32 columns
      uint32_t d[32];
      tc::tmem_ld32(tc::taddr(tb, lane_base, dcol_of(e) + 32 * (flat ? 0 : q)), d);
      tc::tmem_wait_ld();
      // four partial sums over heads h = 4i + j (two f32x2 accumulators),
      // added pairwise.  ReLU(x) is taken as (x + |x|) / 2, exactly: the
      // sums run over x + |x| (an add with an absolute-value operand, on the
      // FMA pipe like the packed adds, rather than a max on the ALU pipe) and
      // the half comes with the weights or at the end, both exact scalings
      // by two, so every partial sum is bit for bit the ReLU sum's.
      float2 p01 = make_float2(0.0f, 0.0f), p23 = make_float2(0.0f, 0.0f);
      auto relu2x = [&](int hh, int j) {  // 2 ReLU(x), exactly
        const float x = __uint_as_float(d[hh + j]);
        return x + fabsf(x);
      };
      if (a.head_w) {
#pragma unroll
        for (int hh = 0; hh < kIdxHeads; hh += 4) {
          p01 = ffma2(make_float2(hw[q][hh], hw[q][hh + 1]), make_float2(relu2x(hh, 0), relu2x(hh, 1)), p01);
          p23 = ffma2(make_float2(hw[q][hh + 2], hw[q][hh + 3]), make_float2(relu2x(hh, 2), relu2x(hh, 3)), p23);
        }
      } else {
#pragma unroll
        for (int hh = 0; hh < kIdxHeads; hh += 4) {
          p01 = fadd2(p01, make_float2(relu2x(hh, 0), relu2x(hh, 1)));
          p23 = fadd2(p23, make_float2(relu2x(hh, 2), relu2x(hh, 3)));
        }
      }
      float sc = (p01.x + p01.y) + (p23.x + p23.y);
      sc = a.head_w ? sc + 0.0f : 0.5f * sc;
      const int qc = qc0 + q;
      const bool valid = kGather ? (gtab[ie * 128 + lt] >= 0) : (pos < nv32[q]);
      if (!ok) sc = -INFINITY;
      float* srow = kRows ? srow_q[q] : a.scores + (int64_t)qc * a.stride;
      if (kGather) {
        if (pos < npos) srow[pos] = valid ? sc : __uint_as_float(kScoreInvalid);
      } else if (valid) {
        srow[pos] = sc;
      }
      if (valid) {
        const uint32_t kk = order_key(sc);
        klo[q] = min(klo[q], kk);
        khi[q] = max(khi[q], kk);
      }
      if (!kGather && a.bmax) {
        float m = valid ? sc : -INFINITY;
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        if ((lt & 7) == 0 && valid) (kRows ? brow_q[q] : a.bmax + (int64_t)qc * ((a.max_entries + 7) / 8))[pos >> 3] = m;
      }
    }
  };

  // own tile u's entry (this thread's) from the ring, decoded into 64
  // registers of f16 (or bf16) pairs; the ring slot is released
  // An FP4 entry as read from the ring: 64 bytes of codes and its scales
  struct Fp4Entry {
    uint4 cw[4];
    uint2 sc;
    bool present;
  };
  // own tile u's entry (this thread's) read from the ring, whose slot is
  // then released
  auto fetch = [&](int u, Fp4Entry& e) {
    const int i = g + kWG * u;
    const int s = i % kStages;
    if (kGather) {
      gather(u + 1);
      cp_wait<1>();
    } else if (!tc::mbar_wait(&full_bar[s], (i / kStages) & 1)) {
      atomicExch(&abort_flag, 1);
    }
    const uint8_t* slot = ring + (size_t)s * F::kSlotBytes;
    e.present = !kGather || gtab[i * 128 + lt] >= 0;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      e.cw[c] = *reinterpret_cast<const uint4*>(slot + h * kIdxFp4Data + (c * kPage + sl) * 16);
    // the entry's scales: 8 bytes (one per 16 channels) or 4 (one per 32)
    if (kDtype == CSA2_CACHE_FP4)
      e.sc = *reinterpret_cast<const uint2*>(slot + 2 * kIdxFp4Data + h * F::kPageScales + sl * 8);
    else
      e.sc = make_uint2(*reinterpret_cast<const uint32_t*>(slot + 2 * kIdxFp4Data + h * F::kPageScales + sl * 4), 0u);
    if (!kGather && !kIss) tc::mbar_arrive(&empty_bar[s]);
  };
  // the entry decoded into 64 registers of f16 pairs
  auto convert = [&](const Fp4Entry& e, uint32_t (&r)[64]) {
    // the scales, two per f16 pair as decoded (exact); each product takes
    // its scale as the pair's low or high half, which the f16 multiply reads
    // as an operand selection rather than a separate broadcast
    uint32_t sraw[4];
    sraw[0] = score::e4m3_pair(e.sc.x);
    sraw[1] = score::e4m3_pair(e.sc.x >> 16);
    if (kDtype == CSA2_CACHE_FP4) {
      sraw[2] = score::e4m3_pair(e.sc.y);
      sraw[3] = score::e4m3_pair(e.sc.y >> 16);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // 32 channels -> 16 registers
      const uint32_t w4[4] = {e.cw[c].x, e.cw[c].y, e.cw[c].z, e.cw[c].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // scale group of these 8 channels: 16-channel groups, or 32-channel ones
        const int gg = kDtype == CSA2_CACHE_FP4 ? 2 * c + (q >> 1) : c;
        const __half2 sp = *reinterpret_cast<const __half2*>(&sraw[gg >> 1]);
        const __half2 s2 = (gg & 1) ? __high2half2(sp) : __low2half2(sp);
        uint32_t h4[4];
        e2m1x8_to_f16x2(w4[q], h4);
#pragma unroll
        for (int by = 0; by < 4; ++by) {
          const __half2 prod = __hmul2(*reinterpret_cast<const __half2*>(&h4[by]), s2);  // exact
          r[16 * c + q * 4 + by] = e.present ? *reinterpret_cast<const uint32_t*>(&prod) : 0u;
        }
      }
    }
  };

  // own tile u's entry (this thread's) from the ring, decoded into 64
  // registers of f16 (or bf16) pairs; the ring slot is released
  auto decode = [&](int u, uint32_t (&r)[64]) {
    if (kDtype != CSA2_CACHE_BF16) {
      Fp4Entry e;
      fetch(u, e);
      convert(e, r);
      return;
    }
    const int i = g + kWG * u;
    const int s = i % kStages;
    if (kGather) {
      gather(u + 1);
      cp_wait<1>();
    } else if (!tc::mbar_wait(&full_bar[s], (i / kStages) & 1)) {
      atomicExch(&abort_flag, 1);
    }
    const uint8_t* slot = ring + (size_t)s * F::kSlotBytes;
    const bool present = !kGather || gtab[i * 128 + lt] >= 0;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(slot + h * kIdxBf16Data + (c * kPage + sl) * 16);
      r[4 * c] = present ? v.x : 0u;
      r[4 * c + 1] = present ? v.y : 0u;
      r[4 * c + 2] = present ? v.z : 0u;
      r[4 * c + 3] = present ? v.w : 0u;
    }
    if (!kGather && !kIss) tc::mbar_arrive(&empty_bar[s]);
  };

  // the decoded tile into the A buffer (shared or tensor memory)
  auto store_a = [&](const uint32_t (&r)[64]) {
    if (kSmemA) {
#pragma unroll
      for (int c = 0; c < 16; ++c)
        *reinterpret_cast<uint4*>(atile + tc::kmajor_off(lt, 8 * c, kIdxDim)) =
            make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
      tc::fence_async_smem();  // the K tile is read by the tensor core
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r16[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) r16[x] = r[16 * c + x];
        tc::tmem_st16(tc::taddr(tb, lane_base, acol + 16 * c), r16);
      }
      tc::tmem_wait_st();
    }
  };

  auto issue = [&](int u) {
    if (lt == 0) {
#pragma unroll
      for (int ks = 0; ks < kIdxDim / 16; ++ks) {
        const uint64_t bdesc =
            tc::sdesc(tc::smem_u32(qtile) + tile_slot(g + kWG * u) * 256 * 32 + ks * 256, 128, kIdxDim * 16);
        if (kSmemA)
          tc::mma_ss(tb + dcol_of(u), tc::sdesc(tc::smem_u32(atile) + ks * 256, 128, kIdxDim * 16), bdesc, kIdesc,
                     ks > 0);
        else
          tc::mma_ts(tb + dcol_of(u), tb + acol + ks * 8, bdesc, kIdesc, ks > 0);
      }
      tc::mma_commit(&mma_bar[g]);
    }
  };

  // wait for MMA u (its A buffer is free again and its D holds the products)
  auto wait_mma = [&](int u) {
    const bool ok = tc::mbar_wait(&mma_bar[g], u & 1);
    waited = u;
    if (!ok) {
      report(a.status, CSA2_ERR_TIMEOUT);
      atomicExch(&abort_flag, 1);
    }
    tc::fence_after_sync();
    return ok;
  };

  // Per own tile u: wait for MMA u-1 (the A buffer is free and D(u-1) holds
  // its products), decode and store A, issue MMA u; then the epilogue of u-1
  // while MMA u runs (with one D buffer the epilogue of u-1 comes before the
  // decode of u instead).
  // The tile is decoded after the wait, straight into the A buffer: decoding
  // it into registers before the wait (kEarly) was measured slower on the
  // single-query scans, whose 544-thread CTAs then spill, and so was a second
  // A buffer per warpgroup in shared memory (odd tiles) that let the MMA of
  // one tile run under the decode of the next.
  constexpr bool kEarly = false;
  if (kIss) {
    // With an issuer warp: wait for MMA u-1 (A free again), decode and store
    // A and signal the issuer, then the epilogue of u-1 while MMA u is issued
    // and runs.  The warps of the warpgroup do not wait for one another.
    // Reading the next tile's entry from the ring before the wait was
    // measured slower (the registers it holds across the wait spill).
    for (int u = 0; u <= n_own; ++u) {
      bool ok = true;
      if (u >= 1) ok = wait_mma(u - 1);
      if (u < n_own) {
        uint32_t r[64];
        decode(u, r);
        store_a(r);
        tc::fence_before_sync();
        tc::mbar_arrive(&a_full[g]);
      }
      if (u >= 1) epilogue(u - 1, ok);
      if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
    }
  }
  for (int u = 0; !kIss && u <= n_own; ++u) {
    const bool have = u < n_own;
    uint32_t r[64];
    if (kEarly && have) decode(u, r);
    bool ok = true;
    if (u >= 1) {
      ok = wait_mma(u - 1);
      if (kDBuf == 1) epilogue(u - 1, ok);
    }
    if (!kEarly && have) decode(u, r);
    if (have) store_a(r);
    tc::fence_before_sync();
    wg_sync(g);
    tc::fence_after_sync();
    if (*reinterpret_cast<volatile int*>(&abort_flag)) break;  // uniform within the warpgroup
    if (have) {
      issue(u);
      last_issued = u;
    }
    if (kDBuf == 2 && u >= 1) epilogue(u - 1, ok);
  }
  if (kGather) cp_wait<0>();  // no copies into this CTA's shared memory outlive it
#pragma unroll
  for (int q = 0; q < kQS; ++q) {
    uint32_t lo = klo[q], hi = khi[q];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if ((tid & 31) == 0 && lo <= hi) {
      atomicMin(&rng_lo[q], lo);
      atomicMax(&rng_hi[q], hi);
    }
  }
  // after an abort, let the last issued MMA finish before TMEM is released
  if (last_issued > waited) {
    if (!tc::mbar_wait(&mma_bar[g], last_issued & 1)) report(a.status, CSA2_ERR_TIMEOUT);
  }
  tc::fence_before_sync();
  if (kIss)
    all_sync_n<kThreads>();  // the issuers' MMAs have completed
  else
    consumers_sync(kConsumers);
  if (warp == 0) tc::tmem_dealloc(tb, kTmemCols);
  // one slot per CTA and query: no initialisation of global state needed
  if (tid < n_act) put_range(tid, rng_lo[tid], rng_hi[tid]);
}

}  // namespace

template <int kDtype, int QPC, bool kGather>
static cudaError_t launch_one(const ScoreArgs& a, int groups, int splits, cudaStream_t stream) {
  using F = TileFmt<kDtype>;
  using Sh = Shape<kDtype, QPC, kGather>;
  constexpr int kQS = (QPC == 1 && !kGather) ? 2 : QPC;  // query tiles held
  size_t smem = 256 * 32 * kQS + (size_t)Sh::kStages * F::kSlotBytes + (Sh::kSmemA ? (size_t)Sh::kWG * kABytes : 0);
  // one CTA per SM: its TMEM allocation may take all 512 columns
  smem = std::max<size_t>(smem, 116 * 1024);
  auto kern = score_tc_kernel<kDtype, QPC, kGather>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return launch_k(kern, dim3(splits, groups), dim3(Sh::kThreads), smem, stream, 0, a);
}

namespace {

// Grid of the scorer for queries [q0, q0 + nq): query groups sharing every
// K tile and the tile ranges (scoring CTAs) per group.
struct ScoreGrid {
  int qpc, seg, gps, groups;
  int64_t per;
  int splits;
  // one-wave flattened partition of single-query page scans: `splits` CTAs
  // over nq x tq tiles, kr_pad key-range slots per query
  bool flat;
  int64_t tq, total;
  int kr_pad;
};

ScoreGrid score_grid(const csa2_cfg& cfg, int q0, int nq, int Tq, int64_t max_entries, bool gather, int num_sms) {
  // query groups sharing every K tile: runs of 4 queries when the chunk splits
  // into them without crossing a sequence (prefill chunks); whole sequences of
  // a chunk of whole sequences otherwise (multi-query decode: up to 6 queries
  // in one group, longer blocks in groups of 4); single queries else
  ScoreGrid g{1, 1, 1, 0, 0, 0, false, 0, 0, 0};
  if (!gather && Tq % 4 == 0 && q0 % 4 == 0 && nq % 4 == 0) {
    g.qpc = 4;
    g.seg = 4;
  } else if (!gather && Tq > 1 && q0 % Tq == 0 && nq % Tq == 0) {
    g.qpc = Tq <= 6 ? 6 : 4;
    g.seg = Tq;
  }
  g.gps = (g.seg + g.qpc - 1) / g.qpc;
  g.groups = nq / g.seg * g.gps;
  const int64_t tiles = gather ? ((int64_t)cfg.hsi_blocks * kHsiBlock + 127) / 128 : (max_entries + 127) / 128;
  // CTAs per query group: one wave of one CTA per SM when there are few
  // groups (latency-bound: every CTA starts at once), else two waves for
  // balance; at least 4 tiles each
  const int waves = (g.qpc == 1 && (int64_t)g.groups * 8 > num_sms) ? 2 : 1;
  const int64_t want = std::max<int64_t>(1, (int64_t)waves * num_sms / std::max(g.groups, 1));
  const int64_t cap = gather ? kMaxGatherTiles : kMaxTilesPerCta;
  g.per = std::min<int64_t>(cap, std::max<int64_t>(4, (tiles + want - 1) / want));
  g.splits = (int)((tiles + g.per - 1) / g.per);
  g.kr_pad = g.splits;
  // Single queries: one CTA per SM over the queries' tiles laid end to end
  // instead, when that gives an SM fewer tiles (more than one wave of
  // per-query ranges, or ranges that leave SMs idle).  With at most as many
  // queries as CTAs a CTA's range (at most tq tiles) touches at most two
  // queries; each query's key-range slots are those of the CTAs over its
  // tiles, padded to the most any query has.
  const int64_t total = (int64_t)nq * tiles;
  const int64_t ctas = (int64_t)g.groups * g.splits;
  const int64_t per_sm = g.per * ((ctas + num_sms - 1) / num_sms);  // tiles of the busiest SM
  if (g.qpc == 1 && !gather && (total + num_sms - 1) / num_sms < per_sm && nq <= num_sms &&
      total >= 4 * (int64_t)num_sms && (total + num_sms - 1) / num_sms <= kMaxTilesPerCta) {
    int64_t pad = 0;
    for (int q = 0; q < nq; ++q)
      pad = std::max<int64_t>(pad, flat_cta_of((int64_t)(q + 1) * tiles - 1, total, num_sms) -
                                       flat_cta_of((int64_t)q * tiles, total, num_sms) + 1);
    if (pad <= score_range_slots(tiles)) {
      g.flat = true;
      g.tq = tiles;
      g.total = total;
      g.splits = num_sms;
      g.groups = 1;
      g.per = (total + num_sms - 1) / num_sms;
      g.kr_pad = (int)pad;
    }
  }
  return g;
}

}  // namespace

int score_slots_used(const csa2_cfg& cfg, int q0, int nq, int Tq, int64_t max_entries, bool gather, int num_sms) {
  return score_grid(cfg, q0, nq, Tq, max_entries, gather, num_sms).kr_pad;
}

cudaError_t launch_score_tc(const csa2_cfg& cfg, int q0, int nq, int Tq, const uint16_t* q_idx, const float* head_w,
                            const int64_t* q_pos, const csa2_cache& idx_c, const int32_t* n_entries,
                            int64_t max_entries, const int32_t* pool, float* scores, int64_t stride, float* bmax,
                            uint32_t* krange, int kr_stride, int* n_slots, int32_t* status, int num_sms,
                            cudaStream_t stream) {
  const bool gather = pool != nullptr;
  const ScoreGrid sg = score_grid(cfg, q0, nq, Tq, max_entries, gather, num_sms);
  const int qpc = sg.qpc, seg = sg.seg, gps = sg.gps, groups = sg.groups, splits = sg.splits;
  const int64_t per = sg.per;
  if (sg.kr_pad > kr_stride) return cudaErrorInvalidValue;
  *n_slots = sg.kr_pad;
  ScoreArgs a{q0, Tq, cfg.ratio, seg, gps, (cfg.formats & CSA2_FMT_IDX_QFP4) ? 1 : 0,
              (!gather && (int64_t)splits * groups <= num_sms) ? 1 : 0, q_idx, head_w, q_pos, view_of(idx_c),
              n_entries, max_entries, (int)per, pool, cfg.hsi_blocks, scores, stride, bmax, krange, kr_stride, status,
              sg.flat ? 1 : 0, sg.tq, sg.total, sg.kr_pad};
  if (idx_dtype(cfg) == CSA2_CACHE_FP4_S32) {
    if (gather) return launch_one<CSA2_CACHE_FP4_S32, 1, true>(a, groups, splits, stream);
    if (qpc == 6) return launch_one<CSA2_CACHE_FP4_S32, 6, false>(a, groups, splits, stream);
    return qpc == 4 ? launch_one<CSA2_CACHE_FP4_S32, 4, false>(a, groups, splits, stream)
                    : launch_one<CSA2_CACHE_FP4_S32, 1, false>(a, groups, splits, stream);
  }
  if (cfg.cache_dtype == CSA2_CACHE_FP4) {
    if (gather) return launch_one<CSA2_CACHE_FP4, 1, true>(a, groups, splits, stream);
    if (qpc == 6) return launch_one<CSA2_CACHE_FP4, 6, false>(a, groups, splits, stream);
    return qpc == 4 ? launch_one<CSA2_CACHE_FP4, 4, false>(a, groups, splits, stream)
                    : launch_one<CSA2_CACHE_FP4, 1, false>(a, groups, splits, stream);
  }
  if (gather) return launch_one<CSA2_CACHE_BF16, 1, true>(a, groups, splits, stream);
  if (qpc == 6) return launch_one<CSA2_CACHE_BF16, 6, false>(a, groups, splits, stream);
  return qpc == 4 ? launch_one<CSA2_CACHE_BF16, 4, false>(a, groups, splits, stream)
                  : launch_one<CSA2_CACHE_BF16, 1, false>(a, groups, splits, stream);
}

}  // namespace csa2
