// a3 / a5 -- indexer scores of single queries over FP4 indexer pages, with
// the work split by warp role (the long decode-time scans).
//
// s_j = sum_h w_h ReLU(q_h . K_j) (DeepSeek-V4.1 Flash, hn.213312.xyz
// sec. 2.3.1; 36kr "CSA2") for every visible entry of each query, plus the
// 8-entry block maxima of the HSI (hn.213312.xyz sec. 2.3.4).  One wave of
// CTAs shares the flattened range of (query, 128-entry tile) pairs: CTA c
// takes tiles [c T / G, (c + 1) T / G) of the T = queries x tiles-per-query
// tiles, so every SM streams the same number of pages whatever the batch,
// and a CTA's range touches at most two queries.  Inside a CTA:
//  - the producer warp copies whole pages (two per tile: FP4 codes and E4M3
//    scales) into a ring of shared-memory slots with 1-D bulk copies that
//    complete on mbarriers;
//  - three decode warpgroups take the tiles in turn: thread t decodes entry
//    t of its tile (FP4 -> f16, exact: `cvt.rn.f16x2.e2m1x2` times the
//    group's scale) into one of its warpgroup's two tensor-memory A slots;
//  - the MMA warp issues D[128 entries x 32 heads] = K_tile . Q^T into one
//    of four tensor-memory D slots as soon as an A slot is full and a D slot
//    is free (A from tensor memory, Q from shared memory, fp32 accumulate);
//  - two epilogue warpgroups read the D slots back (one entry per thread),
//    form the ReLU-weighted head sum as (sum w d + sum w |d|) / 2, which
//    keeps the FP32 work on the FMA pipe, and write the scores, the HSI
//    block maxima and this CTA's key range per query.
// Decoding, the tensor core and the epilogue of different tiles overlap;
// every wait is bounded and reports CSA2_ERR_TIMEOUT.
#include <algorithm>

#include "internal.h"
#include "score_common.cuh"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kDecWG = 3;                               // decode warpgroups
constexpr int kEpiWG = 2;                               // epilogue warpgroups
constexpr int kCtlWarp0 = 4 * (kDecWG + kEpiWG);        // first warp of the control warpgroup
constexpr int kProducerWarp = kCtlWarp0;                // TMA bulk copies
constexpr int kMmaWarp = kCtlWarp0 + 1;                 // tcgen05.mma issue (and TMEM owner)
constexpr int kThreads = 32 * (kCtlWarp0 + 4);          // 768
constexpr int kASlots = 2;                              // A slots per decode warpgroup
constexpr int kDSlots = 4;
constexpr int kAcols = 64;                              // 128 f16 channels per entry
constexpr int kDcols = 32;                              // 32 heads
constexpr int kTmemCols = 512;
static_assert(kDecWG * kASlots * kAcols + kDSlots * kDcols <= kTmemCols, "tensor-memory budget");
constexpr int kStages = 16;                             // ring slots (one tile = two pages each)
constexpr int kMaxTiles = 1024;                         // tiles of one CTA (page table in shared memory)
constexpr int kQBytes = kIdxHeads * kIdxDim * 2;        // one query's f16 tile, 8 KB

template <int kDtype>
struct Fmt {
  static constexpr int kPageData = kIdxFp4Data;
  static constexpr int kPageScales = kDtype == CSA2_CACHE_FP4 ? kIdxFp4Scales : kIdxS32Scales;
  static constexpr int kSlot = 2 * (kPageData + kPageScales);
};

struct WsArgs {
  int q0, nq, Tq, r;
  int q_fp4;
  int prefetch;          // bring the first ring pass into L2 before the wait on the previous kernel
  const uint16_t* q_idx;
  const float* head_w;
  const int64_t* q_pos;
  CacheView ic;
  const int32_t* n_entries;
  int64_t max_entries;
  int64_t tq;            // tiles per query: ceil(max_entries / 128)
  int64_t total;         // nq * tq
  float* scores;         // [nq][stride]
  int64_t stride;
  float* bmax;           // [nq][ceil(max_entries / 8)] or null
  uint32_t* krange;      // [nq][kr_stride][2]
  int kr_stride;
  int32_t* status;
};

__device__ __forceinline__ int64_t first_tile(int64_t c, int64_t total, int64_t grid) { return c * total / grid; }

// CTA of the flattened range holding global tile x (the largest c with
// first_tile(c) <= x).
__device__ __forceinline__ int64_t cta_of(int64_t x, int64_t total, int64_t grid) {
  return ((x + 1) * grid - 1) / total;
}

template <int kDtype>
__global__ void __launch_bounds__(kThreads, 1) score_ws_kernel(WsArgs a) {
  using F = Fmt<kDtype>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t G = gridDim.x, c = blockIdx.x;
  const int64_t gt0 = first_tile(c, a.total, G), gt1 = first_tile(c + 1, a.total, G);
  const int qa = (int)(gt0 / a.tq);
  const bool two = gt1 > (int64_t)(qa + 1) * a.tq;  // the range reaches into the next query
  if (a.prefetch && warp == kProducerWarp) {
    // While the previous kernel (the compressor) runs: the pages of the first
    // ring pass into L2.  Hints only; the block-table entries read to aim
    // them are read again after the wait, and every page lies in the pool.
    const int64_t gt = gt0 + lane / 2;
    const int gq = a.q0 + (int)(gt / a.tq);
    const int64_t pp = 2 * (gt % a.tq) + (lane & 1);
    if (lane < 2 * kStages && gt < gt1 && pp < a.ic.max_pages && pp * kPage < a.max_entries) {
      const int32_t pg = tc::ld_cg_s32(a.ic.block_table + (int64_t)(gq / a.Tq) * a.ic.max_pages + pp);
      if (pg >= 0 && pg < a.ic.num_pages) {
        tc::bulk_prefetch_l2(a.ic.data + (int64_t)pg * F::kPageData, F::kPageData);
        tc::bulk_prefetch_l2(a.ic.scales + (int64_t)pg * F::kPageScales, F::kPageScales);
      }
    }
  }
  griddep_wait();  // before any other global read or tensor-memory allocation
  griddep_launch();

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* qtile = smem;                                   // [2 queries][32 heads x 128] f16, K-major
  uint8_t* ring = smem + 2 * kQBytes;                      // kStages slots
  int32_t* ptab = reinterpret_cast<int32_t*>(ring + kStages * F::kSlot);  // [tile][2] page ids
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ __align__(8) uint64_t afull[kDecWG][kASlots], aempty[kDecWG][kASlots];
  __shared__ __align__(8) uint64_t dfull[kDSlots], dempty[kDSlots], drain_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float hw[2][kIdxHeads];
  __shared__ uint32_t rng_lo[2], rng_hi[2];

  // this CTA's queries (chunk-local qa and qa + 1), their visible entries and
  // the active tiles: query qa's tiles ta0 .. ta0 + ka - 1, then query qa + 1's
  // tiles 0 .. kb - 1 (tiles past a query's visible entries are skipped)
  auto visible = [&](int gq) {
    const int64_t ne = a.n_entries[gq / a.Tq] < a.max_entries ? a.n_entries[gq / a.Tq] : a.max_entries;
    return visible_entries(a.q_pos[gq], a.r, ne);
  };
  const int64_t nv0 = visible(a.q0 + qa), nv1 = two ? visible(a.q0 + qa + 1) : 0;
  const int64_t ta0 = gt0 - (int64_t)qa * a.tq;
  const int64_t na = (two ? (int64_t)(qa + 1) * a.tq : gt1) - gt0;
  const int64_t nb = two ? gt1 - (int64_t)(qa + 1) * a.tq : 0;
  const int64_t tva = (nv0 + 127) / 128, tvb = (nv1 + 127) / 128;
  const int ka = (int)std::min<int64_t>(na, std::max<int64_t>(0, tva - ta0));
  const int kb = (int)std::min<int64_t>(nb, tvb);
  const int n_act = ka + kb;
  auto tile_q = [&](int k) { return k < ka ? 0 : 1; };
  auto tile_t = [&](int k) -> int64_t { return k < ka ? ta0 + k : (int64_t)(k - ka); };

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 128);
    }
    for (int g = 0; g < kDecWG; ++g)
      for (int j = 0; j < kASlots; ++j) {
        tc::mbar_init(&afull[g][j], 128);
        tc::mbar_init(&aempty[g][j], 1);
      }
    for (int d = 0; d < kDSlots; ++d) {
      tc::mbar_init(&dfull[d], 1);
      tc::mbar_init(&dempty[d], 128);
    }
    tc::mbar_init(&drain_bar, 1);
    abort_flag = 0;
    rng_lo[0] = rng_lo[1] = 0xFFFFFFFFu;
    rng_hi[0] = rng_hi[1] = 0u;
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  // pages of the active tiles, the query tiles and the head weights
  for (int i = tid; i < 2 * n_act; i += kThreads) {
    const int k = i >> 1, h = i & 1;
    const int j = tile_q(k);
    const int64_t p = 2 * tile_t(k) + h;  // logical page of the query's sequence
    const int gq = a.q0 + qa + j;
    ptab[i] = (p * kPage < (j ? nv1 : nv0)) ? (int32_t)page_of(a.ic, gq / a.Tq, p * kPage, a.status) : -1;
  }
  {
    // 2 x 512 pieces of 8 channels; lanes 2m and 2m + 1 share one 16-channel
    // group (the FP4-query encoding's shuffle), and every thread runs both
    // rounds
    constexpr int kPieces = 2 * kIdxHeads * kIdxDim / 8;
    for (int i0 = 0; i0 < kPieces; i0 += kThreads) {
      const int i = i0 + tid;
      const int j = i / (kPieces / 2), row = (8 * (i % (kPieces / 2))) / kIdxDim, kk = (8 * i) % kIdxDim;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      const bool have = i < kPieces && (j == 0 || two);
      if (have)
        v = __ldg(reinterpret_cast<const uint4*>(a.q_idx + ((int64_t)(a.q0 + qa + j) * kIdxHeads + row) * kIdxDim + kk));
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
      if (score::q_operand8<false>(w, a.q_fp4 != 0) && have) report(a.status, CSA2_ERR_RANGE);
      if (i < kPieces)
        *reinterpret_cast<uint4*>(qtile + j * kQBytes + tc::kmajor_off(row, kk, kIdxDim)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  if (tid < 2 * kIdxHeads) {
    const int j = tid / kIdxHeads, h = tid % kIdxHeads;
    hw[j][h] = (a.head_w && (j == 0 || two)) ? __ldg(a.head_w + (int64_t)(a.q0 + qa + j) * kIdxHeads + h) : 1.0f;
  }
  tc::fence_async_smem();  // the query tiles are read by the tensor core
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = tmem_base;
  auto aborted = [&] { return *reinterpret_cast<volatile int*>(&abort_flag) != 0; };
  auto fail = [&] {
    report(a.status, CSA2_ERR_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };

  // roles: decode warpgroups (warps 0..11), epilogue warpgroups (12..19), the
  // producer and MMA warps; the control warpgroup's last two warps only join
  // the final barrier
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int k = 0; k < n_act; ++k) {
        const int s = k % kStages;
        if (k >= kStages && !tc::mbar_wait(&empty_bar[s], ((k / kStages) & 1) ^ 1)) {
          fail();
          break;
        }
        if (aborted()) break;
        uint8_t* slot = ring + (size_t)s * F::kSlot;
        const int32_t p0 = ptab[2 * k], p1 = ptab[2 * k + 1];
        const uint32_t bytes = (p0 >= 0 ? F::kPageData + F::kPageScales : 0) + (p1 >= 0 ? F::kPageData + F::kPageScales : 0);
        tc::mbar_arrive_expect_tx(&full_bar[s], bytes);
        if (p0 >= 0) {
          tc::bulk_g2s(slot, a.ic.data + (int64_t)p0 * F::kPageData, F::kPageData, &full_bar[s]);
          tc::bulk_g2s(slot + 2 * F::kPageData, a.ic.scales + (int64_t)p0 * F::kPageScales, F::kPageScales,
                       &full_bar[s]);
        }
        if (p1 >= 0) {
          tc::bulk_g2s(slot + F::kPageData, a.ic.data + (int64_t)p1 * F::kPageData, F::kPageData, &full_bar[s]);
          tc::bulk_g2s(slot + 2 * F::kPageData + F::kPageScales, a.ic.scales + (int64_t)p1 * F::kPageScales,
                       F::kPageScales, &full_bar[s]);
        }
        ++issued;
      }
      // no copy into this CTA's shared memory outlives it
      for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
        if (!tc::mbar_wait(&full_bar[k % kStages], (k / kStages) & 1)) report(a.status, CSA2_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    constexpr uint32_t kIdesc = tc::idesc_f16(128, kDcols, false, false, false, false);
    int issued = 0;
    if (lane == 0) {
      for (int k = 0; k < n_act; ++k) {
        const int g = k % kDecWG, u = k / kDecWG, j = u % kASlots, d = k % kDSlots;
        if (!tc::mbar_wait(&afull[g][j], (u / kASlots) & 1)) {
          fail();
          break;
        }
        if (k >= kDSlots && !tc::mbar_wait(&dempty[d], ((k / kDSlots) & 1) ^ 1)) {
          fail();
          break;
        }
        if (aborted()) break;
        tc::fence_after_sync();
        const uint32_t qbase = tc::smem_u32(qtile + tile_q(k) * kQBytes);
        const uint32_t acol = (uint32_t)((g * kASlots + j) * kAcols);
        const uint32_t dcol = (uint32_t)(kDecWG * kASlots * kAcols + d * kDcols);
#pragma unroll
        for (int ks = 0; ks < kIdxDim / 16; ++ks)
          tc::mma_ts(tb + dcol, tb + acol + ks * 8, tc::sdesc(qbase + ks * 256, 128, kIdxDim * 16), kIdesc, ks > 0);
        tc::mma_commit(&aempty[g][j]);
        tc::mma_commit(&dfull[d]);
        ++issued;
      }
      // every issued MMA has completed before tensor memory is released
      tc::mma_commit(&drain_bar);
      if (!tc::mbar_wait(&drain_bar, 0)) report(a.status, CSA2_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp < 4 * kDecWG) {
    // -------------------------------------------------------------- decode
    const int g = warp >> 2;
    const int lt = 32 * (warp & 3) + lane;        // entry of the tile, TMEM lane
    const int h = lt >> 6, sl = lt & 63;          // its page of the tile, slot of the page
    const uint32_t lane_base = 32u * (warp & 3);
    for (int k = g, u = 0; k < n_act; k += kDecWG, ++u) {
      const int s = k % kStages, j = u % kASlots;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&full_bar[s], (k / kStages) & 1)) && lane == 0) fail();
      if (__any_sync(0xffffffffu, aborted())) break;  // uniform in the warp: tcgen05.st is warp-wide
      const uint8_t* slot = ring + (size_t)s * F::kSlot;
      uint4 cw[4];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        cw[cc] = *reinterpret_cast<const uint4*>(slot + h * F::kPageData + (cc * kPage + sl) * 16);
      uint2 sc;
      if (kDtype == CSA2_CACHE_FP4)
        sc = *reinterpret_cast<const uint2*>(slot + 2 * F::kPageData + h * F::kPageScales + sl * 8);
      else
        sc = make_uint2(*reinterpret_cast<const uint32_t*>(slot + 2 * F::kPageData + h * F::kPageScales + sl * 4), 0u);
      tc::mbar_arrive(&empty_bar[s]);
      // the scales as broadcast f16x2: s2g[x] for 16-channel group x (or
      // 32-channel group x with one scale per 32 channels)
      uint32_t s2g[8];
      score::e4m3_pair_bcast(sc.x, s2g[0], s2g[1]);
      score::e4m3_pair_bcast(sc.x >> 16, s2g[2], s2g[3]);
      if (kDtype == CSA2_CACHE_FP4) {
        score::e4m3_pair_bcast(sc.y, s2g[4], s2g[5]);
        score::e4m3_pair_bcast(sc.y >> 16, s2g[6], s2g[7]);
      }
      // the A slot is free once the MMA that read it two tiles ago is done
      if (u >= kASlots && !__all_sync(0xffffffffu, tc::mbar_wait(&aempty[g][j], ((u / kASlots) & 1) ^ 1))) {
        if (lane == 0) fail();
        break;
      }
      tc::fence_after_sync();
      const uint32_t acol = (uint32_t)((g * kASlots + j) * kAcols);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {  // 32 channels -> 16 TMEM columns
        const uint32_t w4[4] = {cw[cc].x, cw[cc].y, cw[cc].z, cw[cc].w};
        uint32_t r16[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t s2 = kDtype == CSA2_CACHE_FP4 ? s2g[2 * cc + (q >> 1)] : s2g[cc];
          uint32_t h4[4];
          score::e2m1x8_to_f16x2(w4[q], h4);
#pragma unroll
          for (int by = 0; by < 4; ++by) r16[q * 4 + by] = score::hmul2(h4[by], s2);
        }
        tc::tmem_st16(tc::taddr(tb, lane_base, acol + 16 * cc), r16);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive(&afull[g][j]);
    }
  } else if (warp < kCtlWarp0) {
    // ------------------------------------------------------------ epilogue
    const int e = (warp >> 2) - kDecWG;
    const int lt = 32 * (warp & 3) + lane;
    const uint32_t lane_base = 32u * (warp & 3);
    uint32_t klo0 = 0xFFFFFFFFu, klo1 = 0xFFFFFFFFu, khi0 = 0u, khi1 = 0u;
    const bool weighted = a.head_w != nullptr;
    for (int k = e; k < n_act; k += kEpiWG) {
      const int d = k % kDSlots;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&dfull[d], (k / kDSlots) & 1)) && lane == 0) fail();
      if (__any_sync(0xffffffffu, aborted())) break;  // uniform in the warp: tcgen05.ld is warp-wide
      tc::fence_after_sync();
      uint32_t v[32];
      tc::tmem_ld32(tc::taddr(tb, lane_base, (uint32_t)(kDecWG * kASlots * kAcols + d * kDcols)), v);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      tc::mbar_arrive(&dempty[d]);
      const int j = tile_q(k);
      const int64_t pos = tile_t(k) * 128 + lt;
      const bool valid = pos < (j ? nv1 : nv0);
      // sum_h w_h ReLU(d_h) = (sum_h w_h d_h + sum_h w_h |d_h|) / 2, as two
      // sums of four partial sums each (FMA-pipe adds only)
      float p[4] = {0.0f, 0.0f, 0.0f, 0.0f}, m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (weighted) {
#pragma unroll
        for (int hh = 0; hh < kIdxHeads; ++hh) {
          const float x = __uint_as_float(v[hh]), wv = j ? hw[1][hh] : hw[0][hh];
          p[hh & 3] = fmaf(wv, x, p[hh & 3]);
          m[hh & 3] = fmaf(wv, fabsf(x), m[hh & 3]);
        }
      } else {
#pragma unroll
        for (int hh = 0; hh < kIdxHeads; ++hh) {
          const float x = __uint_as_float(v[hh]);
          p[hh & 3] += x;
          m[hh & 3] += fabsf(x);
        }
      }
      const float sp = (p[0] + p[1]) + (p[2] + p[3]), sm = (m[0] + m[1]) + (m[2] + m[3]);
      const float sc = 0.5f * (sp + sm);
      if (valid) {
        a.scores[(int64_t)(qa + j) * a.stride + pos] = sc;
        const uint32_t kk = order_key(sc);
        if (j) {
          klo1 = min(klo1, kk);
          khi1 = max(khi1, kk);
        } else {
          klo0 = min(klo0, kk);
          khi0 = max(khi0, kk);
        }
      }
      if (a.bmax) {
        float mx = valid ? sc : -INFINITY;
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        if ((lt & 7) == 0 && valid) a.bmax[(int64_t)(qa + j) * ((a.max_entries + 7) / 8) + pos / 8] = mx;
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t lo = j ? klo1 : klo0, hi = j ? khi1 : khi0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      }
      if (lane == 0 && lo <= hi) {
        atomicMin(&rng_lo[j], lo);
        atomicMax(&rng_hi[j], hi);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kMmaWarp) tc::tmem_dealloc(tb, kTmemCols);
  // this CTA's slot of each query it touched: slot c - (first CTA of the query)
  if (tid < 2 && (tid == 0 || two)) {
    const int j = tid;
    const int64_t c0 = cta_of((int64_t)(qa + j) * a.tq, a.total, G);
    uint32_t* kr = a.krange + ((int64_t)(qa + j) * a.kr_stride + (c - c0)) * 2;
    kr[0] = rng_lo[j];
    kr[1] = rng_hi[j];
  }
}

}  // namespace

bool score_ws_usable(const csa2_cfg& cfg, int nq, int64_t max_entries, int num_sms, int* grid) {
  const int dt = idx_dtype(cfg);
  if (dt != CSA2_CACHE_FP4 && dt != CSA2_CACHE_FP4_S32) return false;
  const int64_t tq = (max_entries + 127) / 128;
  if (nq < 1 || nq > num_sms || tq < 1) return false;
  const int64_t total = (int64_t)nq * tq;
  // one wave, at least one CTA per query (so a CTA's range touches at most
  // two queries), about eight tiles per CTA at least
  const int64_t g = std::max<int64_t>(nq, std::min<int64_t>(num_sms, total / 8));
  if ((total + g - 1) / g > kMaxTiles) return false;
  *grid = (int)g;
  return true;
}

cudaError_t launch_score_ws(const csa2_cfg& cfg, int q0, int nq, int Tq, const uint16_t* q_idx, const float* head_w,
                            const int64_t* q_pos, const csa2_cache& idx_c, const int32_t* n_entries,
                            int64_t max_entries, float* scores, int64_t stride, float* bmax, uint32_t* krange,
                            int kr_stride, int grid, int32_t* status, cudaStream_t stream) {
  const int64_t tq = (max_entries + 127) / 128;
  WsArgs a{q0, nq, Tq, cfg.ratio, (cfg.formats & CSA2_FMT_IDX_QFP4) ? 1 : 0, 1, q_idx, head_w, q_pos, view_of(idx_c),
           n_entries, max_entries, tq, (int64_t)nq * tq, scores, stride, bmax, krange, kr_stride, status};
  const int dt = idx_dtype(cfg);
  if (dt == CSA2_CACHE_FP4) {
    const size_t smem = 2 * kQBytes + (size_t)kStages * Fmt<CSA2_CACHE_FP4>::kSlot + 2 * kMaxTiles * 4;
    auto kern = score_ws_kernel<CSA2_CACHE_FP4>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_k(kern, dim3(grid), dim3(kThreads), smem, stream, 0, a);
  }
  const size_t smem = 2 * kQBytes + (size_t)kStages * Fmt<CSA2_CACHE_FP4_S32>::kSlot + 2 * kMaxTiles * 4;
  auto kern = score_ws_kernel<CSA2_CACHE_FP4_S32>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return launch_k(kern, dim3(grid), dim3(kThreads), smem, stream, 0, a);
}

}  // namespace csa2
