// a3 / a5 -- CSA2 indexer scores on the tensor cores (Full mode).
//
// s_j = sum_h w_h ReLU(q_h . K_j) over the visible indexer-K entries
// (DeepSeek-V4.1 Flash, hn.213312.xyz sec. 2.3.1; 36kr "CSA2").  Per CTA: a
// range of 128-entry tiles of one group of QPC queries of one sequence.
//  - warp 4 (one elected lane) streams whole cache pages into a shared-memory
//    ring with 1-D bulk copies (two pages = one tile; mbarrier completion);
//  - warps 0-3 (thread t <-> entry t of the tile <-> TMEM lane t) decode their
//    entry (FP4 -> f16, exact; bf16 kept) straight into TMEM as the A operand;
//  - thread 0 issues tcgen05.mma: D[128 entries x 32*QPC] += K_tile . Q^T with
//    A from TMEM and Q_idx (f16 / bf16) from shared memory;
//  - the epilogue reads D back (one row per thread), forms the ReLU-weighted
//    head sums, writes the scores and the 8-entry block maxima for HSI.
// A and D are double-buffered in TMEM so that the MMA of tile i overlaps the
// epilogue of tile i-1 and the decode of tile i+1.  Every wait is bounded.
#include <algorithm>

#include "internal.h"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kConsumers = 128;
constexpr int kThreads = kConsumers + 32;
constexpr uint32_t kSpin = 1u << 26;
constexpr int kMaxTilesPerCta = 512;

template <int kDtype>
struct TileFmt {
  static constexpr int kPageData = (kDtype == CSA2_CACHE_FP4) ? kIdxFp4Data : kIdxBf16Data;
  static constexpr int kPageScales = (kDtype == CSA2_CACHE_FP4) ? kIdxFp4Scales : 0;
  static constexpr int kSlotBytes = 2 * (kPageData + kPageScales);
  static constexpr int kStages = (kDtype == CSA2_CACHE_FP4) ? 4 : 2;
};

struct ScoreArgs {
  int q0, Tq, r;
  const uint16_t* q_idx;
  const float* head_w;
  const int64_t* q_pos;
  CacheView ic;
  const int32_t* n_entries;
  int64_t max_entries;
  int tiles_per_cta;
  float* scores;   // [chunk][max_entries]
  float* bmax;     // [chunk][ceil(max_entries/8)] or null
  uint32_t* kmin;  // [chunk] key range of each query's scores
  uint32_t* kmax;
  int32_t* status;
};

__device__ __forceinline__ uint32_t f16x2_scale(uint32_t sbyte) {
  uint32_t r;
  uint16_t pair = (uint16_t)(sbyte | (sbyte << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(pair));
  return r;
}

// Four bytes of packed E2M1 pairs -> four f16x2 (element 2i of a byte in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ void named_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

template <int kDtype, int QPC>
__global__ void __launch_bounds__(kThreads) score_tc_kernel(ScoreArgs a) {
  using F = TileFmt<kDtype>;
  constexpr int kN = 32 * QPC;                    // MMA N: QPC queries x 32 heads
  constexpr int kAcols = 64;                      // 128 channels of f16 pairs
  constexpr int kTmemCols = (2 * kAcols + 2 * kN) <= 256 ? 256 : 512;
  constexpr int S = F::kStages;
  constexpr bool kBf16 = (kDtype == CSA2_CACHE_BF16);
  constexpr uint32_t kIdesc = tc::idesc_f16(128, kN, kBf16, kBf16, false, false);

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* qtile = smem;                                   // [kN rows][128] K-major, 256*kN B
  uint8_t* ring = smem + 256 * kN;                         // S slots
  __shared__ float hw[QPC][kIdxHeads];
  __shared__ __align__(8) uint64_t full_bar[S], empty_bar[S], mma_bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int32_t ptab[2 * kMaxTilesPerCta];  // resolved pages of this CTA's tiles

  const int tid = threadIdx.x, warp = tid >> 5;
  const int g0 = a.q0 + blockIdx.y * QPC;   // first query of the group (same sequence)
  const int b = g0 / a.Tq;
  int64_t nv[QPC];
  int64_t nv_max = 0;
#pragma unroll
  for (int q = 0; q < QPC; ++q) {
    const int64_t ne = a.n_entries[b] < a.max_entries ? a.n_entries[b] : a.max_entries;
    nv[q] = visible_entries(a.q_pos[g0 + q], a.r, ne);
    nv_max = nv[q] > nv_max ? nv[q] : nv_max;
  }
  const int64_t n_tiles = (nv_max + 127) / 128;
  const int64_t t_begin = (int64_t)blockIdx.x * a.tiles_per_cta;
  const int64_t t_end = t_begin + a.tiles_per_cta < n_tiles ? t_begin + a.tiles_per_cta : n_tiles;
  if (t_begin >= t_end) return;  // uniform: the whole CTA leaves before any barrier
  const int n_my = (int)(t_end - t_begin);

  // ---- set-up: Q_idx (f16 or bf16) into the B tile, head weights, barriers, TMEM
  for (int i = tid; i < kN * kIdxDim / 8; i += kThreads) {
    const int row = (8 * i) / kIdxDim, k = (8 * i) % kIdxDim;  // row = q*32 + h; 8 channels per load
    uint4 v = __ldg(reinterpret_cast<const uint4*>(a.q_idx + (int64_t)(g0 + row / kIdxHeads) * kIdxHeads * kIdxDim +
                                                   (row % kIdxHeads) * kIdxDim + k));
    if (!kBf16) {
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h2 = __floats2half2_rn(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
        w[j] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4*>(qtile + tc::kmajor_off(row, k, kIdxDim)) = v;
  }
  for (int i = tid; i < QPC * kIdxHeads; i += kThreads)
    hw[i / kIdxHeads][i % kIdxHeads] = a.head_w ? __ldg(a.head_w + (int64_t)g0 * kIdxHeads + i) : 1.0f;
  for (int i = tid; i < 2 * n_my; i += kThreads) {
    const int64_t p = 2 * t_begin + i;  // logical page
    ptab[i] = (p * kPage < nv_max) ? (int32_t)page_of(a.ic, b, p * kPage, a.status) : -1;
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], kConsumers);
    }
    tc::mbar_init(&mma_bar[0], 1);
    tc::mbar_init(&mma_bar[1], 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = tmem_base;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if ((tid & 31) == 0) {
      int issued = 0;
      for (int i = 0; i < n_my; ++i) {
        const int s = i % S;
        if (!tc::mbar_wait(&empty_bar[s], ((i / S) & 1) ^ 1, kSpin)) {
          report(a.status, CSA2_ERR_TIMEOUT);
          atomicExch(&abort_flag, 1);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
        uint8_t* slot = ring + (size_t)s * F::kSlotBytes;
        uint32_t bytes = 0;
        int64_t pages[2] = {-1, -1};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          pages[h] = ptab[2 * i + h];
          if (pages[h] >= 0) bytes += F::kPageData + F::kPageScales;
        }
        tc::mbar_arrive_expect_tx(&full_bar[s], bytes);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (pages[h] < 0) continue;
          tc::bulk_g2s(slot + h * F::kPageData, a.ic.data + pages[h] * F::kPageData, F::kPageData, &full_bar[s]);
          if (F::kPageScales)
            tc::bulk_g2s(slot + 2 * F::kPageData + h * F::kPageScales, a.ic.scales + pages[h] * F::kPageScales,
                         F::kPageScales, &full_bar[s]);
        }
        ++issued;
      }
      // do not leave while copies into this CTA's shared memory are in flight
      for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
        if (!tc::mbar_wait(&full_bar[i % S], (i / S) & 1, kSpin)) report(a.status, CSA2_ERR_TIMEOUT);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int lane_base = 32 * warp;  // TMEM lanes of this warp
  int i = 0;
  int last_issued = -1, waited = -1;
  uint32_t klo[QPC], khi[QPC];
#pragma unroll
  for (int q = 0; q < QPC; ++q) {
    klo[q] = 0xFFFFFFFFu;
    khi[q] = 0u;
  }
  for (; i <= n_my; ++i) {
    if (i < n_my) {
      const int s = i % S;
      const bool ok = tc::mbar_wait(&full_bar[s], (i / S) & 1, kSpin);
      if (!ok) atomicExch(&abort_flag, 1);
      uint32_t av[64];
      const uint8_t* slot = ring + (size_t)s * F::kSlotBytes;
      const int h = tid >> 6, sl = tid & 63;
      if (kDtype == CSA2_CACHE_FP4) {
        uint4 cw[4];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          cw[c] = *reinterpret_cast<const uint4*>(slot + h * kIdxFp4Data + (c * kPage + sl) * 16);
        const uint2 sc = *reinterpret_cast<const uint2*>(slot + 2 * kIdxFp4Data + h * kIdxFp4Scales + sl * 8);
        tc::mbar_arrive(&empty_bar[s]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t w4[4] = {cw[c].x, cw[c].y, cw[c].z, cw[c].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int g = 2 * c + (q >> 1);  // 16-channel group of these 8 channels
            const uint32_t sb = ((g < 4 ? sc.x : sc.y) >> (8 * (g & 3))) & 0xFFu;
            const uint32_t s2 = f16x2_scale(sb);
            uint32_t h4[4];
            e2m1x8_to_f16x2(w4[q], h4);
#pragma unroll
            for (int by = 0; by < 4; ++by) av[c * 16 + q * 4 + by] = hmul2(h4[by], s2);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(slot + h * kIdxBf16Data + (c * kPage + sl) * 16);
          av[4 * c] = v.x;
          av[4 * c + 1] = v.y;
          av[4 * c + 2] = v.z;
          av[4 * c + 3] = v.w;
        }
        tc::mbar_arrive(&empty_bar[s]);
      }
      const uint32_t acol = (uint32_t)((i & 1) * kAcols);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r16[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) r16[j] = av[16 * c + j];
        tc::tmem_st16(tc::taddr(tb, lane_base, acol + 16 * c), r16);
      }
      tc::tmem_wait_st();
    }
    tc::fence_before_sync();
    named_sync();
    tc::fence_after_sync();
    if (*reinterpret_cast<volatile int*>(&abort_flag)) break;  // uniform after the barrier
    if (i < n_my && tid == 0) {
      const uint32_t acol = (uint32_t)((i & 1) * kAcols);
      const uint32_t dcol = (uint32_t)(2 * kAcols + (i & 1) * kN);
#pragma unroll
      for (int ks = 0; ks < kIdxDim / 16; ++ks) {
        const uint64_t bdesc = tc::sdesc(tc::smem_u32(qtile) + ks * 256, 128, kIdxDim * 16);
        tc::mma_ts(tb + dcol, tb + acol + ks * 8, bdesc, kIdesc, ks > 0);
      }
      tc::mma_commit(&mma_bar[i & 1]);
    }
    if (i < n_my) last_issued = i;
    if (i >= 1) {
      // epilogue of tile i-1
      const int e = i - 1;
      const bool ok = tc::mbar_wait(&mma_bar[e & 1], (e >> 1) & 1, kSpin);
      waited = e;
      if (!ok) {
        report(a.status, CSA2_ERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
      tc::fence_after_sync();
      const int64_t j = (t_begin + e) * 128 + tid;
      const uint32_t dcol = (uint32_t)(2 * kAcols + (e & 1) * kN);
#pragma unroll
      for (int q = 0; q < QPC; ++q) {
        uint32_t d[32];
        tc::tmem_ld32(tc::taddr(tb, lane_base, dcol + 32 * q), d);
        tc::tmem_wait_ld();
        float s = 0.0f;
#pragma unroll
        for (int hh = 0; hh < kIdxHeads; ++hh) s = fmaf(hw[q][hh], fmaxf(__uint_as_float(d[hh]), 0.0f), s);
        s += 0.0f;
        if (j >= nv[q] || !ok) s = -INFINITY;
        const int qc = blockIdx.y * QPC + q;
        if (j < nv[q]) {
          a.scores[(int64_t)qc * a.max_entries + j] = s;
          const uint32_t kk = order_key(s);
          klo[q] = min(klo[q], kk);
          khi[q] = max(khi[q], kk);
        }
        if (a.bmax) {
          float m = s;
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((tid & 7) == 0 && j < nv[q]) a.bmax[(int64_t)qc * ((a.max_entries + 7) / 8) + j / 8] = m;
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < QPC; ++q)
    fold_key_range(klo[q], khi[q], a.kmin + blockIdx.y * QPC + q, a.kmax + blockIdx.y * QPC + q);
  // after an abort, let the last issued MMAs finish before TMEM is released
  if (last_issued > waited) {
    if (!tc::mbar_wait(&mma_bar[last_issued & 1], (last_issued >> 1) & 1, kSpin)) report(a.status, CSA2_ERR_TIMEOUT);
  }
  tc::fence_before_sync();
  named_sync();
  if (warp == 0) tc::tmem_dealloc(tb, kTmemCols);
}

}  // namespace

template <int kDtype, int QPC>
static cudaError_t launch_one(const ScoreArgs& a, int groups, int splits, cudaStream_t stream) {
  using F = TileFmt<kDtype>;
  size_t smem = 256 * 32 * QPC + (size_t)F::kStages * F::kSlotBytes;
  // at most two CTAs per SM: their TMEM (256 columns each) then always fits
  const size_t min_smem = (QPC == 1) ? 80 * 1024 : 120 * 1024;
  if (smem < min_smem) smem = min_smem;
  auto kern = score_tc_kernel<kDtype, QPC>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  kern<<<dim3(splits, groups), kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_score_tc(const csa2_cfg& cfg, int q0, int nq, int Tq, const uint16_t* q_idx, const float* head_w,
                            const int64_t* q_pos, const csa2_cache& idx_c, const int32_t* n_entries,
                            int64_t max_entries, float* scores, float* bmax, uint32_t* kmin, uint32_t* kmax,
                            int32_t* status, int num_sms, cudaStream_t stream) {
  const int qpc = (Tq % 4 == 0 && q0 % 4 == 0 && nq % 4 == 0) ? 4 : 1;
  const int groups = nq / qpc;
  const int64_t tiles = (max_entries + 127) / 128;
  // enough CTAs for a few waves, at least 4 tiles each
  const int64_t want = std::max<int64_t>(1, (int64_t)(qpc == 1 ? 4 : 2) * num_sms / std::max(groups, 1));
  int64_t per = std::min<int64_t>(kMaxTilesPerCta, std::max<int64_t>(4, (tiles + want - 1) / want));
  const int splits = (int)((tiles + per - 1) / per);
  ScoreArgs a{q0, Tq, cfg.ratio, q_idx, head_w, q_pos, view_of(idx_c), n_entries, max_entries, (int)per,
              scores, bmax, kmin, kmax, status};
  if (cfg.cache_dtype == CSA2_CACHE_FP4)
    return qpc == 4 ? launch_one<CSA2_CACHE_FP4, 4>(a, groups, splits, stream)
                    : launch_one<CSA2_CACHE_FP4, 1>(a, groups, splits, stream);
  return qpc == 4 ? launch_one<CSA2_CACHE_BF16, 4>(a, groups, splits, stream)
                  : launch_one<CSA2_CACHE_BF16, 1>(a, groups, splits, stream);
}

}  // namespace csa2
