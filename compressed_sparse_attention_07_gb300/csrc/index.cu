// a3..a6 -- CSA2 lightweight indexer: per-query scores over the visible
// indexer-K entries (or over an HSI pool), HSI block maxima, and exact
// top-k selection with the (score desc, id asc) order.
// (DeepSeek-V4.1 Flash, hn.213312.xyz sec. 2.3.1, 2.3.2, 2.3.4; 36kr "CSA2".)
// The selection kernel holds a query's keys in registers when they fit one
// CTA (up to 32768 positions, 16 or 32 keys a thread), stages them through
// shared memory in rounds otherwise, with a sampled one-pass variant for
// very long rows and clusters of CTAs when few queries leave SMs idle;
// every variant gives the same exact result.
#include <algorithm>

#include "internal.h"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kSelThreads = 1024;   // one CTA (or a cluster of them) selects for one query
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kPer = 16;              // keys a thread holds per round
constexpr int kRound = kSelThreads * kPer;  // positions per round
constexpr int kHistBins = 8192;       // linear bins over a query's key range
constexpr int kDigitBins = 2048;      // refinement digit: 11 bits
constexpr int kCandMax = 8192;        // keys of the threshold bin listed in shared memory

// ---------------------------------------------------------------- select ----

constexpr int kMinCtaKeys = kRound;  // positions per CTA of a selection cluster, at least
                                     // (below that the cluster's merges cost more than they save)
constexpr int kRankMax = 512;  // threshold-bin candidates ranked directly (else refined by digits)
static_assert(kCandMax <= kHistBins, "one CTA keeps the listed keys' positions in the cluster histogram's space");

struct SelShared {
  uint32_t keys[kRound];       // this CTA's keys of the current round (slots: kslot)
  uint32_t hist[kHistBins];    // this CTA's histogram (the cluster's peers read it)
  uint32_t merged[kHistBins];  // the cluster's histogram; one CTA: positions of the threshold-bin keys
  uint32_t cand[kCandMax];     // this CTA's keys of the threshold bin, minus kmin (peers read them)
  uint32_t all[kRankMax];      // the cluster's threshold-bin keys; one CTA: positions above the bin
  uint32_t part[kSelThreads];  // bin sums per thread (find_cut); rank counts per candidate
  uint32_t wsum[kSelWarps + 1];
  uint32_t cut_bin, cut_above, cut_total, cand_n, c_all, t_x, t_krem, carry_eq, carry_gt, grand;
  uint32_t tot_gt, tot_eq;     // this CTA's counts for the compaction (peers read them)
  uint32_t above_n;
  uint32_t peer_off[9];
};

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// id emitted for position p
struct IdMap {
  const int32_t* pool;  // Reindex: pool row of this query; NULL: id = p
  __device__ __forceinline__ int32_t operator()(int64_t p) const {
    return pool ? pool[p / kHsiBlock] * kHsiBlock + (int32_t)(p % kHsiBlock) : (int32_t)p;
  }
};

// The bin, counting down from the top, where the running count reaches
// `need` (>= 1): s.cut_bin, s.cut_above = keys in higher bins, s.cut_total =
// all keys (the cut is set only when cut_total >= need).  Every thread sums
// nbins/kSelThreads bins (thread t from the top) and scans them within its
// warp; warp 0 scans the warp totals; the one thread whose bins hold the
// cut walks them.
__device__ void find_cut(const uint32_t* hist, int nbins, uint32_t need, SelShared& s) {
  const int per = nbins / kSelThreads;
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int top = nbins - 1 - per * t;
  uint32_t sum = 0;
  for (int i = 0; i < per; ++i) sum += hist[top - i];
  const uint32_t incl = warp_incl_scan(sum);
  if (lane == 31) s.wsum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const uint32_t ws = lane < kSelWarps ? s.wsum[lane] : 0u, wi = warp_incl_scan(ws);
    __syncwarp();
    if (lane < kSelWarps) s.wsum[lane] = wi - ws;
    if (lane == 31) s.cut_total = wi;
  }
  __syncthreads();
  const uint32_t excl = s.wsum[wid] + incl - sum;
  if (excl < need && excl + sum >= need) {
    uint32_t above = excl;
    for (int i = 0; i < per; ++i) {
      const uint32_t h = hist[top - i];
      if (above + h >= need) {
        s.cut_bin = (uint32_t)(top - i);
        s.cut_above = above;
        break;
      }
      above += h;
    }
  }
  __syncthreads();
}

// s.merged[0, nbins) = sum over the cluster's CTAs of their s.hist.
__device__ void merge_hist(SelShared& s, int nbins, int cs) {
  const uint32_t base = tc::smem_u32(s.hist);
  for (int b = threadIdx.x; b < nbins; b += kSelThreads) {
    uint32_t v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) v[r] = r < cs ? tc::ld_dsmem_u32(tc::map_rank(base + 4u * b, r)) : 0u;
    uint32_t acc = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) acc += v[r];
    s.merged[b] = acc;
  }
}

__device__ __forceinline__ void csync(int cs) {
  if (cs > 1)
    tc::cluster_sync();
  else
    __syncthreads();
}

__device__ __forceinline__ float ld_score(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// Shared-memory slot of key i of a round: 16-byte units are XOR-swizzled so
// that both the coalesced pattern (thread t, key t + 1024j) and one thread
// reading the 16 consecutive keys of its own range hit distinct banks.  The
// XOR term depends on bits 5-7 of i only, so kslot(t + 1024 j) = kslot(t) + 1024 j.
__device__ __forceinline__ int kslot(int i) {
  const int u = i >> 2;
  return ((u ^ ((u >> 3) & 7)) << 2) | (i & 3);
}

// Sort keys[0, total) ascending (total <= 4096, the largest pool of blocks)
// with a bitonic network over the next power of two >= total, at least
// kSelThreads; the slots from total on take 0xFFFFFFFF and end up last.
// Every thread of the CTA calls it; keys[] has room for 4096 entries.
__device__ void sort_positions(uint32_t* keys, uint32_t total) {
  uint32_t n = kSelThreads;
  while (n < total) n <<= 1;
  for (uint32_t i = total + threadIdx.x; i < n; i += kSelThreads) keys[i] = 0xFFFFFFFFu;
  __syncthreads();
  for (uint32_t k2 = 2; k2 <= n; k2 <<= 1) {
    for (uint32_t j = k2 >> 1; j > 0; j >>= 1) {
      for (uint32_t p = threadIdx.x; p < n / 2; p += kSelThreads) {
        const uint32_t i = 2 * j * (p / j) + (p % j), ixj = i + j;  // the pair (i, i + j), bit j of i clear
        const uint32_t x = keys[i], y = keys[ixj];
        if ((x > y) == ((i & k2) == 0)) {
          keys[i] = y;
          keys[ixj] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Select the k largest keys among n positions of `vals` by (key desc,
// position asc); `forced` (>= 0) always takes a slot.  Writes the chosen ids
// in ascending position order to out[k], -1 padded.  The cs CTAs of a
// cluster (cs = 1, 2, 4 or 8) each take one contiguous range of positions:
//   1. histogram of the keys over kHistBins linear bins of the query's key
//      range [kmin, kmax] (recorded by the scoring kernel), summed over the
//      cluster through distributed shared memory -> the bin where the count
//      from the top reaches k;
//   2. the keys of that bin are listed; when there are at most kRankMax of
//      them in the cluster, each one's rank among them gives the exact
//      threshold key T and the number krem of keys equal to T that still fit
//      (the first krem by position); more are refined 11 bits at a time
//      (cluster-summed digit histograms);
//   3. ordered compaction: each CTA starts after the selections of the lower
//      ranks; thread t owns kPer consecutive positions of a round, offsets
//      from warp scans and one scan over the warps.
// Keys are staged in shared memory a round of kRound positions at a time; a
// range of at most kRound positions is read from global memory once.
// One CTA over n positions far beyond its registers, with the query's key
// range known: a 1/16 sample of the keys (one 128-byte block in 16) picks a
// bin low enough that about twice the needed keys lie at or above it, one
// pass over the scores lists those keys with their positions, and the
// selection is finished among them in shared memory: the exact threshold bin
// by their histogram, the threshold key by ranking the bin's keys, the
// positions sorted.  Returns false, with nothing written, when the sample
// missed (too few or too many keys listed), the threshold bin holds too many
// keys to rank, or ties straddle the threshold; the caller then runs the
// general passes.  Every decision is taken from shared memory (uniform).
__device__ bool select_sampled(const float* vals, int64_t n, int k, int64_t forced, IdMap idmap, int32_t* out,
                               uint32_t kmin, int sh, uint32_t need, SelShared& s) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  auto bin_of = [&](uint32_t kk) -> uint32_t {
    const uint32_t x = kk > kmin ? kk - kmin : 0u;
    return min(x >> sh, (uint32_t)(kHistBins - 1));
  };
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) s.hist[i] = 0;
  if (threadIdx.x == 0) {
    s.cand_n = 0;
    s.above_n = 0;
  }
  __syncthreads();
  // ---- the sample: block b of 32 keys at positions 512 b .. 512 b + 31,
  // eight blocks a warp in flight at once
  const int64_t nsb = (n + 511) / 512;
  constexpr int kSampleBatch = 8;
  for (int64_t b0 = wid; b0 < nsb; b0 += (int64_t)kSelWarps * kSampleBatch) {
    float sv[kSampleBatch];
#pragma unroll
    for (int u = 0; u < kSampleBatch; ++u) {
      const int64_t p = 512 * (b0 + (int64_t)kSelWarps * u) + lane;
      sv[u] = p < n ? ld_score(vals + p) : __uint_as_float(kScoreInvalid);
    }
#pragma unroll
    for (int u = 0; u < kSampleBatch; ++u) {
      const int64_t p = 512 * (b0 + (int64_t)kSelWarps * u) + lane;
      const uint32_t kk = p != forced ? order_key(sv[u]) : 0u;
      if (kk) atomicAdd(&s.hist[bin_of(kk)], 1u);
    }
  }
  __syncthreads();
  const uint32_t target = (2 * need + 1024) / 16 + 32;
  find_cut(s.hist, kHistBins, target, s);
  const uint32_t tb_lo = s.cut_total >= target ? s.cut_bin : 0u;
  __syncthreads();
  // ---- one pass: every key in a bin >= tb_lo (key >= klo1; bin 0 takes
  // every key, those below kmin too), with its position.  Rounds of kRound
  // positions, the next round's loads in flight while this one is listed.
  const uint32_t klo1 = tb_lo == 0u ? 1u : kmin + (tb_lo << sh);
  auto load_round = [&](float (&v)[kPer], int64_t base) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int64_t p = base + threadIdx.x + kSelThreads * j;
      v[j] = p < n ? ld_score(vals + p) : __uint_as_float(kScoreInvalid);
    }
  };
  auto list_round = [&](const float (&v)[kPer], int64_t base) {
    // j of this thread's forced position in the round, else -1
    const int64_t fo = forced - base - threadIdx.x;
    const int jf = (forced >= 0 && fo >= 0 && fo < (int64_t)kRound && fo % kSelThreads == 0) ? (int)(fo / kSelThreads) : -1;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint32_t kk = order_key(v[j]);
      const bool m = kk >= klo1 && j != jf;
      const uint32_t bal = __ballot_sync(0xffffffffu, m);
      if (!bal) continue;
      uint32_t at = 0;
      if (lane == 0) at = atomicAdd(&s.cand_n, (uint32_t)__popc(bal));
      at = __shfl_sync(0xffffffffu, at, 0) + __popc(bal & lt);
      if (m && at < (uint32_t)kCandMax) {
        s.cand[at] = kk - kmin;
        s.merged[at] = (uint32_t)(base + threadIdx.x + kSelThreads * j);
      }
    }
  };
  {
    float va[kPer], vb[kPer];
    load_round(va, 0);
    for (int64_t base = 0; base < n; base += 2 * (int64_t)kRound) {
      if (base + kRound < n) load_round(vb, base + kRound);
      list_round(va, base);
      if (base + kRound >= n) break;
      if (base + 2 * kRound < n) load_round(va, base + 2 * kRound);
      list_round(vb, base + kRound);
    }
  }
  __syncthreads();
  const uint32_t c = s.cand_n;
  if (c < need || c > (uint32_t)kCandMax) return false;
  // ---- the exact threshold bin among the listed keys
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) s.hist[i] = 0;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < c; i += kSelThreads) atomicAdd(&s.hist[bin_of(s.cand[i] + kmin)], 1u);
  __syncthreads();
  find_cut(s.hist, kHistBins, need, s);
  uint32_t tx = 0;  // take every listed key x > tx, and the keys x == tx
  if (s.cut_total > need) {
    const uint32_t tb = s.cut_bin, krem = need - s.cut_above, cb = s.hist[tb];
    if (cb > (uint32_t)kRankMax) return false;
    // the bin's keys into s.all, then each ranked among them (tpc threads each)
    if (threadIdx.x == 0) s.c_all = 0;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < c; i += kSelThreads) {
      const uint32_t x = s.cand[i];
      if (bin_of(x + kmin) == tb) s.all[atomicAdd(&s.c_all, 1u)] = x;
    }
    __syncthreads();
    const uint32_t tpc = max(1u, (uint32_t)kSelThreads / cb);
    for (uint32_t i = threadIdx.x; i < cb; i += kSelThreads) s.part[i] = 0;
    __syncthreads();
    if (threadIdx.x < cb * tpc) {
      const uint32_t i = threadIdx.x % cb, part = threadIdx.x / cb;
      const uint32_t x = s.all[i];
      uint32_t gt = 0, eq = 0;
      for (uint32_t j = part; j < cb; j += tpc) {
        const uint32_t y = s.all[j];
        gt += y > x;
        eq += y == x;
      }
      atomicAdd(&s.part[i], gt | (eq << 16));
    }
    __syncthreads();
    if (threadIdx.x == 0) s.grand = 0;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < cb; i += kSelThreads) {
      const uint32_t gt = s.part[i] & 0xFFFFu, eq = s.part[i] >> 16;
      if (gt < krem && krem <= gt + eq) {  // the same key for every such i
        s.t_x = s.all[i];
        s.grand = (gt + eq == krem) ? 1u : 0u;  // every key equal to it is taken
      }
    }
    __syncthreads();
    if (!s.grand) return false;  // ties straddle the threshold
    tx = s.t_x;
  }
  // ---- the selection (need keys, and the forced position), sorted by position
  if (threadIdx.x == 0) s.grand = 0;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < c; i += kSelThreads)
    if (s.cand[i] >= tx) s.keys[atomicAdd(&s.grand, 1u)] = s.merged[i];
  __syncthreads();
  if (threadIdx.x == 0 && forced >= 0) s.keys[s.grand++] = (uint32_t)forced;
  __syncthreads();
  const uint32_t total = s.grand;
  sort_positions(s.keys, total);
  for (int i = threadIdx.x; i < k; i += kSelThreads) out[i] = (uint32_t)i < total ? idmap(s.keys[i]) : -1;
  return true;
}

template <bool kOne>  // a single CTA (cs == 1)
__device__ void select_topk(const float* vals, int64_t n, int k, int64_t forced, IdMap idmap, int32_t* out,
                            uint32_t kmin, uint32_t kmax, SelShared& s, int cs, int rk) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const bool has_forced = forced >= 0 && forced < n;
  const uint32_t need = (uint32_t)k - (has_forced ? 1u : 0u);
  const bool any = kmin <= kmax;
  const uint32_t range = any ? kmax - kmin : 0u;
  const int nbits = range ? 32 - __clz(range) : 0;
  const int sh = nbits > 13 ? nbits - 13 : 0;
  int64_t L = (n + cs - 1) / cs;
  L = (L + 511) & ~(int64_t)511;
  const int64_t lo = min(n, (int64_t)rk * L), hi = min(n, lo + L);
  forced = (forced >= lo && forced < hi) ? forced : -1;  // only the CTA whose range holds it
  const bool resident = L <= kRound;
  const bool ranked = need > 0 && any;
  const uint32_t lt = (1u << lane) - 1u;
  auto bin_of = [&](uint32_t kk) -> uint32_t {
    const uint32_t x = kk > kmin ? kk - kmin : 0u;
    return min(x >> sh, (uint32_t)(kHistBins - 1));
  };
  // stage round `base`: position lo + base + i -> s.keys[kslot(i)] (0 past hi
  // and at the forced position), every load issued before the first is
  // used; optionally histogram the keys on the way
  auto load = [&](int64_t base, bool count) {
    float v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int64_t p = lo + base + threadIdx.x + kSelThreads * j;
      v[j] = p < hi ? ld_score(vals + p) : __uint_as_float(kScoreInvalid);
    }
    const int ks0 = kslot(threadIdx.x);  // kslot(t + 1024 j) = kslot(t) + 1024 j
    const int64_t f = forced - (lo + base) - threadIdx.x;  // j * 1024 at the forced position
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint32_t kk = (f == (int64_t)kSelThreads * j) ? 0u : order_key(v[j]);
      s.keys[ks0 + kSelThreads * j] = kk;
      if (count && kk) atomicAdd(&s.hist[bin_of(kk)], 1u);
    }
  };
  // make round `base` the staged one (a no-op for a resident range)
  auto stage = [&](int64_t base) {
    if (resident) return;
    __syncthreads();
    load(base, false);
    __syncthreads();
  };

  if (kOne && !resident && ranked && n >= 2 * (int64_t)kRound && need <= 2048u) {
    if (select_sampled(vals, n, k, forced, idmap, out, kmin, sh, need, s)) return;
    __syncthreads();  // the general passes reuse the shared memory
  }
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) s.hist[i] = 0;
  if (threadIdx.x == 0) {
    s.cand_n = 0;
    s.tot_gt = 0;
    s.tot_eq = 0;
    s.carry_gt = 0;
    s.carry_eq = 0;
    s.above_n = 0;
  }
  __syncthreads();
  uint32_t T = 0xFFFFFFFFu, krem = 0;  // select key > T, then the first krem keys == T
  // one CTA whose threshold bin is listed: the listing pass also keeps the
  // positions above the bin and of the bin's keys, and the selection is
  // sorted out of shared memory instead of a compaction pass over the scores
  bool kept = false;
  uint32_t kept_x = 0;
  if (ranked) {
    for (int64_t base = 0; base < L; base += kRound) {
      if (base > 0) __syncthreads();
      load(base, true);
    }
    csync(cs);
    const uint32_t* H = s.hist;
    if (cs > 1) {
      merge_hist(s, kHistBins, cs);
      H = s.merged;
      __syncthreads();
    }
    find_cut(H, kHistBins, need, s);
    if (s.cut_total <= need) {
      T = 0;  // every valid key
    } else {
      const uint32_t tb = s.cut_bin;
      uint32_t prefix = tb;
      int rem = sh;
      krem = need - s.cut_above;
      const bool listed = s.hist[tb] <= (uint32_t)kCandMax;  // this CTA's share of the bin
      kept = kOne && rem > 0 && listed && s.cut_above + (has_forced ? 1u : 0u) <= (uint32_t)kRankMax;
      if (rem > 0 && listed) {
        for (int64_t base = 0; base < L; base += kRound) {
          stage(base);
#pragma unroll 4
          for (int j = 0; j < kPer; ++j) {
            const uint32_t kk = s.keys[kslot(threadIdx.x) + kSelThreads * j];
            const int64_t pos = lo + base + threadIdx.x + (int64_t)kSelThreads * j;
            const uint32_t bn = bin_of(kk);
            const bool m = kk != 0u && bn == tb;
            const uint32_t bal = __ballot_sync(0xffffffffu, m);
            if (kOne && kept) {
              const bool up = (kk != 0u && bn > tb) || pos == forced;
              const uint32_t bu = __ballot_sync(0xffffffffu, up);
              if (bu) {
                uint32_t au = 0;
                if (lane == 0) au = atomicAdd(&s.above_n, (uint32_t)__popc(bu));
                au = __shfl_sync(0xffffffffu, au, 0);
                if (up && au + __popc(bu & lt) < (uint32_t)kRankMax) s.all[au + __popc(bu & lt)] = (uint32_t)pos;
              }
            }
            if (!bal) continue;
            uint32_t at = 0;
            if (lane == 0) at = atomicAdd(&s.cand_n, (uint32_t)__popc(bal));
            at = __shfl_sync(0xffffffffu, at, 0);
            if (m) {
              s.cand[at + __popc(bal & lt)] = kk - kmin;
              if (kOne && kept) s.merged[at + __popc(bal & lt)] = (uint32_t)pos;
            }
          }
        }
      }
      if (rem > 0) {
        // the cluster's count of threshold-bin keys (all CTAs agree on `small`)
        csync(cs);
        if (threadIdx.x == 0) {
          uint32_t c = 0, ok = 1;
          for (int r = 0; r < cs; ++r) {
            s.peer_off[r] = c;
            const uint32_t cr = cs > 1 ? tc::ld_dsmem_u32(tc::map_rank(tc::smem_u32(&s.cand_n), r)) : s.cand_n;
            const uint32_t hr = cs > 1 ? tc::ld_dsmem_u32(tc::map_rank(tc::smem_u32(&s.hist[tb]), r)) : s.hist[tb];
            ok &= cr == hr;  // every CTA listed its share
            c += hr;
          }
          s.peer_off[cs] = c;
          s.c_all = ok ? c : 0xFFFFFFFFu;
        }
        __syncthreads();
        const uint32_t c_all = s.c_all;
        if (c_all <= (uint32_t)kRankMax) {
          const uint32_t* C = s.cand;
          if (cs > 1) {
            for (uint32_t i = threadIdx.x; i < c_all; i += kSelThreads) {
              int r = 0;
              while (i >= s.peer_off[r + 1]) ++r;
              s.all[i] = tc::ld_dsmem_u32(tc::map_rank(tc::smem_u32(&s.cand[i - s.peer_off[r]]), r));
            }
            C = s.all;
            __syncthreads();
          }
          // rank of each candidate among the threshold-bin keys: the c x c
          // comparisons spread over all threads (tpc threads per candidate,
          // counts gathered in shared memory: gt in the low 16 bits, eq high)
          const uint32_t tpc = c_all ? max(1u, (uint32_t)kSelThreads / c_all) : 1u;
          for (uint32_t i = threadIdx.x; i < c_all; i += kSelThreads) s.part[i] = 0;
          __syncthreads();
          if (threadIdx.x < c_all * tpc) {
            const uint32_t i = threadIdx.x % c_all, part = threadIdx.x / c_all;
            const uint32_t x = C[i];
            uint32_t gt = 0, eq = 0;
            for (uint32_t j = part; j < c_all; j += tpc) {
              const uint32_t y = C[j];
              gt += y > x;
              eq += y == x;
            }
            atomicAdd(&s.part[i], gt | (eq << 16));
          }
          __syncthreads();
          for (uint32_t i = threadIdx.x; i < c_all; i += kSelThreads) {
            const uint32_t gt = s.part[i] & 0xFFFFu, eq = s.part[i] >> 16;
            if (gt < krem && krem <= gt + eq) {  // the same key and counts for every such i
              s.t_x = C[i];
              s.t_krem = krem - gt;
            }
          }
          __syncthreads();
          prefix = s.t_x;
          krem = s.t_krem;
          rem = 0;
        }
      }
      while (rem > 0) {
        const int w = rem < 11 ? rem : 11;
        const int s2 = rem - w;
        const uint32_t dmask = (1u << w) - 1u;
        csync(cs);  // every CTA is done reading the previous histograms
        for (int i = threadIdx.x; i < kDigitBins; i += kSelThreads) s.hist[i] = 0;
        __syncthreads();
        if (listed) {
          const uint32_t cn = s.cand_n;
          for (uint32_t i = threadIdx.x; i < cn; i += kSelThreads) {
            const uint32_t x = s.cand[i];
            if ((x >> rem) == prefix) atomicAdd(&s.hist[(x >> s2) & dmask], 1u);
          }
        } else {
          for (int64_t base = 0; base < L; base += kRound) {
            stage(base);
#pragma unroll 1
            for (int i = threadIdx.x; i < kRound; i += kSelThreads) {
              const uint32_t kk = s.keys[kslot(i)], x = kk - kmin;
              if (kk != 0u && kk >= kmin && (x >> rem) == prefix) atomicAdd(&s.hist[(x >> s2) & dmask], 1u);
            }
          }
        }
        csync(cs);
        const uint32_t* D = s.hist;
        if (cs > 1) {
          merge_hist(s, kDigitBins, cs);
          D = s.merged;
          __syncthreads();
        }
        find_cut(D, kDigitBins, krem, s);
        krem -= s.cut_above;
        prefix = (prefix << w) | s.cut_bin;
        rem = s2;
      }
      T = kmin + prefix;
      kept_x = prefix;
    }
  } else if (resident) {
    load(0, false);
    __syncthreads();
  }

  if (kOne && kept) {
    // every key of the bin equal to T is taken (else the ties straddle the
    // threshold and the compaction pass orders them by position)
    __syncthreads();
    if (threadIdx.x == 0) s.grand = 0;
    __syncthreads();
    uint32_t eq = 0;
    for (uint32_t i = threadIdx.x; i < s.cand_n; i += kSelThreads) eq += s.cand[i] == kept_x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) eq += __shfl_xor_sync(0xffffffffu, eq, o);
    if (lane == 0 && eq) atomicAdd(&s.grand, eq);
    __syncthreads();
    kept = s.grand == krem && s.above_n == s.cut_above + (has_forced ? 1u : 0u);
    __syncthreads();
  }
  if (kOne && kept) {
    // the selection: the positions above the bin, then the bin's keys >= T,
    // sorted by position
    const uint32_t na = s.above_n;
    s.keys[threadIdx.x] = threadIdx.x < na ? s.all[threadIdx.x] : 0xFFFFFFFFu;
    if (threadIdx.x == 0) s.grand = na;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < s.cand_n; i += kSelThreads)
      if (s.cand[i] >= kept_x) s.keys[atomicAdd(&s.grand, 1u)] = s.merged[i];
    __syncthreads();
    const uint32_t total = s.grand;  // need (+ the forced position) <= k
    sort_positions(s.keys, total);
    for (int i = threadIdx.x; i < k; i += kSelThreads) out[i] = (uint32_t)i < total ? idmap(s.keys[i]) : -1;
    return;
  }

  // ---- ordered compaction: in a round, thread t owns keys kPer t .. kPer t + kPer - 1
  auto sel_gt = [&](uint32_t kk, int64_t p) { return kk > T || p == forced; };
  auto sel_eq = [&](uint32_t kk) { return kk == T && T != 0u; };
  if (cs > 1) {
    // this CTA's keys above T (and the forced position) and equal to T
    uint32_t gt = 0, eq = 0;
    for (int64_t base = 0; base < L; base += kRound) {
      stage(base);
#pragma unroll 4
      for (int j = 0; j < kPer; ++j) {
        const int i = threadIdx.x + kSelThreads * j;
        const uint32_t kk = s.keys[kslot(threadIdx.x) + kSelThreads * j];
        gt += sel_gt(kk, lo + base + i);
        eq += sel_eq(kk);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      gt += __shfl_xor_sync(0xffffffffu, gt, o);
      eq += __shfl_xor_sync(0xffffffffu, eq, o);
    }
    if (lane == 0) {
      atomicAdd(&s.tot_gt, gt);
      atomicAdd(&s.tot_eq, eq);
    }
    csync(cs);
    if (threadIdx.x == 0) {
      // the keys above T and equal to T in lower ranks
      const uint32_t tg = tc::smem_u32(&s.tot_gt), te = tc::smem_u32(&s.tot_eq);
      uint32_t g_all = 0, e_all = 0;
      for (int r = 0; r < cs; ++r) {
        if (r == rk) {
          s.carry_gt = g_all;
          s.carry_eq = e_all;
        }
        g_all += tc::ld_dsmem_u32(tc::map_rank(tg, r));
        e_all += tc::ld_dsmem_u32(tc::map_rank(te, r));
      }
    }
    csync(cs);  // no CTA reads another's shared memory after this
  }
  for (int64_t base = 0; base < L; base += kRound) {
    stage(base);
    uint32_t kk[kPer];
#pragma unroll
    for (int m = 0; m < kPer / 4; ++m) {
      const uint4 v4 = *reinterpret_cast<const uint4*>(s.keys + kslot(kPer * threadIdx.x + 4 * m));
      kk[4 * m] = v4.x;
      kk[4 * m + 1] = v4.y;
      kk[4 * m + 2] = v4.z;
      kk[4 * m + 3] = v4.w;
    }
    const int64_t p0 = lo + base + kPer * threadIdx.x;
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      gt += sel_gt(kk[m], p0 + m);
      eq += sel_eq(kk[m]);
    }
    const uint32_t v = gt | (eq << 16);
    const uint32_t incl = warp_incl_scan(v);
    if (lane == 31) s.wsum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const uint32_t ws = lane < kSelWarps ? s.wsum[lane] : 0u, wi = warp_incl_scan(ws);
      __syncwarp();
      if (lane < kSelWarps) s.wsum[lane] = wi - ws;
      if (lane == 31) s.wsum[kSelWarps] = wi;
    }
    __syncthreads();
    const uint32_t before = s.wsum[wid] + incl - v;
    uint32_t E = s.carry_eq + (before >> 16);
    uint32_t off = s.carry_gt + (before & 0xFFFFu) + min(krem, E);
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      bool take = sel_gt(kk[m], p0 + m);
      if (!take && sel_eq(kk[m])) take = E++ < krem;
      if (take) {
        if (off < (uint32_t)k) out[off] = idmap(p0 + m);
        ++off;
      }
    }
    __syncthreads();  // every thread has read the carries and the warp offsets
    if (threadIdx.x == 0) {
      s.carry_gt += s.wsum[kSelWarps] & 0xFFFFu;
      s.carry_eq += s.wsum[kSelWarps] >> 16;
    }
  }
  // the last rank pads after every selection of the cluster
  if (rk == cs - 1) {
    __syncthreads();
    const uint32_t total = s.carry_gt + min(krem, s.carry_eq);
    for (uint32_t i = total + threadIdx.x; i < (uint32_t)k; i += kSelThreads) out[i] = -1;
  }
}

// The same selection for a single CTA holding all n <= kSelThreads * kP positions
// (one copy of its code shared by every call site: when the code is not
// cached its instructions are fetched once, which was measured faster than
// inlining it into each caller):
// thread t owns positions kP t .. kP t + kP - 1 (kP = 16 or 32) and keeps their keys in registers
// from the one read of the scores to the ordered write of the ids
// (histogram, cut search, threshold-bin keys ranked or refined by digits,
// then one scan of packed (above, equal) counts).
// gpool != NULL: position p reads vals[gpool[p / 8] * 8 + p % 8] (a pool of
// 8-entry blocks written earlier by this CTA; ids >= nv_lim or blocks < 0 are
// not candidates).  Keys below kmin are not candidates either (the caller
// knows at least k keys lie at or above it).  out_copy: the ids also written
// there (shared memory); t_out: the threshold key (every selected key but the
// forced one is at or above it).
template <int kP>
__device__ __noinline__ void select_small(const float* vals, int64_t n, int k, int64_t forced, IdMap idmap, int32_t* out,
                             uint32_t kmin, uint32_t kmax, SelShared& s, const int32_t* gpool = nullptr,
                             int64_t nv_lim = 0, int32_t* out_copy = nullptr, uint32_t* t_out = nullptr) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const bool has_forced = forced >= 0 && forced < n;
  const uint32_t need = (uint32_t)k - (has_forced ? 1u : 0u);
  const bool any = kmin <= kmax;
  const uint32_t range = any ? kmax - kmin : 0u;
  const int nbits = range ? 32 - __clz(range) : 0;
  const int sh = nbits > 13 ? nbits - 13 : 0;
  const bool ranked = need > 0 && any;
  const int64_t p0 = (int64_t)kP * threadIdx.x;
  float v[kP];
  // the ids this thread may emit come from two 8-position pool blocks (a
  // pool-mapped selection): their block ids are kept in registers, so the
  // ordered writes below need no dependent load per selected position
  const int32_t* pmap = gpool ? gpool : idmap.pool;
  int32_t blkr[kP / kHsiBlock];
#pragma unroll
  for (int h = 0; h < kP / kHsiBlock; ++h) {
    const int64_t pb = (p0 >> 3) + h;
    blkr[h] = (pmap && pb * kHsiBlock < n) ? *reinterpret_cast<const volatile int32_t*>(pmap + pb) : -1;
  }
  if (gpool) {
    const bool al = ((uintptr_t)vals & 15u) == 0;
#pragma unroll
    for (int h = 0; h < kP / kHsiBlock; ++h) {
      const int32_t blk = blkr[h];  // pool slot's block (written by this CTA just before)
      const int64_t j0 = (int64_t)blk * kHsiBlock;
      if (blk >= 0 && al && j0 + kHsiBlock <= nv_lim) {  // a whole visible block: two 16-byte loads
#pragma unroll
        for (int q = 0; q < kHsiBlock / 4; ++q) {
          float4 f4;
          asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(f4.x), "=f"(f4.y), "=f"(f4.z), "=f"(f4.w)
                       : "l"(vals + j0 + 4 * q));
          v[kHsiBlock * h + 4 * q] = f4.x;
          v[kHsiBlock * h + 4 * q + 1] = f4.y;
          v[kHsiBlock * h + 4 * q + 2] = f4.z;
          v[kHsiBlock * h + 4 * q + 3] = f4.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < kHsiBlock; ++i) {
          const int64_t j = j0 + i;
          v[kHsiBlock * h + i] = (blk >= 0 && j < nv_lim) ? ld_score(vals + j) : __uint_as_float(kScoreInvalid);
        }
      }
    }
  } else if (((uintptr_t)vals & 15u) == 0 && p0 + kP <= n) {
#pragma unroll
    for (int q = 0; q < kP / 4; ++q) {
      float4 f4;
      asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(f4.x), "=f"(f4.y), "=f"(f4.z), "=f"(f4.w)
                   : "l"(vals + p0 + 4 * q));
      v[4 * q] = f4.x;
      v[4 * q + 1] = f4.y;
      v[4 * q + 2] = f4.z;
      v[4 * q + 3] = f4.w;
    }
  } else {
#pragma unroll
    for (int m = 0; m < kP; ++m) v[m] = p0 + m < n ? ld_score(vals + p0 + m) : __uint_as_float(kScoreInvalid);
  }
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) s.hist[i] = 0;
  if (threadIdx.x == 0) s.cand_n = 0;
  // this thread's positions as bits of kP-bit masks (bit m: position p0 + m)
  const uint32_t fm = (has_forced && forced >= p0 && forced < p0 + kP) ? 1u << (int)(forced - p0) : 0u;
  uint32_t kk[kP];
#pragma unroll
  for (int m = 0; m < kP; ++m) kk[m] = ((fm >> m) & 1u) ? 0u : order_key(v[m]);
  __syncthreads();

  const uint32_t kmin1 = kmin > 0u ? kmin : 1u;  // candidates: keys >= kmin (key 0: none)
  uint32_t T = 0xFFFFFFFFu, krem = 0;  // select key > T, then the first krem keys == T
  if (ranked) {
#pragma unroll
    for (int m = 0; m < kP; ++m)
      if (kk[m] >= kmin1) atomicAdd(&s.hist[min((kk[m] - kmin) >> sh, (uint32_t)(kHistBins - 1))], 1u);
    __syncthreads();
    find_cut(s.hist, kHistBins, need, s);
    if (s.cut_total <= need) {
      T = kmin > 0u ? kmin - 1u : 0u;  // every candidate key
    } else {
      const uint32_t tb = s.cut_bin;
      uint32_t prefix = tb;
      int rem = sh;
      krem = need - s.cut_above;
      if (rem > 0) {
        {  // this thread's keys of the cut bin, one shared-memory atomic per warp
          // the bin's keys: kmin + [tb << sh, (tb + 1) << sh), the top bin open above
          const uint32_t klo = kmin + (tb << sh);
          const uint32_t span = (1u << sh) - 1u;
          const uint32_t khi = (tb == (uint32_t)(kHistBins - 1) || klo > 0xFFFFFFFFu - span) ? 0xFFFFFFFFu : klo + span;
          const uint32_t klo1 = klo > kmin1 ? klo : kmin1;
          uint32_t cutm = 0;
#pragma unroll
          for (int m = 0; m < kP; ++m) cutm |= (kk[m] >= klo1 && kk[m] <= khi) ? 1u << m : 0u;
          const uint32_t mine = __popc(cutm);
          const uint32_t incl = warp_incl_scan(mine);
          uint32_t at = 0;
          if (lane == 31 && incl) at = atomicAdd(&s.cand_n, incl);
          at = __shfl_sync(0xffffffffu, at, 31) + incl - mine;
          if (cutm) {
#pragma unroll
            for (int m = 0; m < kP; ++m)
              if ((cutm >> m) & 1u) {
                if (at < (uint32_t)kCandMax) s.cand[at] = kk[m] - kmin;
                ++at;
              }
          }
        }
        __syncthreads();
        const uint32_t c = s.cand_n;
        if (c <= (uint32_t)kRankMax) {
          // rank of each candidate among the threshold-bin keys: 2^lg adjacent
          // lanes per candidate (one while there are fewer than 32, at most 8),
          // their counts summed by shuffles
          int lg = 0;
          while ((c << (lg + 1)) <= (uint32_t)kSelThreads && (2u << lg) <= c / 16u) ++lg;
          const uint32_t i = threadIdx.x >> lg, part = threadIdx.x & ((1u << lg) - 1u);
          uint32_t gt = 0, eq = 0, x = 0;
          if (i < c) {
            x = s.cand[i];
            for (uint32_t j = part; j < c; j += 1u << lg) {
              const uint32_t y = s.cand[j];
              gt += y > x;
              eq += y == x;
            }
          }
          for (int o = 1; o < (1 << lg); o <<= 1) {
            gt += __shfl_xor_sync(0xffffffffu, gt, o);
            eq += __shfl_xor_sync(0xffffffffu, eq, o);
          }
          if (i < c && part == 0 && gt < krem && krem <= gt + eq) {  // the same key and counts for every such i
            s.t_x = x;
            s.t_krem = krem - gt;
          }
          __syncthreads();
          prefix = s.t_x;
          krem = s.t_krem;
          rem = 0;
        }
        // many keys in the cut bin: 11-bit digits over the list (or the registers)
        while (rem > 0) {
          const int w = rem < 11 ? rem : 11;
          const int s2 = rem - w;
          const uint32_t dmask = (1u << w) - 1u;
          for (int i = threadIdx.x; i < kDigitBins; i += kSelThreads) s.hist[i] = 0;
          __syncthreads();
          if (c <= (uint32_t)kCandMax) {
            for (uint32_t i = threadIdx.x; i < c; i += kSelThreads) {
              const uint32_t x = s.cand[i];
              if ((x >> rem) == prefix) atomicAdd(&s.hist[(x >> s2) & dmask], 1u);
            }
          } else {
#pragma unroll
            for (int m = 0; m < kP; ++m) {
              const uint32_t x = kk[m] - kmin;
              if (kk[m] != 0u && kk[m] >= kmin && (x >> rem) == prefix) atomicAdd(&s.hist[(x >> s2) & dmask], 1u);
            }
          }
          __syncthreads();
          find_cut(s.hist, kDigitBins, krem, s);
          krem -= s.cut_above;
          prefix = (prefix << w) | s.cut_bin;
          rem = s2;
        }
      }
      T = kmin + prefix;
    }
  }

  // ---- ordered compaction
  uint32_t gtm = fm, eqm = 0;  // keys above T (and the forced position); keys equal to T
#pragma unroll
  for (int m = 0; m < kP; ++m) {
    gtm |= kk[m] > T ? 1u << m : 0u;
    eqm |= (kk[m] == T && T != 0u) ? 1u << m : 0u;
  }
  const uint32_t vpk = __popc(gtm) | (__popc(eqm) << 16);
  const uint32_t incl = warp_incl_scan(vpk);
  if (lane == 31) s.wsum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const uint32_t ws = lane < kSelWarps ? s.wsum[lane] : 0u, wi = warp_incl_scan(ws);
    __syncwarp();
    if (lane < kSelWarps) s.wsum[lane] = wi - ws;
    if (lane == 31) s.wsum[kSelWarps] = wi;
  }
  __syncthreads();
  const uint32_t before = s.wsum[wid] + incl - vpk;
  const uint32_t E = before >> 16;
  uint32_t off = (before & 0xFFFFu) + min(krem, E);
  // taken: every key above T, and the first krem - E of this thread's keys
  // equal to T (by position); written in position order
  uint32_t takem = gtm;
  for (uint32_t em = eqm, left = krem > E ? krem - E : 0u; em && left; --left) {
    takem |= em & (0u - em);
    em &= em - 1u;
  }
  static_assert(kP <= 32 && kP % kHsiBlock == 0, "a thread's positions: bits of one mask, whole pool blocks");
  while (takem) {
    const int m = __ffs(takem) - 1;
    takem &= takem - 1u;
    if (off < (uint32_t)k) {
      int32_t blk = blkr[0];
#pragma unroll
      for (int h = 1; h < kP / kHsiBlock; ++h) blk = (m >> 3) == h ? blkr[h] : blk;
      const int32_t id = pmap ? blk * kHsiBlock + (m & (kHsiBlock - 1)) : (int32_t)(p0 + m);
      out[off] = id;
      if (out_copy) out_copy[off] = id;
    }
    ++off;
  }
  const uint32_t all = s.wsum[kSelWarps];
  const uint32_t total = (all & 0xFFFFu) + min(krem, all >> 16);
  for (uint32_t i = total + threadIdx.x; i < (uint32_t)k; i += kSelThreads) {
    out[i] = -1;
    if (out_copy) out_copy[i] = -1;
  }
  if (t_out && threadIdx.x == 0) *t_out = T;
}

// grid (cs, queries, selections), clusters of cs CTAs along x.  Selection 0:
// entry top-k (Full or Reindex); 1: HSI block pool (Full).
template <bool kSmall>
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(int q0, int Tq, int r, int k, int n_blocks,
                                                                int64_t max_entries,
                                                                const int64_t* __restrict__ q_pos,
                                                                const int32_t* __restrict__ n_entries,
                                                                const int32_t* __restrict__ pool, const float* scores,
                                                                const float* bmax, int64_t score_stride,
                                                                const uint32_t* krange, int kr_stride, int n_slots,
                                                                int32_t* topk_out, int32_t* pool_out, int fused) {
  extern __shared__ __align__(16) unsigned char sel_raw[];
  SelShared& s = *reinterpret_cast<SelShared*>(sel_raw);
  __shared__ uint32_t r_lo, r_hi;
  const int cs = (int)tc::cluster_size(), rk = (int)tc::cluster_rank();
  const int qc = blockIdx.y, qi = q0 + qc, b = qi / Tq;
  // the query's position and entry count are read before the wait: the
  // previous kernel is always the scoring kernel of the same call, which
  // writes neither and waited itself for whatever wrote them
  const int64_t qp = q_pos[qi];
  const int32_t ne = n_entries[b];
  if (threadIdx.x == 0) {
    r_lo = 0xFFFFFFFFu;
    r_hi = 0u;
  }
  griddep_wait();  // the scores are the previous kernel's output
  griddep_launch();
  const int64_t nv = visible_entries(qp, r, ne < max_entries ? ne : (int32_t)max_entries);
  // the query's key range: the scoring CTAs' slots reduced
  __syncthreads();
  {
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    const uint32_t* kr = krange + (int64_t)qc * kr_stride * 2;
    for (int i = threadIdx.x; i < n_slots; i += kSelThreads) {
      lo = min(lo, kr[2 * i]);
      hi = max(hi, kr[2 * i + 1]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if ((threadIdx.x & 31) == 0 && lo <= hi) {
      atomicMin(&r_lo, lo);
      atomicMax(&r_hi, hi);
    }
  }
  __syncthreads();
  const uint32_t lo = r_lo, hi = r_hi;
  auto run = [&](const float* v, int64_t n, int kk, int64_t forced, IdMap idmap, int32_t* o) {
    if (kSmall)
      select_small<kPer>(v, n, kk, forced, idmap, o, lo, hi, s);
    else if (cs == 1 && n <= kRound)
      select_small<kPer>(v, n, kk, forced, idmap, o, lo, hi, s);
    else if (cs == 1 && n <= 2 * kRound)
      select_small<2 * kPer>(v, n, kk, forced, idmap, o, lo, hi, s);
    else
      cs == 1 ? select_topk<true>(v, n, kk, forced, idmap, o, lo, hi, s, cs, rk)
              : select_topk<false>(v, n, kk, forced, idmap, o, lo, hi, s, cs, rk);
  };
  if (fused) {
    // Full with HSI, one CTA: the pool first, then the top-k over the pool's
    // positions.  Exact when the pool holds k blocks besides the forced one:
    // every block ranking above a block that holds a top-k entry e (block max
    // desc, block id asc) contains an entry ranking above e (score desc, id
    // asc), so at most k - 1 blocks rank above it.
    // The pool also goes to shared memory (the second selection reads its
    // block ids from there), and its threshold key bounds the second one from
    // below: each of the pool's blocks but the forced one has its maximum at
    // or above it, so at least k of the pool's positions do (n_blocks > k).
    const int64_t nb = (nv + kHsiBlock - 1) / kHsiBlock;
    int32_t* prow = pool_out + (int64_t)qi * n_blocks;
    const float* bm = bmax + (int64_t)qc * ((max_entries + 7) / 8);
    __shared__ uint32_t t_pool;
    if (kSmall || (cs == 1 && nb <= 2 * kRound)) {
      // the pool over up to 2 kRound blocks held in registers (16 or 32 keys
      // a thread), then the top-k over its positions
      int32_t* pool_s = reinterpret_cast<int32_t*>(s.keys);  // unused by the register-resident selection
      if (!kSmall && nb > kRound)
        select_small<2 * kPer>(bm, nb, n_blocks, nb - 1, IdMap{nullptr}, prow, lo, hi, s, nullptr, 0, pool_s,
                               &t_pool);
      else
        select_small<kPer>(bm, nb, n_blocks, nb - 1, IdMap{nullptr}, prow, lo, hi, s, nullptr, 0, pool_s, &t_pool);
      __syncthreads();  // the pool ids and its threshold are visible to the whole CTA
      const uint32_t lo2 = (t_pool != 0xFFFFFFFFu && t_pool > lo) ? t_pool : lo;
      select_small<kPer>(scores + (int64_t)qc * score_stride, (int64_t)n_blocks * kHsiBlock, k, -1, IdMap{prow},
                         topk_out + (int64_t)qi * k, lo2, hi, s, pool_s, nv);
    } else {
      run(bm, nb, n_blocks, nb - 1, IdMap{nullptr}, prow);
      __syncthreads();  // the pool ids are visible to the whole CTA
      select_small<kPer>(scores + (int64_t)qc * score_stride, (int64_t)n_blocks * kHsiBlock, k, -1, IdMap{prow},
                         topk_out + (int64_t)qi * k, lo, hi, s, prow, nv);
    }
  } else if (blockIdx.z == 0) {
    const float* v = scores + (int64_t)qc * score_stride;
    if (pool)
      run(v, (int64_t)n_blocks * kHsiBlock, k, -1, IdMap{pool + (int64_t)qi * n_blocks}, topk_out + (int64_t)qi * k);
    else
      run(v, nv, k, -1, IdMap{nullptr}, topk_out + (int64_t)qi * k);
  } else {
    const int64_t nb = (nv + kHsiBlock - 1) / kHsiBlock;
    const float* v = bmax + (int64_t)qc * ((max_entries + 7) / 8);
    run(v, nb, n_blocks, nb - 1, IdMap{nullptr}, pool_out + (int64_t)qi * n_blocks);
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// Per query: scores (Full: max_entries, Reindex: pool positions), HSI block
// maxima (Full with HSI), and the scoring CTAs' key-range slots (8 bytes each).
static int64_t score_tiles(const csa2_cfg& cfg, int max_entries, bool reindex) {
  return reindex ? ((int64_t)cfg.hsi_blocks * kHsiBlock + 127) / 128 : ((int64_t)max_entries + 127) / 128;
}

size_t index_query_ws_bytes(const csa2_cfg& cfg, int max_entries, bool reindex) {
  const size_t slots = align256((size_t)score_range_slots(score_tiles(cfg, max_entries, reindex)) * 8);
  if (reindex) return align256((size_t)cfg.hsi_blocks * kHsiBlock * sizeof(float)) + slots;
  size_t b = align256((size_t)max_entries * sizeof(float));
  if (cfg.hsi_blocks > 0) b += align256((size_t)((max_entries + 7) / 8) * sizeof(float));
  return b + slots;
}

namespace {

// Where the indexer's per-query data sits in a workspace, and the shape of
// the selection launch, for one call over B * Tq queries.  The layout does
// not depend on whether the HSI pool is asked for: with hsi_blocks > 0 (Full)
// the block maxima always have their place after the scores.
struct IndexPlan {
  int Q, chunk;
  bool reindex;
  float* scores;
  int64_t stride;
  float* bmax_area;  // block maxima (Full with hsi_blocks > 0), else null
  uint32_t* krange;
  int kr_stride;
  bool fused;
  int n_sel, cs;
  bool small;
};

cudaError_t plan_index(const csa2_cfg& cfg, int B, int Tq, int max_entries, bool reindex, bool hsi_out, void* ws,
                       size_t ws_bytes, IndexPlan* p) {
  p->Q = B * Tq;
  p->reindex = reindex;
  const size_t per_q = index_query_ws_bytes(cfg, max_entries, reindex);
  p->chunk = (int)std::min<size_t>(std::min<size_t>((size_t)p->Q, ws_bytes / per_q), 65535);  // grid y
  if (p->chunk < 1) return cudaErrorInvalidValue;
  p->scores = static_cast<float*>(ws);
  p->stride = reindex ? (int64_t)cfg.hsi_blocks * kHsiBlock : (int64_t)max_entries;
  char* cur = static_cast<char*>(ws) + align256((size_t)p->chunk * p->stride * sizeof(float));
  p->bmax_area = nullptr;
  if (!reindex && cfg.hsi_blocks > 0) {
    p->bmax_area = reinterpret_cast<float*>(cur);
    cur += align256((size_t)p->chunk * ((max_entries + 7) / 8) * sizeof(float));
  }
  p->krange = reinterpret_cast<uint32_t*>(cur);
  p->kr_stride = score_range_slots(score_tiles(cfg, max_entries, reindex));
  // a cluster of up to 8 CTAs per selection, each with at least kMinCtaKeys
  // positions, but no more CTAs than one wave holds (one CTA per SM)
  const int64_t n_max = reindex ? (int64_t)cfg.hsi_blocks * kHsiBlock : (int64_t)max_entries;
  // Full with HSI: one CTA selects the pool and then the top-k among the
  // pool's positions, when they fit one CTA's registers and the pool has at
  // least k blocks besides the forced one (what makes it exact)
  p->fused = !reindex && hsi_out && (int64_t)cfg.hsi_blocks * kHsiBlock <= kRound && cfg.hsi_blocks >= cfg.topk + 1;
  p->n_sel = (!reindex && hsi_out && !p->fused) ? 2 : 1;
  // (a selection one CTA holds in registers, up to 2 kRound positions at 32
  // keys a thread, stays on one CTA)
  const int64_t sel_groups = (int64_t)std::min(p->chunk, p->Q) * p->n_sel;
  p->cs = 1;
  while (!p->fused && n_max > 2 * kRound && p->cs < 8 && (int64_t)p->cs * kMinCtaKeys < n_max &&
         2 * p->cs * sel_groups <= num_sms())
    p->cs <<= 1;
  // one CTA holding every position of each selection: the register-resident
  // path only, compiled without the general one
  p->small = p->cs == 1 && (p->fused ? ((int64_t)max_entries + 7) / 8 <= kRound : n_max <= kRound);
  return cudaSuccess;
}

cudaError_t run_scores(const IndexPlan& p, const csa2_cfg& cfg, int q0, int nq, int Tq, const uint16_t* q_idx,
                       const float* head_w, const int64_t* q_pos, const csa2_cache& idx_c, const int32_t* n_entries,
                       int max_entries, const int32_t* pool, bool hsi_out, int* n_slots, int32_t* status,
                       cudaStream_t stream) {
  return launch_score_tc(cfg, q0, nq, Tq, q_idx, head_w, q_pos, idx_c, n_entries, max_entries, pool, p.scores,
                         p.stride, hsi_out ? p.bmax_area : nullptr, p.krange, p.kr_stride, n_slots, status, num_sms(),
                         stream);
}

cudaError_t run_select(const IndexPlan& p, const csa2_cfg& cfg, int q0, int nq, int Tq, const int64_t* q_pos,
                       const int32_t* n_entries, int max_entries, const int32_t* pool, int n_slots,
                       int32_t* topk_out, int32_t* pool_out, cudaStream_t stream) {
  const size_t sel_smem = sizeof(SelShared);
  auto sel = p.small ? select_kernel<true> : select_kernel<false>;
  cudaFuncSetAttribute(sel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sel_smem);
  return launch_k(sel, dim3(p.cs, nq, p.n_sel), dim3(kSelThreads), sel_smem, stream, p.cs, q0, Tq, cfg.ratio,
                  cfg.topk, cfg.hsi_blocks, (int64_t)max_entries, q_pos, n_entries, pool, (const float*)p.scores,
                  (const float*)(pool_out ? p.bmax_area : nullptr), p.stride, (const uint32_t*)p.krange, p.kr_stride,
                  n_slots, topk_out, pool_out, p.fused ? 1 : 0);
}

}  // namespace

cudaError_t launch_index_topk(const csa2_cfg& cfg, int B, int Tq, const uint16_t* q_idx,
                              const float* head_w, const int64_t* q_pos, const csa2_cache& idx_c,
                              const int32_t* n_entries, int max_entries, const int32_t* pool,
                              int32_t* topk_out, int32_t* pool_out, void* ws, size_t ws_bytes,
                              int32_t* status, cudaStream_t stream) {
  if (B * Tq == 0) return cudaSuccess;
  IndexPlan p;
  cudaError_t e = plan_index(cfg, B, Tq, max_entries, pool != nullptr, pool_out != nullptr, ws, ws_bytes, &p);
  if (e != cudaSuccess) return e;
  for (int q0 = 0; q0 < p.Q; q0 += p.chunk) {
    const int nq = std::min(p.chunk, p.Q - q0);
    int n_slots = 0;
    e = run_scores(p, cfg, q0, nq, Tq, q_idx, head_w, q_pos, idx_c, n_entries, max_entries, pool, pool_out != nullptr,
                   &n_slots, status, stream);
    if (e != cudaSuccess) return e;
    e = run_select(p, cfg, q0, nq, Tq, q_pos, n_entries, max_entries, pool, n_slots, topk_out, pool_out, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_index_score(const csa2_cfg& cfg, int B, int Tq, const uint16_t* q_idx, const float* head_w,
                               const int64_t* q_pos, const csa2_cache& idx_c, const int32_t* n_entries,
                               int max_entries, const int32_t* pool, bool hsi_out, void* ws, size_t ws_bytes,
                               int32_t* status, cudaStream_t stream) {
  if (B * Tq == 0) return cudaSuccess;
  IndexPlan p;
  cudaError_t e = plan_index(cfg, B, Tq, max_entries, pool != nullptr, hsi_out, ws, ws_bytes, &p);
  if (e != cudaSuccess) return e;
  if (p.chunk < p.Q) return cudaErrorInvalidValue;  // the workspace holds every query
  int n_slots = 0;
  return run_scores(p, cfg, 0, p.Q, Tq, q_idx, head_w, q_pos, idx_c, n_entries, max_entries, pool, hsi_out, &n_slots,
                    status, stream);
}

cudaError_t launch_index_select(const csa2_cfg& cfg, int B, int Tq, const int64_t* q_pos, const int32_t* n_entries,
                                int max_entries, const int32_t* pool, int32_t* topk_out, int32_t* pool_out, void* ws,
                                size_t ws_bytes, cudaStream_t stream) {
  if (B * Tq == 0) return cudaSuccess;
  IndexPlan p;
  cudaError_t e = plan_index(cfg, B, Tq, max_entries, pool != nullptr, pool_out != nullptr, ws, ws_bytes, &p);
  if (e != cudaSuccess) return e;
  if (p.chunk < p.Q) return cudaErrorInvalidValue;
  const int n_slots = score_slots_used(cfg, 0, p.Q, Tq, max_entries, pool != nullptr, num_sms());
  return run_select(p, cfg, 0, p.Q, Tq, q_pos, n_entries, max_entries, pool, n_slots, topk_out, pool_out, stream);
}

}  // namespace csa2
