// a3..a6 -- CSA2 lightweight indexer: per-query scores over the visible
// indexer-K entries (or over an HSI pool), HSI block maxima, and exact
// top-k selection with the (score desc, id asc) order.
// (DeepSeek-V4.1 Flash, hn.213312.xyz sec. 2.3.1, 2.3.2, 2.3.4; 36kr "CSA2".)
#include <algorithm>

#include "internal.h"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kSelThreads = 1024;   // one CTA selects for one query
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kPer = 16;              // keys a lane holds per round
constexpr int kRound = kSelThreads * kPer;  // positions per round; a warp covers 512 consecutive ones
constexpr int kHistBins = 8192;       // linear bins over a query's key range
constexpr int kDigitBins = 2048;      // refinement digit: 11 bits
constexpr int kCandMax = 8192;        // keys of the threshold bin listed in shared memory

// ---------------------------------------------------------------- select ----

struct SelShared {
  uint32_t hist[kHistBins];    // this CTA's histogram (the cluster's peers read it)
  uint32_t merged[kHistBins];  // the cluster's histogram
  uint32_t cand[kCandMax];
  uint32_t wa[kSelWarps + 1], wb[kSelWarps + 1];
  uint32_t cut_bin, cut_above, cut_total, cand_n, carry_eq, carry_off, grand;
  uint32_t tot_gt, tot_eq;     // this CTA's counts for the compaction (peers read them)
};

// Exclusive prefix sum over the CTA; returns the total in `total`.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    const uint32_t w = warp_sums[lane];
    uint32_t ws = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, ws, o);
      if (lane >= o) ws += y;
    }
    warp_sums[lane] = ws - w;
    if (lane == 31) warp_sums[32] = ws;
  }
  __syncthreads();
  const uint32_t res = warp_sums[wid] + x - v;
  total = warp_sums[32];
  __syncthreads();
  return res;
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
// all keys.  Thread t owns nbins/kSelThreads bins from the top.
__device__ void find_cut(const uint32_t* hist, int nbins, uint32_t need, SelShared& s) {
  const int per = nbins / kSelThreads;
  const int top = nbins - 1 - per * (int)threadIdx.x;
  uint32_t sum = 0;
  for (int i = 0; i < per; ++i) sum += hist[top - i];
  uint32_t total;
  const uint32_t excl = block_exclusive_scan(sum, s.wa, total);
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
  if (threadIdx.x == 0) s.cut_total = total;
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

// Keys of one round of the range [lo, hi): lane l of warp w holds positions
// lo + base + 512w + 32j + l (j < kPer); 0 past hi and at the forced one.
// The loads are issued together and the values stay in registers.
__device__ __forceinline__ void load_round(const float* vals, int64_t lo, int64_t hi, int64_t forced, int64_t base,
                                           uint32_t (&key)[kPer]) {
  const int64_t p0 = lo + base + (threadIdx.x >> 5) * (32 * kPer) + (threadIdx.x & 31);
  float v[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int64_t p = p0 + 32 * j;
    v[j] = p < hi ? ld_score(vals + p) : __uint_as_float(kScoreInvalid);
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) key[j] = (p0 + 32 * j == forced) ? 0u : order_key(v[j]);
}

// Select the k largest keys among n positions of `vals` by (key desc,
// position asc); `forced` (>= 0) always takes a slot.  Writes the chosen ids
// in ascending position order to out[k], -1 padded.  The cs CTAs of a
// cluster (cs = 1, 2, 4 or 8) each take one contiguous range of positions:
//   1. histogram of the keys over kHistBins linear bins of the query's key
//      range [kmin, kmax] (recorded by the scoring kernel), summed over the
//      cluster through distributed shared memory -> the bin where the count
//      from the top reaches k;
//   2. the keys of that bin are listed in shared memory and refined 11 bits
//      at a time (cluster-summed digit histograms) down to the exact
//      threshold key T and the number krem of keys equal to T that still fit
//      (the first krem by position);
//   3. ordered compaction: each CTA starts after the selections of the lower
//      ranks; within a CTA, warp ballots over 512-position runs and one scan
//      over the warps per round.
// A range of at most kRound positions stays in registers after one read.
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
  // a CTA's round layout spans kRound positions from lo, past hi when L < kRound:
  // only the CTA whose range holds the forced position may count it
  forced = (forced >= lo && forced < hi) ? forced : -1;
  const bool resident = L <= kRound;
  const bool ranked = need > 0 && any;
  auto bin_of = [&](uint32_t kk) -> uint32_t {
    const uint32_t x = kk > kmin ? kk - kmin : 0u;
    return min(x >> sh, (uint32_t)(kHistBins - 1));
  };
  uint32_t key[kPer];

  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) s.hist[i] = 0;
  if (threadIdx.x == 0) {
    s.cand_n = 0;
    s.tot_gt = 0;
    s.tot_eq = 0;
  }
  __syncthreads();
  uint32_t T = 0xFFFFFFFFu, krem = 0;  // select key > T, then the first krem keys == T
  if (ranked) {
    for (int64_t base = 0; base < L; base += kRound) {
      load_round(vals, lo, hi, forced, base, key);
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (key[j]) atomicAdd(&s.hist[bin_of(key[j])], 1u);
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
      if (rem > 0 && listed) {
        for (int64_t base = 0; base < L; base += kRound) {
          if (!resident) load_round(vals, lo, hi, forced, base, key);
#pragma unroll
          for (int j = 0; j < kPer; ++j) {
            const bool m = key[j] != 0u && bin_of(key[j]) == tb;
            const uint32_t bal = __ballot_sync(0xffffffffu, m);
            if (!bal) continue;
            uint32_t at = 0;
            if (lane == 0) at = atomicAdd(&s.cand_n, (uint32_t)__popc(bal));
            at = __shfl_sync(0xffffffffu, at, 0);
            if (m) s.cand[at + __popc(bal & ((1u << lane) - 1u))] = key[j] - kmin;
          }
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
            if (!resident) load_round(vals, lo, hi, forced, base, key);
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
              const uint32_t x = key[j] - kmin;
              if (key[j] != 0u && key[j] >= kmin && (x >> rem) == prefix) atomicAdd(&s.hist[(x >> s2) & dmask], 1u);
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
    }
  }

  // ---- ordered compaction
  const uint32_t lt = (1u << lane) - 1u;
  // this CTA's counts of keys above T (and the forced position) and equal to T
  {
    uint32_t gt = 0, eq = 0;
    for (int64_t base = 0; base < L; base += kRound) {
      if (!resident || !ranked) load_round(vals, lo, hi, forced, base, key);
      const int64_t p0 = lo + base + wid * (32 * kPer) + lane;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        gt += __popc(__ballot_sync(0xffffffffu, key[j] > T || p0 + 32 * j == forced));
        eq += __popc(__ballot_sync(0xffffffffu, key[j] == T && T != 0u));
      }
    }
    if (lane == 0) {
      atomicAdd(&s.tot_gt, gt);
      atomicAdd(&s.tot_eq, eq);
    }
  }
  csync(cs);
  if (threadIdx.x == 0) {
    // ranks in order: equal keys before this CTA, outputs before it, all outputs
    const uint32_t tg = tc::smem_u32(&s.tot_gt), te = tc::smem_u32(&s.tot_eq);
    uint32_t ce = 0, co = 0, ce_me = 0, co_me = 0;
    for (int r = 0; r < cs; ++r) {
      const uint32_t g = cs > 1 ? tc::ld_dsmem_u32(tc::map_rank(tg, r)) : s.tot_gt;
      const uint32_t e = cs > 1 ? tc::ld_dsmem_u32(tc::map_rank(te, r)) : s.tot_eq;
      if (r == rk) {
        ce_me = ce;
        co_me = co;
      }
      const uint32_t take = krem > ce ? min(krem - ce, e) : 0u;
      co += g + take;
      ce += e;
    }
    s.carry_eq = ce_me;
    s.carry_off = co_me;
    s.grand = co;
  }
  csync(cs);  // no CTA reads another's shared memory after this
  for (int64_t base = 0; base < L; base += kRound) {
    if (!resident || !ranked) load_round(vals, lo, hi, forced, base, key);
    const int64_t p0 = lo + base + wid * (32 * kPer) + lane;
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      gt += __popc(__ballot_sync(0xffffffffu, key[j] > T || p0 + 32 * j == forced));
      eq += __popc(__ballot_sync(0xffffffffu, key[j] == T && T != 0u));
    }
    if (lane == 0) {
      s.wa[wid] = gt;
      s.wb[wid] = eq;
    }
    __syncthreads();
    if (wid == 0) {
      const uint32_t g = s.wa[lane], e = s.wb[lane];
      uint32_t ie = e;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, ie, o);
        if (lane >= o) ie += y;
      }
      const uint32_t e_before = s.carry_eq + ie - e;
      const uint32_t take = krem > e_before ? min(krem - e_before, e) : 0u;
      const uint32_t v = g + take;
      uint32_t iv = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, iv, o);
        if (lane >= o) iv += y;
      }
      const uint32_t off = s.carry_off + iv - v;
      __syncwarp();
      s.wa[lane] = off;
      s.wb[lane] = e_before;
      if (lane == 31) {
        s.carry_eq += ie;
        s.carry_off += iv;
      }
    }
    __syncthreads();
    uint32_t off = s.wa[wid], e_run = s.wb[wid];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int64_t p = p0 + 32 * j;
      const bool is_eq = key[j] == T && T != 0u;
      const uint32_t be = __ballot_sync(0xffffffffu, is_eq);
      const bool sel = key[j] > T || p == forced || (is_eq && e_run + __popc(be & lt) < krem);
      const uint32_t bs = __ballot_sync(0xffffffffu, sel);
      const uint32_t o = off + __popc(bs & lt);
      if (sel && o < (uint32_t)k) out[o] = idmap(p);
      off += __popc(bs);
      e_run += __popc(be);
    }
    __syncthreads();
  }
  if (rk == cs - 1)
    for (uint32_t i = s.grand + threadIdx.x; i < (uint32_t)k; i += kSelThreads) out[i] = -1;
}

// grid (cs, queries, selections), clusters of cs CTAs along x.  Selection 0:
// entry top-k (Full or Reindex); 1: HSI block pool (Full).
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(int q0, int Tq, int r, int k, int n_blocks,
                                                                int64_t max_entries,
                                                                const int64_t* __restrict__ q_pos,
                                                                const int32_t* __restrict__ n_entries,
                                                                const int32_t* __restrict__ pool, const float* scores,
                                                                const float* bmax, int64_t score_stride,
                                                                const uint32_t* kmin, const uint32_t* kmax,
                                                                int32_t* topk_out, int32_t* pool_out) {
  extern __shared__ __align__(16) unsigned char sel_raw[];
  SelShared& s = *reinterpret_cast<SelShared*>(sel_raw);
  const int cs = (int)tc::cluster_size(), rk = (int)tc::cluster_rank();
  const int qc = blockIdx.y, qi = q0 + qc, b = qi / Tq;
  const int64_t nv = visible_entries(q_pos[qi], r, n_entries[b] < max_entries ? n_entries[b] : max_entries);
  const uint32_t lo = kmin[qc], hi = kmax[qc];
  if (blockIdx.z == 0) {
    const float* v = scores + (int64_t)qc * score_stride;
    if (pool)
      select_topk(v, (int64_t)n_blocks * kHsiBlock, k, -1, IdMap{pool + (int64_t)qi * n_blocks},
                  topk_out + (int64_t)qi * k, lo, hi, s, cs, rk);
    else
      select_topk(v, nv, k, -1, IdMap{nullptr}, topk_out + (int64_t)qi * k, lo, hi, s, cs, rk);
  } else {
    const int64_t nb = (nv + kHsiBlock - 1) / kHsiBlock;
    const float* v = bmax + (int64_t)qc * ((max_entries + 7) / 8);
    select_topk(v, nb, n_blocks, nb - 1, IdMap{nullptr}, pool_out + (int64_t)qi * n_blocks, lo, hi, s, cs, rk);
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// Per query: scores (Full: max_entries, Reindex: pool positions), HSI block
// maxima (Full with HSI), and the [min, max] key range (8 bytes, padded).
size_t index_query_ws_bytes(const csa2_cfg& cfg, int max_entries, bool reindex) {
  if (reindex) return align256((size_t)cfg.hsi_blocks * kHsiBlock * sizeof(float)) + 512;
  size_t b = align256((size_t)max_entries * sizeof(float));
  if (cfg.hsi_blocks > 0) b += align256((size_t)((max_entries + 7) / 8) * sizeof(float));
  return b + 512;
}

cudaError_t launch_index_topk(const csa2_cfg& cfg, int B, int Tq, const uint16_t* q_idx,
                              const float* head_w, const int64_t* q_pos, const csa2_cache& idx_c,
                              const int32_t* n_entries, int max_entries, const int32_t* pool,
                              int32_t* topk_out, int32_t* pool_out, void* ws, size_t ws_bytes,
                              int32_t* status, cudaStream_t stream) {
  const int Q = B * Tq;
  if (Q == 0) return cudaSuccess;
  const bool reindex = pool != nullptr;
  const size_t per_q = index_query_ws_bytes(cfg, max_entries, reindex);
  const int chunk = (int)std::min<size_t>(std::min<size_t>((size_t)Q, ws_bytes / per_q), 65535);  // grid y
  if (chunk < 1) return cudaErrorInvalidValue;
  float* scores = static_cast<float*>(ws);
  const int64_t stride = reindex ? (int64_t)cfg.hsi_blocks * kHsiBlock : (int64_t)max_entries;
  char* cur = static_cast<char*>(ws) + align256((size_t)chunk * stride * sizeof(float));
  float* bmax = nullptr;
  if (!reindex && pool_out) {
    bmax = reinterpret_cast<float*>(cur);
    cur += align256((size_t)chunk * ((max_entries + 7) / 8) * sizeof(float));
  }
  uint32_t* kmin = reinterpret_cast<uint32_t*>(cur);
  uint32_t* kmax = reinterpret_cast<uint32_t*>(cur + align256((size_t)chunk * sizeof(uint32_t)));
  for (int q0 = 0; q0 < Q; q0 += chunk) {
    const int nq = std::min(chunk, Q - q0);
    cudaMemsetAsync(kmin, 0xFF, (size_t)nq * sizeof(uint32_t), stream);  // empty ranges
    cudaMemsetAsync(kmax, 0x00, (size_t)nq * sizeof(uint32_t), stream);
    cudaError_t e = launch_score_tc(cfg, q0, nq, Tq, q_idx, head_w, q_pos, idx_c, n_entries, max_entries, pool, scores,
                                    stride, bmax, kmin, kmax, status, num_sms(), stream);
    if (e != cudaSuccess) return e;
    // one CTA per kRound positions of the longest selection, up to a cluster of 8
    const int64_t n_max = reindex ? (int64_t)cfg.hsi_blocks * kHsiBlock : (int64_t)max_entries;
    int cs = 1;
    while (cs < 8 && (int64_t)cs * kRound < n_max) cs <<= 1;
    const size_t sel_smem = sizeof(SelShared);
    cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sel_smem);
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(cs, nq, (!reindex && pool_out) ? 2 : 1);
    lc.blockDim = dim3(kSelThreads);
    lc.dynamicSmemBytes = sel_smem;
    lc.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    e = cudaLaunchKernelEx(&lc, select_kernel, q0, Tq, cfg.ratio, cfg.topk, cfg.hsi_blocks, (int64_t)max_entries,
                           q_pos, n_entries, pool, (const float*)scores, (const float*)bmax, stride,
                           (const uint32_t*)kmin, (const uint32_t*)kmax, topk_out, pool_out);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa2
