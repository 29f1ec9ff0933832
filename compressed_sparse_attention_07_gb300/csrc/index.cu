// a3..a6 -- CSA2 lightweight indexer: per-query scores over the visible
// indexer-K entries (or over an HSI pool), HSI block maxima, and exact
// top-k selection with the (score desc, id asc) order.
// (DeepSeek-V4.1 Flash, hn.213312.xyz sec. 2.3.1, 2.3.2, 2.3.4; 36kr "CSA2".)
#include <algorithm>

#include "internal.h"

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
  uint32_t hist[kHistBins];
  uint32_t cand[kCandMax];
  uint32_t wa[kSelWarps + 1], wb[kSelWarps + 1];
  uint32_t cut_bin, cut_above, cut_total, cand_n, carry_eq, carry_off;
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

// Keys of one round: lane l of warp w holds positions base + 512w + 32j + l
// (j < kPer); 0 for positions past n and for the forced one.
__device__ __forceinline__ void load_round(const float* vals, int64_t n, int64_t forced, int64_t base,
                                           uint32_t (&key)[kPer]) {
  const int64_t p0 = base + (threadIdx.x >> 5) * (32 * kPer) + (threadIdx.x & 31);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int64_t p = p0 + 32 * j;
    key[j] = (p < n && p != forced) ? order_key(vals[p]) : 0u;
  }
}

// Select the k largest keys among n positions of `vals` by (key desc,
// position asc); `forced` (>= 0) always takes a slot.  Writes the chosen ids
// in ascending position order to out[k], -1 padded.
//   1. histogram of the keys over kHistBins linear bins of the query's key
//      range [kmin, kmax] (recorded by the scoring kernel) -> the bin where
//      the count from the top reaches k;
//   2. the keys of that bin are listed in shared memory and refined 11 bits
//      at a time down to the exact threshold key T and the number krem of
//      keys equal to T that still fit (the first krem by position);
//   3. ordered compaction: warp ballots within 512-position runs, one scan
//      over the warps per round.
// Rounds of kRound positions; for n <= kRound the keys stay in registers
// after the first read.
__device__ void select_topk(const float* vals, int64_t n, int k, int64_t forced, IdMap idmap, int32_t* out,
                            uint32_t kmin, uint32_t kmax, SelShared& s) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const bool has_forced = forced >= 0 && forced < n;
  const uint32_t need = (uint32_t)k - (has_forced ? 1u : 0u);
  const bool any = kmin <= kmax;
  const uint32_t range = any ? kmax - kmin : 0u;
  const int nbits = range ? 32 - __clz(range) : 0;
  const int sh = nbits > 13 ? nbits - 13 : 0;
  const bool resident = n <= kRound;
  auto bin_of = [&](uint32_t kk) -> uint32_t {
    const uint32_t x = kk > kmin ? kk - kmin : 0u;
    return min(x >> sh, (uint32_t)(kHistBins - 1));
  };
  uint32_t key[kPer];

  uint32_t T = 0xFFFFFFFFu, krem = 0;  // select key > T, then the first krem keys == T
  if (need > 0 && any) {
    for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) s.hist[i] = 0;
    if (threadIdx.x == 0) s.cand_n = 0;
    __syncthreads();
    for (int64_t base = 0; base < n; base += kRound) {
      load_round(vals, n, forced, base, key);
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (key[j]) atomicAdd(&s.hist[bin_of(key[j])], 1u);
    }
    __syncthreads();
    find_cut(s.hist, kHistBins, need, s);
    if (s.cut_total <= need) {
      T = 0;  // every valid key
    } else {
      const uint32_t tb = s.cut_bin;
      const uint32_t c = s.hist[tb];
      uint32_t prefix = tb;
      int rem = sh;
      krem = need - s.cut_above;
      const bool listed = c <= (uint32_t)kCandMax;
      __syncthreads();  // every thread has read the cut and hist[tb]
      if (rem > 0 && listed) {
        for (int64_t base = 0; base < n; base += kRound) {
          if (!resident) load_round(vals, n, forced, base, key);
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
        __syncthreads();
      }
      while (rem > 0) {
        const int w = rem < 11 ? rem : 11;
        const int s2 = rem - w;
        const uint32_t dmask = (1u << w) - 1u;
        for (int i = threadIdx.x; i < kDigitBins; i += kSelThreads) s.hist[i] = 0;
        __syncthreads();
        if (listed) {
          const uint32_t cn = s.cand_n;
          for (uint32_t i = threadIdx.x; i < cn; i += kSelThreads) {
            const uint32_t x = s.cand[i];
            if ((x >> rem) == prefix) atomicAdd(&s.hist[(x >> s2) & dmask], 1u);
          }
        } else {
          for (int64_t base = 0; base < n; base += kRound) {
            if (!resident) load_round(vals, n, forced, base, key);
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
              const uint32_t x = key[j] - kmin;
              if (key[j] != 0u && key[j] >= kmin && (x >> rem) == prefix) atomicAdd(&s.hist[(x >> s2) & dmask], 1u);
            }
          }
        }
        __syncthreads();
        find_cut(s.hist, kDigitBins, krem, s);
        krem -= s.cut_above;
        prefix = (prefix << w) | s.cut_bin;
        rem = s2;
        __syncthreads();
      }
      T = kmin + prefix;
    }
  }

  // ordered compaction
  if (threadIdx.x == 0) {
    s.carry_eq = 0;
    s.carry_off = 0;
  }
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
  for (int64_t base = 0; base < n; base += kRound) {
    if (!resident || !(need > 0 && any)) load_round(vals, n, forced, base, key);
    const int64_t p0 = base + wid * (32 * kPer) + lane;
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
  for (uint32_t i = s.carry_off + threadIdx.x; i < (uint32_t)k; i += kSelThreads) out[i] = -1;
}

// blockIdx.y == 0: entry top-k (Full or Reindex); == 1: HSI block pool (Full).
__global__ void __launch_bounds__(kSelThreads) select_kernel(int q0, int Tq, int r, int k, int n_blocks,
                                                             int64_t max_entries, const int64_t* __restrict__ q_pos,
                                                             const int32_t* __restrict__ n_entries,
                                                             const int32_t* __restrict__ pool, const float* scores,
                                                             const float* bmax, int64_t score_stride,
                                                             const uint32_t* kmin, const uint32_t* kmax,
                                                             int32_t* topk_out, int32_t* pool_out) {
  extern __shared__ __align__(16) unsigned char sel_raw[];
  SelShared& s = *reinterpret_cast<SelShared*>(sel_raw);
  const int qc = blockIdx.x, qi = q0 + qc, b = qi / Tq;
  const int64_t nv = visible_entries(q_pos[qi], r, n_entries[b] < max_entries ? n_entries[b] : max_entries);
  const uint32_t lo = kmin[qc], hi = kmax[qc];
  if (blockIdx.y == 0) {
    const float* v = scores + (int64_t)qc * score_stride;
    if (pool)
      select_topk(v, (int64_t)n_blocks * kHsiBlock, k, -1, IdMap{pool + (int64_t)qi * n_blocks},
                  topk_out + (int64_t)qi * k, lo, hi, s);
    else
      select_topk(v, nv, k, -1, IdMap{nullptr}, topk_out + (int64_t)qi * k, lo, hi, s);
  } else {
    const int64_t nb = (nv + kHsiBlock - 1) / kHsiBlock;
    const float* v = bmax + (int64_t)qc * ((max_entries + 7) / 8);
    select_topk(v, nb, n_blocks, nb - 1, IdMap{nullptr}, pool_out + (int64_t)qi * n_blocks, lo, hi, s);
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
  const int chunk = (int)std::min<size_t>((size_t)Q, ws_bytes / per_q);
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
    dim3 sg(nq, (!reindex && pool_out) ? 2 : 1);
    const size_t sel_smem = sizeof(SelShared);
    cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sel_smem);
    select_kernel<<<sg, kSelThreads, sel_smem, stream>>>(q0, Tq, cfg.ratio, cfg.topk, cfg.hsi_blocks, max_entries,
                                                         q_pos, n_entries, pool, scores, bmax, stride, kmin, kmax,
                                                         topk_out, pool_out);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa2
