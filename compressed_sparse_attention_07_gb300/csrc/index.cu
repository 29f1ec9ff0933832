// a3..a6 -- CSA2 lightweight indexer: per-query scores over the visible
// indexer-K entries (or over an HSI pool), HSI block maxima, and exact
// top-k selection with the (score desc, id asc) order.
// (DeepSeek-V4.1 Flash, hn.213312.xyz sec. 2.3.1, 2.3.2, 2.3.4; 36kr "CSA2".)
#include <algorithm>

#include "internal.h"

namespace csa2 {
namespace {

constexpr int kSelThreads = 1024;   // one CTA selects for one query
constexpr int kHistBins = 8192;    // linear bins over a query's key range
constexpr int kCandMax = 8192;     // candidates sorted in shared memory
constexpr int kSelOutMax = 4096;   // k of one selection (top-k <= 1024, HSI blocks <= 4096)

// ---------------------------------------------------------------- select ----

// Exclusive prefix sum over the CTA (kSelThreads threads); returns the total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t w = warp_sums[lane];
    uint32_t ws = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, ws, o);
      if (lane >= o) ws += y;
    }
    warp_sums[lane] = ws - w;  // exclusive
    if (lane == 31) warp_sums[32] = ws;
  }
  __syncthreads();
  uint32_t res = warp_sums[wid] + x - v;
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

// Select the k largest keys among n positions of `vals` ((key desc, position
// asc)); `forced` (>= 0) gets the largest key.  Writes ids ascending to out[k],
// -1 padded.  Radix select (11/11/10-bit digits) then an ordered compaction.
// skeys: shared-memory copy of the n keys when it fits (every pass after the
// first then reads shared memory), else nullptr (every pass reads vals).
__device__ void block_select(const float* vals, int64_t n, int k, int64_t forced, IdMap idmap, int32_t* out,
                             uint32_t* skeys) {
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t warp_sums[33];
  __shared__ uint32_t sh_krem, sh_digit;
  auto gkey = [&](int64_t p) -> uint32_t { return p == forced ? 0xFFFFFFFFu : order_key(vals[p]); };
  auto key_at = [&](int64_t p) -> uint32_t { return skeys ? skeys[p] : gkey(p); };

  // count valid candidates (and stage the keys); range of the valid keys
  __shared__ uint32_t sh_min[32], sh_max[32];
  uint32_t cnt = 0, kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int64_t p = threadIdx.x; p < n; p += kSelThreads) {
    const uint32_t kk = gkey(p);
    if (skeys) skeys[p] = kk;
    if (kk != 0u) {
      ++cnt;
      kmin = min(kmin, kk);
      kmax = max(kmax, kk);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if ((threadIdx.x & 31) == 0) {
    sh_min[threadIdx.x >> 5] = kmin;
    sh_max[threadIdx.x >> 5] = kmax;
  }
  uint32_t nvalid;
  block_exclusive_scan(cnt, warp_sums, nvalid);  // (its barriers also publish sh_min / sh_max)
  kmin = sh_min[0];
  kmax = sh_max[0];
  for (int w = 1; w < kSelThreads / 32; ++w) {
    kmin = min(kmin, sh_min[w]);
    kmax = max(kmax, sh_max[w]);
  }

  uint32_t T = 0, krem = 0;  // select key > T, plus the first krem keys == T
  if (nvalid > (uint32_t)k) {
    // Radix select on x = key - kmin, from the top significant bit of the
    // range down, at most 11 bits per pass: binning relative to the range
    // spreads the keys over the bins even when they share their top bits.
    const uint32_t range = kmax - kmin;
    const int nbits = range ? 32 - __clz(range) : 0;
    uint32_t prefix = 0;  // the fixed top bits of x
    int fixed = 0;
    krem = (uint32_t)k;
    while (fixed < nbits) {
      const int w = min(11, nbits - fixed);
      const int sh = nbits - fixed - w;
      const uint32_t dmask = (1u << w) - 1u;
      for (int i = threadIdx.x; i < 2048; i += kSelThreads) hist[i] = 0;
      __syncthreads();
      for (int64_t p = threadIdx.x; p < n; p += kSelThreads) {
        const uint32_t kk = key_at(p);
        if (kk == 0u) continue;
        const uint32_t x = kk - kmin;
        const uint32_t top = (sh + w >= 32) ? 0u : (x >> (sh + w));
        if (top == prefix) atomicAdd(&hist[(x >> sh) & dmask], 1u);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // lane L owns bins [2048 - 64(L+1), 2048 - 64L): scan from the top
        const int lane = threadIdx.x;
        uint32_t sacc = 0;
        for (int i = 0; i < 64; ++i) sacc += hist[2047 - 64 * lane - i];
        uint32_t incl = sacc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - sacc;  // keys in higher bins than this lane's chunk
        const uint32_t kr = (fixed == 0) ? (uint32_t)k : sh_krem;
        if (excl < kr && incl >= kr) {
          uint32_t above = excl;
          for (int i = 0; i < 64; ++i) {
            const int d = 2047 - 64 * lane - i;
            if (above + hist[d] >= kr) {
              sh_digit = (uint32_t)d;
              sh_krem = kr - above;
              break;
            }
            above += hist[d];
          }
        }
      }
      __syncthreads();
      prefix = (prefix << w) | sh_digit;
      fixed += w;
      krem = sh_krem;
      __syncthreads();
    }
    T = kmin + prefix;
  }

  // ordered compaction: thread t scans the contiguous segment [t*seg, (t+1)*seg)
  const int64_t seg = (n + kSelThreads - 1) / kSelThreads;
  const int64_t lo = (int64_t)threadIdx.x * seg, hi = lo + seg < n ? lo + seg : n;
  uint32_t gt = 0, eq = 0;
  for (int64_t p = lo; p < hi; ++p) {
    uint32_t kk = key_at(p);
    gt += kk > T;
    eq += (kk == T) && (T != 0u);
  }
  uint32_t eq_total;
  uint32_t eq_before = block_exclusive_scan(eq, warp_sums, eq_total);
  uint32_t take = krem > eq_before ? min(krem - eq_before, eq) : 0u;
  uint32_t total;
  uint32_t off = block_exclusive_scan(gt + take, warp_sums, total);
  for (int64_t p = lo; p < hi && off < (uint32_t)k; ++p) {
    uint32_t kk = key_at(p);
    if (kk > T) {
      out[off++] = idmap(p);
    } else if (kk == T && T != 0u && take > 0) {
      out[off++] = idmap(p);
      --take;
    }
  }
  for (uint32_t i = total + threadIdx.x; i < (uint32_t)k; i += kSelThreads) out[i] = -1;
}

// Bitonic sort of P (a power of two) 64-bit keys in shared memory, descending
// or ascending; every thread of the CTA calls it.
__device__ void bitonic_sort(unsigned long long* a, int P, bool descending) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P / 2; i += kSelThreads) {
        const int lo = 2 * stride * (i / stride) + (i % stride), hi = lo + stride;
        const bool up = ((lo & size) == 0) != descending;  // this pair sorts ascending
        const unsigned long long x = a[lo], y = a[hi];
        if ((x > y) == up) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Top-k of one query from its scores in global memory in two passes:
// (1) histogram over kHistBins linear bins of the key range [kmin, kmax]
// recorded by the scoring kernel -> the bin holding the k-th key; (2) gather
// every key in that bin or above, as (key << 32 | ~position), sort them
// descending in shared memory -- the first k are the selection by (score
// desc, position asc) -- then sort the chosen positions ascending.  The
// forced position (HSI's latest block) always takes a slot.  Falls back to
// the radix select when more than kCandMax keys tie into the threshold bin.
__device__ void select_two_pass(const float* vals, int64_t n, int k, int64_t forced, IdMap idmap, int32_t* out,
                                uint32_t kmin, uint32_t kmax, uint32_t* hist, unsigned long long* cand) {
  __shared__ uint32_t sh_tb, sh_above, sh_total, sh_count;
  const bool any = kmin <= kmax;
  const uint32_t range = any ? kmax - kmin : 0u;
  const int nbits = range ? 32 - __clz(range) : 0;
  const int sh = nbits > 13 ? nbits - 13 : 0;
  const bool has_forced = forced >= 0 && forced < n;
  const uint32_t kk_need = (uint32_t)k - (has_forced ? 1u : 0u);
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) hist[i] = 0;
  if (threadIdx.x == 0) sh_count = 0;
  __syncthreads();
  if (any) {
    for (int64_t p = threadIdx.x; p < n; p += kSelThreads) {
      if (p == forced) continue;
      const uint32_t kk = order_key(vals[p]);
      if (kk != 0u) atomicAdd(&hist[(kk - kmin) >> sh], 1u);
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    // lane L owns bins [8192 - 256(L+1), 8192 - 256L): counts from the top
    const int lane = threadIdx.x;
    uint32_t sacc = 0;
    for (int i = 0; i < 256; ++i) sacc += hist[kHistBins - 1 - 256 * lane - i];
    uint32_t incl = sacc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    const uint32_t excl = incl - sacc;
    if (lane == 0) {
      sh_total = total;
      sh_tb = 0;
      sh_above = 0;
    }
    __syncwarp();
    if (total > kk_need && excl < kk_need && incl >= kk_need) {
      uint32_t above = excl;
      for (int i = 0; i < 256; ++i) {
        const int d = kHistBins - 1 - 256 * lane - i;
        if (above + hist[d] >= kk_need) {
          sh_tb = (uint32_t)d;
          sh_above = above;
          break;
        }
        above += hist[d];
      }
    }
  }
  __syncthreads();
  const uint32_t tb = sh_tb;
  const uint32_t cand_n = (sh_total > kk_need ? sh_above + hist[tb] : sh_total) + (has_forced ? 1u : 0u);
  if (cand_n > (uint32_t)kCandMax) {
    block_select(vals, n, k, forced, idmap, out, nullptr);
    return;
  }
  // (2) gather the candidates
  for (int64_t p = threadIdx.x; p < n; p += kSelThreads) {
    unsigned long long ck = 0ull;
    if (p == forced) {
      ck = (0xFFFFFFFFull << 32) | (0xFFFFFFFFu - (uint32_t)p);
    } else if (any) {
      const uint32_t kk = order_key(vals[p]);
      if (kk != 0u && ((kk - kmin) >> sh) >= tb) ck = ((unsigned long long)kk << 32) | (0xFFFFFFFFu - (uint32_t)p);
    }
    if (ck) cand[atomicAdd(&sh_count, 1u)] = ck;
  }
  __syncthreads();
  const int C = (int)sh_count;
  int P = 1;
  while (P < C) P <<= 1;
  for (int i = C + threadIdx.x; i < P; i += kSelThreads) cand[i] = 0ull;
  __syncthreads();
  bitonic_sort(cand, P, true);
  const int m = C < k ? C : k;
  // chosen positions, ascending
  int P2 = 1;
  while (P2 < m) P2 <<= 1;
  for (int i = threadIdx.x; i < P2; i += kSelThreads) {
    const unsigned long long v = (i < m) ? (unsigned long long)(0xFFFFFFFFu - (uint32_t)(cand[i] & 0xFFFFFFFFull))
                                         : ~0ull;
    cand[kCandMax + i] = v;
  }
  __syncthreads();
  bitonic_sort(cand + kCandMax, P2, false);
  for (int i = threadIdx.x; i < k; i += kSelThreads) out[i] = i < m ? idmap((int64_t)cand[kCandMax + i]) : -1;
}

// blockIdx.y == 0: entry top-k (Full or Reindex); == 1: HSI block pool (Full).
__global__ void __launch_bounds__(kSelThreads) select2_kernel(int q0, int Tq, int r, int k, int n_blocks,
                                                              int64_t max_entries, const int64_t* __restrict__ q_pos,
                                                              const int32_t* __restrict__ n_entries,
                                                              const int32_t* __restrict__ pool, const float* scores,
                                                              const float* bmax, int64_t score_stride,
                                                              const uint32_t* kmin, const uint32_t* kmax,
                                                              int32_t* topk_out, int32_t* pool_out) {
  extern __shared__ __align__(16) unsigned long long sel_smem[];
  unsigned long long* cand = sel_smem;                                             // [kCandMax + kSelOutMax]
  uint32_t* hist = reinterpret_cast<uint32_t*>(sel_smem + kCandMax + kSelOutMax);  // [kHistBins]
  const int qc = blockIdx.x, qi = q0 + qc, b = qi / Tq;
  const int64_t nv = visible_entries(q_pos[qi], r, n_entries[b] < max_entries ? n_entries[b] : max_entries);
  const uint32_t lo = kmin[qc], hi = kmax[qc];
  if (blockIdx.y == 0) {
    const float* v = scores + (int64_t)qc * score_stride;
    if (pool)
      select_two_pass(v, (int64_t)n_blocks * kHsiBlock, k, -1, IdMap{pool + (int64_t)qi * n_blocks},
                      topk_out + (int64_t)qi * k, lo, hi, hist, cand);
    else
      select_two_pass(v, nv, k, -1, IdMap{nullptr}, topk_out + (int64_t)qi * k, lo, hi, hist, cand);
  } else {
    const int64_t nb = (nv + kHsiBlock - 1) / kHsiBlock;
    const float* v = bmax + (int64_t)qc * ((max_entries + 7) / 8);
    select_two_pass(v, nb, n_blocks, nb - 1, IdMap{nullptr}, pool_out + (int64_t)qi * n_blocks, lo, hi, hist, cand);
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
    const size_t sel_smem = (kCandMax + kSelOutMax) * sizeof(unsigned long long) + kHistBins * sizeof(uint32_t);
    cudaFuncSetAttribute(select2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sel_smem);
    select2_kernel<<<sg, kSelThreads, sel_smem, stream>>>(q0, Tq, cfg.ratio, cfg.topk, cfg.hsi_blocks, max_entries,
                                                          q_pos, n_entries, pool, scores, bmax, stride, kmin, kmax,
                                                          topk_out, pool_out);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa2
