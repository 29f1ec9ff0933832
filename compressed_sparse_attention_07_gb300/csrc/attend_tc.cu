// a7 -- CSA2 sparse attention on the tensor cores.
//
// For one query token: rows E = the selected main-KV entries followed by the
// window rows; logits l = scale * q_h . c_e; one softmax per head over E;
// out_h = sum_e p_e c_e, the same 512-channel latent serving as key and value
// (DeepSeek-V4.1 Flash, hn.213312.xyz sec. 2.2.2 and sec. 3.3.1; 36kr "CSA2").
//
// Four kernels, chosen by the number of 128-row tiles (top-k tiles, then
// window tiles):
//  - attend_qc_kernel (4 or 5 tiles, the model's 512 + 128): a cluster of 4
//    or 5 CTAs per query, each holding 160 or 128 of its rows for all 64
//    heads; each CTA gathers and decodes its rows once, computes S = C.Q^T,
//    a partial softmax and O = C^T.P^T on the tensor cores, and the partial
//    outputs are merged through distributed shared memory; launched while
//    the selection still runs, it loads the query and window rows and
//    brings the block table into L2 before it waits for the selected ids
//    (in a Reuse layer it gathers its selected rows before the wait too);
//  - attend_rows_kernel (other counts up to 6 tiles): one CTA per (query,
//    tile), the query's tiles in one cluster, otherwise the same (these two
//    read MXFP8 window rows);
//  - attend_split_kernel (up to 16 tiles, few queries): the same with 16
//    heads per CTA;
//  - attend_tc_kernel (otherwise): one CTA per (query, group of HG heads)
//    over all of the query's tiles, described below.
//
// attend_tc_kernel processes the rows in tiles of 128 (each padded to 128
// rows) and 128-channel chunks:
//  - thread r of the CTA owns row r of every tile: it gathers that row into
//    a shared-memory staging ring with 16-byte cp.async copies, several units
//    ahead (whole FP4 rows, 256 B codes + 32 B scales, per top-k tile;
//    256-byte bf16 chunks per window or bf16-cache tile and chunk), then
//    decodes its row chunk to f16 into a K-major [128 rows x 128 channels]
//    tile C;
//  - phase A: thread 0 issues S^T[tile] += C . Q_chunk^T (M = 128 rows,
//    N = HG heads) into TMEM for every tile;
//  - softmax: exact two-pass per head over all rows from TMEM, P^T (f16) to
//    shared memory (over the Q tile, which phase A no longer needs);
//  - phase B: the rows are gathered and decoded again and
//    O^T[chunk] += C^T . P^T[tile] (M = 128 channels, A read MN-major from the
//    same C tile, N = HG heads) accumulates in TMEM;
//  - epilogue: O^T / row sums -> fp32 out (coalesced), natural-log LSE.
// FP4 values are exact in f16; bf16 Q / window rows are converted to f16
// (exact for magnitudes in [2^-17, 65504]); accumulation is fp32.
#include <algorithm>

#include "internal.h"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 512;  // four threads per row of a 128-row tile
constexpr int kStageRow = 304;                 // staged FP4 row: 256 codes + 32 scales + pad (bank spread)
constexpr int kStageRowChunk = 272;            // staged bf16 row chunk: 256 + pad
constexpr int kStageBytes = 128 * kStageRow;   // 38912
constexpr int kCBytes = 128 * 128 * 2;         // decoded f16 tile chunk
constexpr float kLog2e = 1.4426950408889634f;

struct AttArgs {
  int Tq, k, W, S;
  int tiles_main, tiles_win;
  const uint16_t* q;
  CacheView mc;
  const int32_t* n_entries;
  int64_t capacity;
  const int32_t* topk;
  const uint16_t* swa;   // bf16 window rows [B][S][512], or
  const uint8_t* swa8;   // MXFP8 window rows [B][S][528 B] (row-tile kernel only)
  const int32_t* swa_len;
  const int64_t* swa_pos0;
  const int64_t* q_pos;
  float scale;
  float* out;
  float* lse;
  int32_t* status;
  // the query-cluster kernel may read topk, n_entries and the main cache
  // before it waits for the previous kernel (a Reuse layer: the kernel
  // enqueued just before wrote none of them)
  int early;
};

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }


__device__ __forceinline__ uint32_t f16x2_from_f32(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return f16x2_from_f32(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Bit 15 / 31 set when the low / high f16 half is an infinity or NaN: the
// bf16 or MXFP8 value it came from lies outside the f16 range (|x| > 65504)
// or was not finite.  Kernels OR these bits over their conversions and
// report CSA2_ERR_RANGE.
__device__ __forceinline__ uint32_t f16x2_nonfinite(uint32_t h) {
  return ((h & 0x7C007C00u) + 0x04000400u) & 0x80008000u;
}

// bf16 pair -> f16 pair, recording an out-of-range value in `flag`.
__device__ __forceinline__ uint32_t to_f16x2(uint32_t w, uint32_t& flag) {
  const uint32_t h = bf16x2_to_f16x2(w);
  flag |= f16x2_nonfinite(h);
  return h;
}


__device__ __forceinline__ uint32_t f16x2_scale(uint32_t sbyte) {
  uint32_t r;
  uint16_t pair = (uint16_t)(sbyte | (sbyte << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(pair));
  return r;
}

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

// 16 MXFP8 elements (E4M3, element 2i in the low byte of pair i) with E8M0
// scale byte `sb` -> 8 f16x2, each the f16 nearest to E4M3 x 2^(sb - 127):
// the E4M3 -> f16 step is exact; the scale is applied by one f16 multiply
// when 2^(sb - 127) is an f16 value, else in fp32 (exact) and rounded once.
__device__ __forceinline__ void mxfp8x16_to_f16x2(uint4 w, uint32_t sb, uint32_t (&o)[8]) {
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint16_t lo = (uint16_t)(wv[i] & 0xFFFFu), hi = (uint16_t)(wv[i] >> 16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * i]) : "h"(lo));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * i + 1]) : "h"(hi));
  }
  const int e = (int)sb - 127;
  if (e >= -24 && e <= 15) {
    const uint32_t sh = e >= -14 ? (uint32_t)(e + 15) << 10 : 1u << (e + 24);
    const uint32_t s2 = sh | (sh << 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = hmul2(h[i], s2);
  } else {
    const float sf = e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << 22);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
      o[i] = f16x2_from_f32(f.x * sf, f.y * sf);
    }
  }
}

// Row source of slot i (tiles padded to 128), page already resolved:
// >= 0 main entry at page * 64 + slot of the page pool, <= -2 window row
// (-2 - row in swa), -1 empty.  Resolving the block table once here keeps
// dependent global loads off the gather path.
__device__ __forceinline__ int32_t slot_source(const AttArgs& a, int qi, int b, int i) {
  const int kp = a.tiles_main * 128;
  if (i < kp) {
    if (i >= a.k) return -1;
    const int32_t id = __ldg(a.topk + (int64_t)qi * a.k + i);
    if (id < 0) return -1;
    if (id >= __ldg(a.n_entries + b) || id >= a.capacity) {
      report(a.status, CSA2_ERR_BAD_INDEX);
      return -1;
    }
    const int64_t page = page_of(a.mc, b, id, a.status);
    if (page < 0) return -1;
    return (int32_t)(page * kPage + id % kPage);
  }
  const int w = i - kp;
  if (w >= a.W) return -1;
  const int64_t pos = __ldg(a.q_pos + qi) - a.W + 1 + w;
  const int64_t p0 = __ldg(a.swa_pos0 + b);
  int64_t len = __ldg(a.swa_len + b);
  len = len < a.S ? len : a.S;
  if (pos < 0 || pos < p0 || pos >= p0 + len) return -1;
  return (int32_t)(-2 - (pos - p0));
}

template <int kDtype, int HG, int kStages>
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(AttArgs a) {
  griddep_wait();  // before any global read or tensor-memory allocation
  griddep_launch();
  uint32_t rflag = 0;  // an f16 operand out of range (CSA2_ERR_RANGE)
  constexpr bool kMainFp4 = (kDtype == CSA2_CACHE_FP4);
  constexpr int CPT = HG / 4;  // TMEM columns (heads) per thread in softmax / epilogue
  const int n_tiles = a.tiles_main + a.tiles_win;
  const int nslot = n_tiles * 128;
  const int n_chunks = n_tiles * 4;                            // per phase
  const int units_main = kMainFp4 ? a.tiles_main : 4 * a.tiles_main;
  const int units_phase = units_main + 4 * a.tiles_win;
  const int tmem_cols = [&] {
    int need = n_tiles * HG > 4 * HG ? n_tiles * HG : 4 * HG;
    int c = 32;
    while (c < need) c <<= 1;
    return c;
  }();

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stage = smem;                                        // kStages x kStageBytes
  uint8_t* ctile = stage + kStages * kStageBytes;               // 2 x kCBytes
  uint8_t* qp = ctile + 2 * kCBytes;                            // Q tile, later P^T
  const int qp_bytes = max(HG * kDim * 2, nslot * HG * 2);
  int32_t* src = reinterpret_cast<int32_t*>(qp + qp_bytes);     // [nslot]
  __shared__ __align__(8) uint64_t cdone[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float red[4][HG];
  __shared__ float m_s[HG], inv_s[HG];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127;         // row of the tile (TMEM lane); channel in the epilogue
  const int p = tid >> 7;          // quarter of the row chunk / column group
  const int quad = warp & 3;       // TMEM lane quadrant this warp may access
  const uint32_t lane_base = 32 * quad;
  const int hg = blockIdx.x, qi = blockIdx.y, b = qi / a.Tq;

  // ---- set-up: row sources, Q (f16, K-major [HG][512]), barriers, TMEM
  for (int i = tid; i < nslot; i += kThreads) src[i] = slot_source(a, qi, b, i);
  for (int i = tid; i < HG * kDim / 8; i += kThreads) {
    const int h = (8 * i) / kDim, kk = (8 * i) % kDim;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(a.q + ((int64_t)qi * kHeads + hg * HG + h) * kDim + kk));
    *reinterpret_cast<uint4*>(qp + tc::kmajor_off(h, kk, kDim)) =
        make_uint4(to_f16x2(w.x, rflag), to_f16x2(w.y, rflag), to_f16x2(w.z, rflag), to_f16x2(w.w, rflag));
  }
  if (tid == 0) {
    tc::mbar_init(&cdone[0], 1);
    tc::mbar_init(&cdone[1], 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = tmem_base;

  // Gather quarter p of row r of staging unit u (2 phases x units_phase units)
  // into ring slot u % kStages with 16-byte cp.async copies; one commit group
  // per unit, empty or not.
  const int total_units = 2 * units_phase;
  auto gather = [&](int u) {
    if (u < total_units) {
      const int up = u % units_phase;
      int t, c;  // tile, chunk (-1: whole FP4 rows)
      if (up < units_main) {
        t = kMainFp4 ? up : up / 4;
        c = kMainFp4 ? -1 : up % 4;
      } else {
        t = a.tiles_main + (up - units_main) / 4;
        c = (up - units_main) % 4;
      }
      uint8_t* slot = stage + (u % kStages) * kStageBytes;
      const int32_t sidx = src[t * 128 + r];
      if (sidx >= 0) {
        const int64_t page = sidx / kPage;
        const int sl = sidx % kPage;
        if (c < 0) {
          const uint8_t* g = a.mc.data + page * kMainFp4Data + sl * (kDim / 2);
          uint8_t* d = slot + r * kStageRow;
#pragma unroll
          for (int j = p; j < 16; j += 4) cp16(d + 16 * j, g + 16 * j);
          if (p < 2) cp16(d + 256 + 16 * p, a.mc.scales + page * kMainFp4Scales + sl * (kDim / 16) + 16 * p);
        } else {
          const uint8_t* g = a.mc.data + page * kMainBf16Data + sl * (kDim * 2) + 256 * c;
          uint8_t* d = slot + r * kStageRowChunk;
#pragma unroll
          for (int j = p; j < 16; j += 4) cp16(d + 16 * j, g + 16 * j);
        }
      } else if (sidx <= -2) {
        const uint16_t* g = a.swa + ((int64_t)b * a.S + (-2 - (int64_t)sidx)) * kDim + 128 * c;
        uint8_t* d = slot + r * kStageRowChunk;
#pragma unroll
        for (int j = p; j < 16; j += 4) cp16(d + 16 * j, g + 8 * j);
      }
    }
    cp_commit();
  };
#pragma unroll
  for (int u = 0; u < kStages - 1; ++u) gather(u);

  constexpr uint32_t kIdescS = tc::idesc_f16(128, HG, false, false, false, false);
  constexpr uint32_t kIdescO = tc::idesc_f16(128, HG, false, false, true, false);
  int last_issued = -1, waited = -1;
  bool aborted = false;
  for (int n = 0; n < 2 * n_chunks; ++n) {
    const int ph = n / n_chunks, t = (n % n_chunks) / 4, c = n % 4;
    const bool fp4_tile = kMainFp4 && t < a.tiles_main;
    const int up = (t < a.tiles_main) ? (kMainFp4 ? t : 4 * t + c) : units_main + 4 * (t - a.tiles_main) + c;
    const int u = ph * units_phase + up;
    const int s = u % kStages;

    if (ph == 1 && n == n_chunks) {
      // ---------------- softmax over all rows (phase A complete)
      const int e = n - 1;
      const bool ok = tc::mbar_wait(&cdone[e & 1], (e >> 1) & 1);
      waited = e;
      if (!ok) atomicExch(&abort_flag, 1);
      tc::fence_after_sync();
      const float sc2 = a.scale * kLog2e;
      float m[CPT];
#pragma unroll
      for (int j = 0; j < CPT; ++j) m[j] = -INFINITY;
      for (int tt = 0; tt < n_tiles; ++tt) {
        const bool valid = src[tt * 128 + r] != -1;
        uint32_t v[CPT];
        tc::tmem_ld_n<CPT>(tc::taddr(tb, lane_base, tt * HG + p * CPT), v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < CPT; ++j)
          if (valid) m[j] = fmaxf(m[j], __uint_as_float(v[j]) * sc2);
      }
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m[j] = fmaxf(m[j], __shfl_xor_sync(0xffffffffu, m[j], o));
      }
      if (lane == 0)
#pragma unroll
        for (int j = 0; j < CPT; ++j) red[quad][p * CPT + j] = m[j];
      __syncthreads();
      if (tid < HG) m_s[tid] = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
      __syncthreads();
      float sum[CPT];
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        m[j] = m_s[p * CPT + j];
        sum[j] = 0.0f;
      }
      for (int tt = 0; tt < n_tiles; ++tt) {
        const bool valid = src[tt * 128 + r] != -1;
        const int row = tt * 128 + r;
        uint32_t v[CPT];
        tc::tmem_ld_n<CPT>(tc::taddr(tb, lane_base, tt * HG + p * CPT), v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          float pr = 0.0f;
          if (valid && m[j] != -INFINITY) pr = exp2f(__uint_as_float(v[j]) * sc2 - m[j]);
          sum[j] += pr;
          *reinterpret_cast<__half*>(qp + tc::kmajor_off(p * CPT + j, row, nslot)) = __float2half_rn(pr);
        }
      }
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum[j] += __shfl_xor_sync(0xffffffffu, sum[j], o);
      }
      __syncthreads();  // everyone has read red (maxima) before it is reused
      if (lane == 0)
#pragma unroll
        for (int j = 0; j < CPT; ++j) red[quad][p * CPT + j] = sum[j];
      __syncthreads();
      if (tid < HG) {
        const float tot = red[0][tid] + red[1][tid] + red[2][tid] + red[3][tid];
        inv_s[tid] = tot > 0.0f ? 1.0f / tot : 0.0f;
        if (a.lse)
          a.lse[(int64_t)qi * kHeads + hg * HG + tid] =
              tot > 0.0f ? (m_s[tid] + log2f(tot)) * 0.6931471805599453f : -INFINITY;
      }
      tc::fence_async_smem();
    }

    if (!fp4_tile || c == 0) {
      // unit u: this thread's copies done, then everyone's (barrier); the
      // barrier also frees the slot of unit u - 1 for the next refill
      cp_wait<kStages - 2>();
      __syncthreads();
      gather(u + kStages - 1);
    }
    // ---------------- decode quarter p of row chunk (t, c) into C tile n % 2
    if (n >= 2) {  // the MMAs that read this C tile two chunks ago must be done
      const int e = n - 2;
      if (e > waited) {
        if (!tc::mbar_wait(&cdone[e & 1], (e >> 1) & 1)) atomicExch(&abort_flag, 1);
        waited = e;
      }
    }
    {
      uint8_t* ct = ctile + (n & 1) * kCBytes;
      const uint8_t* slot = stage + s * kStageBytes;
      const int32_t sidx = src[t * 128 + r];
      uint32_t av[16];
      if (sidx == -1) {
#pragma unroll
        for (int j = 0; j < 16; ++j) av[j] = 0u;
      } else if (fp4_tile) {
        const uint8_t* row = slot + r * kStageRow;
        const uint32_t sc2b = *reinterpret_cast<const uint16_t*>(row + 256 + 8 * c + 2 * p);  // groups 2p, 2p+1
        const uint4 cw = *reinterpret_cast<const uint4*>(row + 64 * c + 16 * p);
        const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
        const uint32_t s_lo = f16x2_scale(sc2b & 0xFFu), s_hi = f16x2_scale(sc2b >> 8);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t h4[4];
          e2m1x8_to_f16x2(w4[q], h4);
#pragma unroll
          for (int by = 0; by < 4; ++by) av[4 * q + by] = hmul2(h4[by], q < 2 ? s_lo : s_hi);
        }
      } else {
        const uint8_t* row = slot + r * kStageRowChunk + 64 * p;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * j);
          av[4 * j] = to_f16x2(v.x, rflag);
          av[4 * j + 1] = to_f16x2(v.y, rflag);
          av[4 * j + 2] = to_f16x2(v.z, rflag);
          av[4 * j + 3] = to_f16x2(v.w, rflag);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(ct + tc::kmajor_off(r, 32 * p + 8 * j, 128)) =
            make_uint4(av[4 * j], av[4 * j + 1], av[4 * j + 2], av[4 * j + 3]);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (*reinterpret_cast<volatile int*>(&abort_flag)) {
      aborted = true;
      break;
    }
    if (tid == 0) {
      const uint32_t cbase = tc::smem_u32(ctile + (n & 1) * kCBytes);
      if (ph == 0) {
        // S^T[t] (+)= C[128 rows x 128 ch] . Q[:, chunk c]^T
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t ad = tc::sdesc(cbase + ks * 256, 128, 2048);
          const uint64_t bd = tc::sdesc(tc::smem_u32(qp) + (c * 16 + ks * 2) * 128, 128, kDim * 16);
          tc::mma_ss(tb + t * HG, ad, bd, kIdescS, (c > 0 || ks > 0) ? 1u : 0u);
        }
      } else {
        // O^T[chunk c] (+)= C^T[128 ch x 128 rows] . P^T[tile t]
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t ad = tc::sdesc(cbase + ks * 2 * 2048, 2048, 128);
          const uint64_t bd = tc::sdesc(tc::smem_u32(qp) + (t * 16 + ks * 2) * 128, 128, nslot * 16);
          tc::mma_ss(tb + c * HG, ad, bd, kIdescO, (t > 0 || ks > 0) ? 1u : 0u);
        }
      }
      tc::mma_commit(&cdone[n & 1]);
    }
    last_issued = n;
  }

  // ---------------- epilogue: O^T -> out
  cp_wait<0>();  // no copies into this CTA's shared memory outlive it
  if (last_issued > waited) {
    const bool ok = tc::mbar_wait(&cdone[last_issued & 1], (last_issued >> 1) & 1);
    if (!ok) aborted = true;
  }
  tc::fence_after_sync();
  if (!aborted) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t v[CPT];
      tc::tmem_ld_n<CPT>(tc::taddr(tb, lane_base, c * HG + p * CPT), v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        const int h = p * CPT + j;
        a.out[((int64_t)qi * kHeads + hg * HG + h) * kDim + c * 128 + r] = __uint_as_float(v[j]) * inv_s[h];
      }
    }
  } else if (tid == 0) {
    report(a.status, CSA2_ERR_TIMEOUT);
  }
  if (rflag) report(a.status, CSA2_ERR_RANGE);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, tmem_cols);
}


// ---------------------------------------------------------------------------
// Tile-split variant for few query tokens (decode).  One CTA per (query
// token, group of 16 heads, 128-row tile); the tiles of a query form a thread
// block cluster.  Each CTA gathers and decodes only its tile, keeps the four
// decoded 128-channel chunks in shared memory for both products, and computes
// a partial softmax (max m_t, sum l_t per head) with O_t = sum_e e^(l-m_t) c_e.
// The partials are merged through distributed shared memory: M = max_t m_t,
// L = sum_t e^(m_t-M) l_t, out = sum_t e^(m_t-M) O_t / L, each CTA of the
// cluster reducing one slice of the output (deterministic order over t).
constexpr int kSplitHG = 16;
constexpr int kSplitCPT = kSplitHG / 4;
constexpr size_t kSplitSmem = 2 * (size_t)kStageBytes + 4 * (size_t)kCBytes + kSplitHG * kDim * 2 + kSplitHG * 128 * 2 +
                              128 * 4 + 2 * kSplitHG * 4;

template <int kDtype>
__global__ void __launch_bounds__(kThreads, 1) attend_split_kernel(AttArgs a) {
  griddep_wait();  // before any global read or tensor-memory allocation
  griddep_launch();
  uint32_t rflag = 0;  // an f16 operand out of range (CSA2_ERR_RANGE)
  constexpr bool kMainFp4 = (kDtype == CSA2_CACHE_FP4);
  constexpr int HG = kSplitHG, CPT = kSplitCPT;
  const int n_tiles = a.tiles_main + a.tiles_win;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stage = smem;                                   // 2 staging slots
  uint8_t* ctile = stage + 2 * kStageBytes;                // 4 decoded chunks [128 rows x 128 ch] f16
  uint8_t* qs = ctile + 4 * kCBytes;                       // Q [16 heads x 512] f16, K-major
  uint8_t* pt = qs + HG * kDim * 2;                        // P^T [16 heads x 128 rows] f16, K-major
  int32_t* src = reinterpret_cast<int32_t*>(pt + HG * 128 * 2);  // [128]
  float* ml = reinterpret_cast<float*>(src + 128);         // m[16] (log2 domain), l[16]
  __shared__ __align__(8) uint64_t cdone;
  __shared__ uint32_t tmem_base;
  __shared__ float red[4][HG];
  __shared__ float m_s[HG], alpha[HG];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127, p = tid >> 7, quad = warp & 3;
  const uint32_t lane_base = 32 * quad;
  const int t = (int)tc::cluster_rank();                   // tile of this CTA
  const int hg = blockIdx.x / n_tiles, qi = blockIdx.y, b = qi / a.Tq;
  const bool fp4_tile = kMainFp4 && t < a.tiles_main;
  const int n_units = fp4_tile ? 1 : 4;

  // ---- set-up: row sources of this tile, Q, barrier, TMEM (S^T 16 cols, O^T 4 x 16)
  if (tid < 128) src[tid] = slot_source(a, qi, b, t * 128 + tid);
  for (int i = tid; i < HG * kDim / 8; i += kThreads) {
    const int h = (8 * i) / kDim, kk = (8 * i) % kDim;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(a.q + ((int64_t)qi * kHeads + hg * HG + h) * kDim + kk));
    *reinterpret_cast<uint4*>(qs + tc::kmajor_off(h, kk, kDim)) =
        make_uint4(to_f16x2(w.x, rflag), to_f16x2(w.y, rflag), to_f16x2(w.z, rflag), to_f16x2(w.w, rflag));
  }
  if (tid == 0) {
    tc::mbar_init(&cdone, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 128);
    tc::tmem_relinquish();
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = tmem_base;

  // quarter p of row r of unit u (whole FP4 rows, or 128-channel chunk u)
  auto gather = [&](int u) {
    if (u < n_units) {
      uint8_t* slot = stage + (u & 1) * kStageBytes;
      const int32_t sidx = src[r];
      if (sidx >= 0) {
        const int64_t page = sidx / kPage;
        const int sl = sidx % kPage;
        if (fp4_tile) {
          const uint8_t* g = a.mc.data + page * kMainFp4Data + sl * (kDim / 2);
          uint8_t* d = slot + r * kStageRow;
#pragma unroll
          for (int j = p; j < 16; j += 4) cp16(d + 16 * j, g + 16 * j);
          if (p < 2) cp16(d + 256 + 16 * p, a.mc.scales + page * kMainFp4Scales + sl * (kDim / 16) + 16 * p);
        } else {
          const uint8_t* g = a.mc.data + page * kMainBf16Data + sl * (kDim * 2) + 256 * u;
          uint8_t* d = slot + r * kStageRowChunk;
#pragma unroll
          for (int j = p; j < 16; j += 4) cp16(d + 16 * j, g + 16 * j);
        }
      } else if (sidx <= -2) {
        const uint16_t* g = a.swa + ((int64_t)b * a.S + (-2 - (int64_t)sidx)) * kDim + 128 * u;
        uint8_t* d = slot + r * kStageRowChunk;
#pragma unroll
        for (int j = p; j < 16; j += 4) cp16(d + 16 * j, g + 8 * j);
      }
    }
    cp_commit();
  };
  gather(0);
  gather(1);

  // ---- phase A: decode chunk c into C[c], S^T += C[c] . Q_c^T
  constexpr uint32_t kIdescS = tc::idesc_f16(128, HG, false, false, false, false);
  constexpr uint32_t kIdescO = tc::idesc_f16(128, HG, false, false, true, false);
  const int32_t sidx = src[r];
  for (int c = 0; c < 4; ++c) {
    const int u = fp4_tile ? 0 : c;
    if (!fp4_tile || c == 0) {
      cp_wait<1>();
      __syncthreads();
    }
    const uint8_t* slot = stage + (u & 1) * kStageBytes;
    uint32_t av[16];
    if (sidx == -1) {
#pragma unroll
      for (int j = 0; j < 16; ++j) av[j] = 0u;
    } else if (fp4_tile) {
      const uint8_t* row = slot + r * kStageRow;
      const uint32_t sc2b = *reinterpret_cast<const uint16_t*>(row + 256 + 8 * c + 2 * p);
      const uint4 cw = *reinterpret_cast<const uint4*>(row + 64 * c + 16 * p);
      const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
      const uint32_t s_lo = f16x2_scale(sc2b & 0xFFu), s_hi = f16x2_scale(sc2b >> 8);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t h4[4];
        e2m1x8_to_f16x2(w4[q], h4);
#pragma unroll
        for (int by = 0; by < 4; ++by) av[4 * q + by] = hmul2(h4[by], q < 2 ? s_lo : s_hi);
      }
    } else {
      const uint8_t* row = slot + r * kStageRowChunk + 64 * p;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * j);
        av[4 * j] = to_f16x2(v.x, rflag);
        av[4 * j + 1] = to_f16x2(v.y, rflag);
        av[4 * j + 2] = to_f16x2(v.z, rflag);
        av[4 * j + 3] = to_f16x2(v.w, rflag);
      }
    }
    uint8_t* ct = ctile + c * kCBytes;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(ct + tc::kmajor_off(r, 32 * p + 8 * j, 128)) =
          make_uint4(av[4 * j], av[4 * j + 1], av[4 * j + 2], av[4 * j + 3]);
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (!fp4_tile) gather(c + 2);  // every thread is done with the slot of unit c
    if (tid == 0) {
      const uint32_t cbase = tc::smem_u32(ct);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t ad = tc::sdesc(cbase + ks * 256, 128, 2048);
        const uint64_t bd = tc::sdesc(tc::smem_u32(qs) + (c * 16 + ks * 2) * 128, 128, kDim * 16);
        tc::mma_ss(tb, ad, bd, kIdescS, (c > 0 || ks > 0) ? 1u : 0u);
      }
      if (c == 3) tc::mma_commit(&cdone);
    }
  }
  cp_wait<0>();
  bool ok = tc::mbar_wait(&cdone, 0);
  tc::fence_after_sync();

  // ---- partial softmax over this tile's rows
  const float sc2 = a.scale * kLog2e;
  const bool valid = sidx != -1;
  float v[CPT];
  {
    uint32_t w[CPT];
    tc::tmem_ld_n<CPT>(tc::taddr(tb, lane_base, p * CPT), w);
    tc::tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < CPT; ++j) v[j] = valid ? __uint_as_float(w[j]) * sc2 : -INFINITY;
  }
  float m[CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    m[j] = v[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m[j] = fmaxf(m[j], __shfl_xor_sync(0xffffffffu, m[j], o));
  }
  if (lane == 0)
#pragma unroll
    for (int j = 0; j < CPT; ++j) red[quad][p * CPT + j] = m[j];
  __syncthreads();
  if (tid < HG) m_s[tid] = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
  __syncthreads();
  float sum[CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const float mh = m_s[p * CPT + j];
    const float pr = (valid && mh != -INFINITY) ? exp2f(v[j] - mh) : 0.0f;
    *reinterpret_cast<__half*>(pt + tc::kmajor_off(p * CPT + j, r, 128)) = __float2half_rn(pr);
    sum[j] = pr;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum[j] += __shfl_xor_sync(0xffffffffu, sum[j], o);
  }
  __syncthreads();  // red (maxima) read by every thread above
  if (lane == 0)
#pragma unroll
    for (int j = 0; j < CPT; ++j) red[quad][p * CPT + j] = sum[j];
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid < HG) {
    ml[tid] = m_s[tid];
    ml[HG + tid] = red[0][tid] + red[1][tid] + red[2][tid] + red[3][tid];
  }
  // ---- phase B: O^T[c] = C[c]^T . P^T for the four chunks
  if (tid == 0) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t cbase = tc::smem_u32(ctile + c * kCBytes);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t ad = tc::sdesc(cbase + ks * 2 * 2048, 2048, 128);
        const uint64_t bd = tc::sdesc(tc::smem_u32(pt) + ks * 256, 128, 2048);
        tc::mma_ss(tb + 32 + 16 * c, ad, bd, kIdescO, ks > 0 ? 1u : 0u);
      }
    }
    tc::mma_commit(&cdone);
  }
  // ---- merge the tiles' (m, l); every CTA of the cluster has written its own,
  // and every CTA is past its gathers, so the staging slots are free
  tc::cluster_sync();
  const int n = n_tiles;
  if (tid < HG) {
    const uint32_t ml_addr = tc::smem_u32(ml);
    float mk[16], lk[16];
#pragma unroll
    for (int k2 = 0; k2 < 16; ++k2) {
      if (k2 < n) {
        mk[k2] = tc::ld_dsmem(tc::map_rank(ml_addr + 4 * tid, k2));
        lk[k2] = tc::ld_dsmem(tc::map_rank(ml_addr + 4 * (HG + tid), k2));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int k2 = 0; k2 < 16; ++k2)
      if (k2 < n) M = fmaxf(M, mk[k2]);
    float L = 0.0f;
#pragma unroll
    for (int k2 = 0; k2 < 16; ++k2)
      if (k2 < n && mk[k2] != -INFINITY) L += exp2f(mk[k2] - M) * lk[k2];
    alpha[tid] = (L > 0.0f && ml[tid] != -INFINITY) ? exp2f(ml[tid] - M) / L : 0.0f;
    if (t == 0 && a.lse)
      a.lse[(int64_t)qi * kHeads + hg * HG + tid] = L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
  ok = tc::mbar_wait(&cdone, 1) && ok;
  tc::fence_after_sync();
  __syncthreads();
  // ---- push the scaled partial output to the CTA owning each output slice:
  // element e = head * 512 + channel belongs to CTA e / slice and lands in its
  // staging area at [sender tile][e - owner start]
  const int E = HG * kDim;
  const int slice = (E + n - 1) / n;
  const uint32_t recv = tc::smem_u32(stage);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t w[CPT];
    tc::tmem_ld_n<CPT>(tc::taddr(tb, lane_base, 32 + 16 * c + p * CPT), w);
    tc::tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int h = p * CPT + j, e = h * kDim + c * 128 + r;
      const int o = e / slice;
      const float val = ok ? __uint_as_float(w[j]) * alpha[h] : 0.0f;
      tc::st_dsmem(tc::map_rank(recv + 4 * (t * slice + (e - o * slice)), o), val);
    }
  }
  if (!ok && tid == 0) report(a.status, CSA2_ERR_TIMEOUT);
  if (rflag) report(a.status, CSA2_ERR_RANGE);
  tc::fence_before_sync();
  tc::cluster_sync();
  // ---- this CTA's slice: sum the tiles' partials in tile order
  {
    const float* rv = reinterpret_cast<const float*>(stage);
    const int lo = t * slice, hi = min(E, lo + slice);
    for (int e = lo + tid; e < hi; e += kThreads) {
      float acc = 0.0f;
      for (int k2 = 0; k2 < n; ++k2) acc += rv[k2 * slice + (e - lo)];
      const int h = e / kDim, ch = e % kDim;
      a.out[((int64_t)qi * kHeads + hg * HG + h) * kDim + ch] = acc;
    }
  }
  if (warp == 0) tc::tmem_dealloc(tb, 128);
}

// ---------------------------------------------------------------------------
// Row-tile variant for every head at once (at most six 128-row tiles per
// query: top-k <= 512 with window <= 256, or similar).  One CTA per (query
// token, 128-row tile), the query's tiles forming a cluster.  Each row is
// read once: thread (r, p) loads quarter p of row r (one 128-channel chunk)
// straight into registers, decodes it and stores it to the K-major chunk
// tile C[p]; then
//   S^T[128 rows x 64 heads]  = sum_c C[c] . Q_c^T       (M 128, N 64, K 512)
//   partial softmax per head over the tile's rows: m_t, l_t, P = 2^(s - m_t)
//   O_t^T[c] = C[c]^T . P^T                            (M 128, N 64, K 128)
// and the tiles are merged through distributed shared memory: every CTA
// keeps its O_t in its own shared memory, and the CTA of rank c % n pulls
// chunk c of every tile and forms out = sum_t 2^(m_t - M) O_t / L in tile
// order (M = max_t m_t, L = sum_t 2^(m_t - M) l_t).
constexpr int kAllHeads = 64;
constexpr size_t kRowQBytes = (size_t)kAllHeads * kDim * 2;   // 65536
constexpr size_t kRowCBytes = 4 * (size_t)kCBytes;            // 131072
constexpr size_t kRowPBytes = (size_t)kAllHeads * 128 * 2;    // 16384
constexpr size_t kRowSmem = kRowQBytes + kRowCBytes + kRowPBytes + 128 * 4 + 2 * kAllHeads * 4;
constexpr int kRowMaxTiles = 6;

// Reduce v[16] over the 32 lanes of a warp (op = max or +): afterwards lane l
// holds the result for entry l >> 1.  Each step hands half of the entries
// still held to the partner lane, 8 + 4 + 2 + 1 + 1 shuffles in all.
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(const float (&v)[16]) {
  const int lane = threadIdx.x & 31;
  auto op = [](float x, float y) { return kMax ? fmaxf(x, y) : x + y; };
  float a8[8], a4[4], a2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float keep = b4 ? v[8 + i] : v[i], send = b4 ? v[i] : v[8 + i];
    a8[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b3 ? a8[4 + i] : a8[i], send = b3 ? a8[i] : a8[4 + i];
    a4[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b2 ? a4[2 + i] : a4[i], send = b2 ? a4[i] : a4[2 + i];
    a2[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  const float keep = b1 ? a2[1] : a2[0], send = b1 ? a2[0] : a2[1];
  float a1 = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  return op(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
}

template <int kDtype, bool kSwaFp8>
__global__ void __launch_bounds__(kThreads, 1)
    attend_rows_kernel(AttArgs a) {
  constexpr bool kMainFp4 = (kDtype == CSA2_CACHE_FP4);
  const int n = a.tiles_main + a.tiles_win;
  uint32_t rflag = 0;  // an f16 operand out of range (CSA2_ERR_RANGE)
  if (threadIdx.x < 32) {
    // While the previous kernel (the selection) runs, the first warp brings
    // this query's inputs that do not depend on the selected ids into L2:
    // the query rows (cluster rank 0), the window rows (rank 1 % n) and, once
    // per sequence, its main-cache block table (rank n - 1).  Only hints are
    // issued; the values read to aim them are read again after the wait.
    const int lane = threadIdx.x, rk = (int)tc::cluster_rank(), qi = blockIdx.y, b = qi / a.Tq;
    if (rk == 0 && lane < 16)  // 64 x 512 bf16 = 64 KB in 4 KB pieces
      tc::bulk_prefetch_l2(a.q + (int64_t)qi * kHeads * kDim + lane * 2048, 4096);
    if (rk == 1 % n && a.W > 0 && a.Tq <= 8) {
      const int64_t pos = tc::ld_cg_s64(a.q_pos + qi), p0 = tc::ld_cg_s64(a.swa_pos0 + b);
      int64_t len = tc::ld_cg_s32(a.swa_len + b);
      len = len < a.S ? len : a.S;
      const int64_t lo = pos - a.W + 1 > p0 ? pos - a.W + 1 : p0, hi = pos < p0 + len - 1 ? pos : p0 + len - 1;
      if (lo <= hi) {  // slab rows lo - p0 .. hi - p0, all in [0, S)
        const int64_t rb = kSwaFp8 ? kSwaFp8Row : kDim * 2;
        const uint8_t* base =
            (kSwaFp8 ? a.swa8 : reinterpret_cast<const uint8_t*>(a.swa)) + ((int64_t)b * a.S + (lo - p0)) * rb;
        const int64_t bytes = (hi - lo + 1) * rb;
        for (int64_t off = (int64_t)lane * 4096; off < bytes; off += 32 * 4096)
          tc::bulk_prefetch_l2(base + off, (uint32_t)(bytes - off < 4096 ? bytes - off : 4096));
      }
    }
    if (rk == n - 1 && qi % a.Tq == 0) {
      int64_t np = (a.capacity + kPage - 1) / kPage;
      np = np < a.mc.max_pages ? np : a.mc.max_pages;
      const char* bt = reinterpret_cast<const char*>(a.mc.block_table + (int64_t)b * a.mc.max_pages);
      for (int64_t off = (int64_t)lane * 128; off < 4 * np; off += 32 * 128) tc::prefetch_l2(bt + off);
    }
  }
  griddep_wait();  // before any other global read or tensor-memory allocation
  griddep_launch();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* qs = smem;                                     // Q [64 heads x 512] f16, K-major
  uint8_t* ctile = qs + kRowQBytes;                       // C [128 rows x 512 ch] f16, K-major
  uint8_t* pt = ctile + kRowCBytes;                       // P^T [64 heads x 128 rows] f16, K-major
  int32_t* srcs = reinterpret_cast<int32_t*>(pt + kRowPBytes);      // row sources [128]
  float* ml = reinterpret_cast<float*>(pt + kRowPBytes + 128 * 4);  // m[64] (log2 domain), l[64]
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ float red_m[4][kAllHeads], red_s[4][kAllHeads];
  __shared__ float mx[kAllHeads], fac[kRowMaxTiles][kAllHeads];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127, p = tid >> 7, quad = warp & 3;
  const uint32_t lane_base = 32 * quad;
  const int t = (int)tc::cluster_rank();
  const int qi = blockIdx.y, b = qi / a.Tq;
  // this CTA's rows: 8-row groups of the query's slots dealt round-robin over
  // the cluster (warp w takes slot group w * n + t), so that every CTA gets
  // about the same share of FP4 top-k rows and bf16 window rows; the softmax
  // and the merge see the rows as a set
  const int slot0 = 8 * (warp * n + t);
  const bool fp4_tile = kMainFp4 && slot0 < a.tiles_main * 128;
  const bool fp8_win = kSwaFp8 && slot0 >= a.tiles_main * 128;  // an 8-row group of MXFP8 window rows

  // ---- loads, coalesced: warp w fills the 8-row group w of C (and half of
  // the 8-head group w % 8 of Q); lane l takes row 8w + l % 8 and 16-byte
  // units 4k + l / 8, so each row is read in 64-byte runs and every warp-wide
  // store covers whole 128-byte core-matrix rows
  const int rl = lane & 7, uq = lane >> 3;
  const int rho = 8 * warp + rl;
  const int32_t sidx_l = slot_source(a, qi, b, slot0 + rl);
  uint4 qv[8];
  {
    const int h = 8 * (warp & 7) + rl, u0 = 32 * (warp >> 3);
    const uint4* g = reinterpret_cast<const uint4*>(a.q + ((int64_t)qi * kHeads + h) * kDim);
#pragma unroll
    for (int k = 0; k < 8; ++k) qv[k] = __ldg(g + u0 + 4 * k + uq);
  }
  uint4 raw[16];
  uint32_t scl[4];
  if (sidx_l >= 0) {
    const int64_t page = sidx_l / kPage;
    const int sl = sidx_l % kPage;
    if (fp4_tile) {
      const uint4* g = reinterpret_cast<const uint4*>(a.mc.data + page * kMainFp4Data + sl * (kDim / 2));
      const uint16_t* gs = reinterpret_cast<const uint16_t*>(a.mc.scales + page * kMainFp4Scales + sl * (kDim / 16));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        raw[k] = __ldg(g + 4 * k + uq);
        scl[k] = __ldg(gs + 4 * k + uq);
      }
    } else {
      const uint4* g = reinterpret_cast<const uint4*>(a.mc.data + page * kMainBf16Data + sl * (kDim * 2));
#pragma unroll
      for (int k = 0; k < 16; ++k) raw[k] = __ldg(g + 4 * k + uq);
    }
  } else if (sidx_l <= -2) {
    if (kSwaFp8) {  // 32 units of 16 elements, lane units 4k + l/8; then the 16 scale bytes
      const uint4* g =
          reinterpret_cast<const uint4*>(a.swa8 + ((int64_t)b * a.S + (-2 - (int64_t)sidx_l)) * kSwaFp8Row);
#pragma unroll
      for (int k = 0; k < 8; ++k) raw[k] = __ldg(g + 4 * k + uq);
      raw[8] = __ldg(g + 32);
    } else {
      const uint4* g = reinterpret_cast<const uint4*>(a.swa + ((int64_t)b * a.S + (-2 - (int64_t)sidx_l)) * kDim);
#pragma unroll
      for (int k = 0; k < 16; ++k) raw[k] = __ldg(g + 4 * k + uq);
    }
  }
  if (uq == 0) srcs[rho] = sidx_l;
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 512);
    tc::tmem_relinquish();
  }
  {
    const int h = 8 * (warp & 7) + rl, u0 = 32 * (warp >> 3);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      *reinterpret_cast<uint4*>(qs + tc::kmajor_off(h, 8 * (u0 + 4 * k + uq), kDim)) =
          make_uint4(to_f16x2(qv[k].x, rflag), to_f16x2(qv[k].y, rflag), to_f16x2(qv[k].z, rflag),
                     to_f16x2(qv[k].w, rflag));
  }
  // ---- decode into C: FP4 code chunk q = 4k + l/8 (32 channels, two scale
  // groups) -> units 4q..4q+3; bf16 unit u = 4k + l/8 -> unit u
  if (fp4_tile) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int q = 4 * k + uq;
      const uint32_t s_lo = f16x2_scale(scl[k] & 0xFFu), s_hi = f16x2_scale((scl[k] >> 8) & 0xFFu);
      const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 o = make_uint4(0, 0, 0, 0);
        if (sidx_l >= 0) {
          uint32_t h4[4];
          e2m1x8_to_f16x2(w4[i], h4);
          const uint32_t s2 = i < 2 ? s_lo : s_hi;
          o = make_uint4(hmul2(h4[0], s2), hmul2(h4[1], s2), hmul2(h4[2], s2), hmul2(h4[3], s2));
        }
        *reinterpret_cast<uint4*>(ctile + tc::kmajor_off(rho, 32 * q + 8 * i, kDim)) = o;
      }
    }
  } else if (fp8_win) {
    // MXFP8 unit u = 4k + l/8: channels 16u..16u+15, scale byte u/2
    const uint32_t sw[4] = {raw[8].x, raw[8].y, raw[8].z, raw[8].w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int u = 4 * k + uq, blk = u >> 1;
      uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (sidx_l != -1) mxfp8x16_to_f16x2(raw[k], (sw[blk >> 2] >> (8 * (blk & 3))) & 0xFFu, o);
#pragma unroll
      for (int i = 0; i < 8; ++i) rflag |= f16x2_nonfinite(o[i]);
      *reinterpret_cast<uint4*>(ctile + tc::kmajor_off(rho, 16 * u, kDim)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(ctile + tc::kmajor_off(rho, 16 * u + 8, kDim)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint4 o = sidx_l == -1 ? make_uint4(0, 0, 0, 0)
                                   : make_uint4(to_f16x2(raw[k].x, rflag), to_f16x2(raw[k].y, rflag),
                                                to_f16x2(raw[k].z, rflag), to_f16x2(raw[k].w, rflag));
      *reinterpret_cast<uint4*>(ctile + tc::kmajor_off(rho, 8 * (4 * k + uq), kDim)) = o;
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = tmem_base;
  const int32_t sidx = srcs[r];  // the row this thread reads from TMEM below
  bool ok = true;

  // ---- S^T = sum over 16-channel steps of C . Q^T
  constexpr uint32_t kIdescS = tc::idesc_f16(128, kAllHeads, false, false, false, false);
  constexpr uint32_t kIdescO = tc::idesc_f16(128, kAllHeads, false, false, true, false);
  if (tid == 0 && ok) {
#pragma unroll 4
    for (int ks = 0; ks < kDim / 16; ++ks) {
      const uint64_t ad = tc::sdesc(tc::smem_u32(ctile) + ks * 256, 128, kDim * 16);
      const uint64_t bd = tc::sdesc(tc::smem_u32(qs) + ks * 256, 128, kDim * 16);
      tc::mma_ss(tb, ad, bd, kIdescS, ks > 0 ? 1u : 0u);
    }
  }
  if (tid == 0) tc::mma_commit(&bar);
  ok = tc::mbar_wait(&bar, 0) && ok;
  tc::fence_after_sync();

  // ---- partial softmax over the tile's rows (thread: row r, heads 16p..16p+15)
  const float sc2 = a.scale * kLog2e;
  const bool valid = sidx != -1;
  float v[16];
  {
    uint32_t w[16];
    tc::tmem_ld16(tc::taddr(tb, lane_base, 16 * p), w);
    tc::tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = valid ? __uint_as_float(w[j]) * sc2 : -INFINITY;
  }
  {
    const float wm = warp_reduce16<true>(v);
    if ((lane & 1) == 0) red_m[quad][16 * p + (lane >> 1)] = wm;
  }
  __syncthreads();
  if (tid < kAllHeads) mx[tid] = fmaxf(fmaxf(red_m[0][tid], red_m[1][tid]), fmaxf(red_m[2][tid], red_m[3][tid]));
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float mh = mx[16 * p + j];
    v[j] = (valid && mh != -INFINITY) ? exp2f(v[j] - mh) : 0.0f;
    *reinterpret_cast<__half*>(pt + tc::kmajor_off(16 * p + j, r, 128)) = __float2half_rn(v[j]);
  }
  {
    const float ws = warp_reduce16<false>(v);
    if ((lane & 1) == 0) red_s[quad][16 * p + (lane >> 1)] = ws;
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid < kAllHeads) {
    ml[tid] = mx[tid];
    ml[kAllHeads + tid] = red_s[0][tid] + red_s[1][tid] + red_s[2][tid] + red_s[3][tid];
  }

  // ---- O^T[c] = C[:, chunk c]^T . P^T (C read MN-major: 8-row groups 8 KB apart)
  if (tid == 0) {
    if (ok) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t cbase = tc::smem_u32(ctile) + c * 16 * 128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t ad = tc::sdesc(cbase + ks * 2 * (kDim * 16), kDim * 16, 128);
          const uint64_t bd = tc::sdesc(tc::smem_u32(pt) + ks * 256, 128, 2048);
          tc::mma_ss(tb + kAllHeads + kAllHeads * c, ad, bd, kIdescO, ks > 0 ? 1u : 0u);
        }
      }
    }
    tc::mma_commit(&bar);
  }
  ok = tc::mbar_wait(&bar, 1) && ok;
  tc::fence_after_sync();
  // ---- this tile's unscaled partial output into its own shared memory (Q and
  // C are free now), [chunk][head][channel]: a warp's stores are 128
  // contiguous bytes
  float* stg = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t w[16];
    tc::tmem_ld16(tc::taddr(tb, lane_base, kAllHeads + kAllHeads * c + 16 * p), w);
    tc::tmem_wait_ld();
    float* dst = stg + (c * kAllHeads + 16 * p) * 128 + r;
#pragma unroll
    for (int j = 0; j < 16; ++j) dst[128 * j] = __uint_as_float(w[j]);
  }
  tc::fence_before_sync();
  // every CTA of the cluster: (m, l) and its partial output written
  tc::cluster_sync();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tb, 512);
  // per-head factor of every tile: 2^(m_t - M) / L, M = max_t m_t, L = sum_t 2^(m_t - M) l_t
  if (tid < kAllHeads) {
    const uint32_t ml_addr = tc::smem_u32(ml);
    float mk[kRowMaxTiles], lk[kRowMaxTiles];
#pragma unroll
    for (int k2 = 0; k2 < kRowMaxTiles; ++k2) {
      mk[k2] = k2 < n ? tc::ld_dsmem(tc::map_rank(ml_addr + 4 * tid, k2)) : -INFINITY;
      lk[k2] = k2 < n ? tc::ld_dsmem(tc::map_rank(ml_addr + 4 * (kAllHeads + tid), k2)) : 0.0f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int k2 = 0; k2 < kRowMaxTiles; ++k2) M = fmaxf(M, mk[k2]);
    float L = 0.0f;
#pragma unroll
    for (int k2 = 0; k2 < kRowMaxTiles; ++k2)
      if (mk[k2] != -INFINITY) L += exp2f(mk[k2] - M) * lk[k2];
#pragma unroll
    for (int k2 = 0; k2 < kRowMaxTiles; ++k2)
      fac[k2][tid] = (ok && L > 0.0f && mk[k2] != -INFINITY) ? exp2f(mk[k2] - M) / L : 0.0f;
    if (t == 0 && a.lse)
      a.lse[(int64_t)qi * kHeads + tid] = L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
  if (!ok && tid == 0) report(a.status, CSA2_ERR_TIMEOUT);
  if (rflag) report(a.status, CSA2_ERR_RANGE);
  __syncthreads();
  // ---- this CTA's chunks c = t, t + n, ...: pull every tile's partial
  // (16-byte distributed loads, all issued before the sums), weight and sum
  // in tile order, 16-byte stores along the channels
  const uint32_t stg_addr = tc::smem_u32(stg);
  for (int c = t; c < 4; c += n) {
#pragma unroll
    for (int it = 0; it < kAllHeads * 32 / kThreads; it += 2) {
      float4 v[2][kRowMaxTiles];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = tid + kThreads * (it + u), h = e >> 5, ch4 = 4 * (e & 31);
        const uint32_t off = 4u * (uint32_t)((c * kAllHeads + h) * 128 + ch4);
#pragma unroll
        for (int k2 = 0; k2 < kRowMaxTiles; ++k2)
          if (k2 < n) v[u][k2] = tc::ld_dsmem_v4(tc::map_rank(stg_addr + off, k2));
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = tid + kThreads * (it + u), h = e >> 5, ch4 = 4 * (e & 31);
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int k2 = 0; k2 < kRowMaxTiles; ++k2)
          if (k2 < n) {
            const float f = fac[k2][h];
            acc.x = fmaf(f, v[u][k2].x, acc.x);
            acc.y = fmaf(f, v[u][k2].y, acc.y);
            acc.z = fmaf(f, v[u][k2].z, acc.z);
            acc.w = fmaf(f, v[u][k2].w, acc.w);
          }
        *reinterpret_cast<float4*>(a.out + ((int64_t)qi * kHeads + h) * kDim + c * 128 + ch4) = acc;
      }
    }
  }
  tc::cluster_sync();  // no CTA leaves while another still reads its shared memory
}

// ---------------------------------------------------------------------------
// Query-cluster variant for decode (top-k + window <= 640 rows): NC = 4 or 5
// CTAs per query token, each holding R = 160 or 128 of the query's rows for
// all 64 heads, the query's CTAs forming a cluster.  Chosen over the
// row-tile kernel so that every query's cluster fits in one wave of CTAs
// (NC = 4 when five CTAs per query would not).  Per CTA:
//  - before waiting for the selection (the kernel is launched while it
//    runs): the query rows (bf16 -> f16) and this CTA's window rows, which
//    no kernel of the step writes, are loaded into shared memory;
//  - after it: this CTA's selected entries are gathered (id, block table,
//    row) and decoded into the K-major row tile C;
//  - S^T = C . Q^T on the tensor cores (M = 128 rows; with R = 160 a second
//    block covers rows 32..159 and only its last 32 lanes are read), a
//    partial softmax per head over the CTA's rows, O^T = C^T . P^T;
//  - the merge: every CTA stages its unscaled partial output in its own
//    shared memory; after one cluster barrier the output's 16 pieces of 128
//    channels x 16 heads are shared out (piece i -> CTA i mod NC), and each
//    owner pulls its pieces of every tile with 16-byte distributed-shared-
//    memory loads and forms out = sum_t 2^(m_t - M) O_t / L in tile order,
//    M = max_t m_t, L = sum_t 2^(m_t - M) l_t (pushing the pieces with
//    remote stores was measured slower).
constexpr int kQcMaxRows = 160;
constexpr size_t kQcQBytes = (size_t)kAllHeads * kDim * 2;   // 65536; after S: P^T and scratch
constexpr size_t kQcSmem = kQcQBytes + (size_t)kQcMaxRows * kDim * 2;   // 229376

template <int kDtype, bool kSwaFp8, int NC>
__global__ void __launch_bounds__(kThreads, 1) attend_qc_kernel(AttArgs a) {
  constexpr bool kMainFp4 = (kDtype == CSA2_CACHE_FP4);
  uint32_t rflag = 0;  // an f16 operand out of range (CSA2_ERR_RANGE)
  constexpr int R = NC == 4 ? 160 : 128;  // rows of this CTA: 8-row groups t, t + NC, ...
  constexpr int NG = R / 8;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* qs = smem;                                    // Q [64 heads x 512] f16, K-major
  uint8_t* pt = smem;                                    // after S: P^T [64 heads x R rows] f16, K-major
  float* scr = reinterpret_cast<float*>(smem + kAllHeads * R * 2);  // after S: reduction scratch
  uint8_t* ctile = smem + kQcQBytes;                     // C [R rows x 512] f16, K-major
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ uint32_t vmask[NG / 4 + 1];                 // valid rows of the tile
  __shared__ float m_all[1][kAllHeads], l_all[1][kAllHeads];  // this CTA's (max, sum) per head
  __shared__ float fac_s[NC][kAllHeads];                       // factor of every tile per head

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127, p = tid >> 7, quad = warp & 3;
  const uint32_t lane_base = 32 * quad;
  const int t = (int)tc::cluster_rank();
  const int qi = blockIdx.y, b = qi / a.Tq;
  const int rl = lane & 7, uq = lane >> 3;
  // global slot of local row i
  auto slot_of = [&](int i) { return 8 * ((i >> 3) * NC + t) + (i & 7); };

  // loads of one 8-row group (this lane: row rl, 16-byte units 4k + uq) and
  // its decode into C
  struct Raw {
    uint4 v[16];
    uint32_t s[4];
  };
  auto load_group = [&](int32_t sidx, Raw& w) {
    if (sidx >= 0) {
      const int64_t page = sidx / kPage;
      const int sl = sidx % kPage;
      if (kMainFp4) {
        const uint4* g = reinterpret_cast<const uint4*>(a.mc.data + page * kMainFp4Data + sl * (kDim / 2));
        const uint16_t* gs = reinterpret_cast<const uint16_t*>(a.mc.scales + page * kMainFp4Scales + sl * (kDim / 16));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          w.v[k] = __ldg(g + 4 * k + uq);
          w.s[k] = __ldg(gs + 4 * k + uq);
        }
      } else {
        const uint4* g = reinterpret_cast<const uint4*>(a.mc.data + page * kMainBf16Data + sl * (kDim * 2));
#pragma unroll
        for (int k = 0; k < 16; ++k) w.v[k] = __ldg(g + 4 * k + uq);
      }
    } else if (sidx <= -2) {
      if (kSwaFp8) {
        const uint4* g =
            reinterpret_cast<const uint4*>(a.swa8 + ((int64_t)b * a.S + (-2 - (int64_t)sidx)) * kSwaFp8Row);
#pragma unroll
        for (int k = 0; k < 8; ++k) w.v[k] = __ldg(g + 4 * k + uq);
        w.v[8] = __ldg(g + 32);
      } else {
        const uint4* g = reinterpret_cast<const uint4*>(a.swa + ((int64_t)b * a.S + (-2 - (int64_t)sidx)) * kDim);
#pragma unroll
        for (int k = 0; k < 16; ++k) w.v[k] = __ldg(g + 4 * k + uq);
      }
    }
  };
  auto store_group = [&](int gi, int32_t sidx, const Raw& w, bool main_row) {
    const int rho = 8 * gi + rl;
    if (main_row && kMainFp4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int q = 4 * k + uq;
        const uint32_t s_lo = f16x2_scale(w.s[k] & 0xFFu), s_hi = f16x2_scale((w.s[k] >> 8) & 0xFFu);
        const uint32_t w4[4] = {w.v[k].x, w.v[k].y, w.v[k].z, w.v[k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 o = make_uint4(0, 0, 0, 0);
          if (sidx >= 0) {
            uint32_t h4[4];
            e2m1x8_to_f16x2(w4[i], h4);
            const uint32_t s2 = i < 2 ? s_lo : s_hi;
            o = make_uint4(hmul2(h4[0], s2), hmul2(h4[1], s2), hmul2(h4[2], s2), hmul2(h4[3], s2));
          }
          *reinterpret_cast<uint4*>(ctile + tc::kmajor_off(rho, 32 * q + 8 * i, kDim)) = o;
        }
      }
    } else if (!main_row && kSwaFp8) {
      const uint32_t sw[4] = {w.v[8].x, w.v[8].y, w.v[8].z, w.v[8].w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int u = 4 * k + uq, blk = u >> 1;
        uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (sidx != -1) mxfp8x16_to_f16x2(w.v[k], (sw[blk >> 2] >> (8 * (blk & 3))) & 0xFFu, o);
#pragma unroll
        for (int i = 0; i < 8; ++i) rflag |= f16x2_nonfinite(o[i]);
        *reinterpret_cast<uint4*>(ctile + tc::kmajor_off(rho, 16 * u, kDim)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(ctile + tc::kmajor_off(rho, 16 * u + 8, kDim)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const uint4 o = sidx == -1 ? make_uint4(0, 0, 0, 0)
                                   : make_uint4(to_f16x2(w.v[k].x, rflag), to_f16x2(w.v[k].y, rflag),
                                                to_f16x2(w.v[k].z, rflag), to_f16x2(w.v[k].w, rflag));
        *reinterpret_cast<uint4*>(ctile + tc::kmajor_off(rho, 8 * (4 * k + uq), kDim)) = o;
      }
    }
    if (uq == 0 && sidx != -1) atomicOr(&vmask[rho >> 5], 1u << (rho & 31));
  };
  // this warp's groups: w and (when R = 160) w + 16 for warps 0..3
  const int g0 = warp, g1 = warp + 16;
  const bool has1 = g1 < NG;
  const bool win0 = slot_of(8 * g0) >= a.tiles_main * 128;
  const bool win1 = has1 && slot_of(8 * g1) >= a.tiles_main * 128;

  // ---------------- before the selection has finished: Q, window rows
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  if (warp == kThreads / 32 - 1 && t == NC - 1 && qi % a.Tq == 0) {
    // once per sequence, its main-cache block table into L2 (hints only)
    int64_t np = (a.capacity + kPage - 1) / kPage;
    np = np < a.mc.max_pages ? np : a.mc.max_pages;
    const char* bt = reinterpret_cast<const char*>(a.mc.block_table + (int64_t)b * a.mc.max_pages);
    for (int64_t off = (int64_t)lane * 128; off < 4 * np; off += 32 * 128) tc::prefetch_l2(bt + off);
  }
  if (tid < NG / 4 + 1) vmask[tid] = 0u;
  {
    const int h = 8 * (warp & 7) + rl, u0 = 32 * (warp >> 3);
    const uint4* g = reinterpret_cast<const uint4*>(a.q + ((int64_t)qi * kHeads + h) * kDim);
    uint4 qv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) qv[k] = __ldg(g + u0 + 4 * k + uq);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      *reinterpret_cast<uint4*>(qs + tc::kmajor_off(h, 8 * (u0 + 4 * k + uq), kDim)) =
          make_uint4(to_f16x2(qv[k].x, rflag), to_f16x2(qv[k].y, rflag), to_f16x2(qv[k].z, rflag),
                     to_f16x2(qv[k].w, rflag));
  }
  __syncthreads();  // vmask cleared
  Raw w0, w1;
  int32_t s0 = -1, s1 = -1;
  if (win0) {
    s0 = slot_source(a, qi, b, slot_of(8 * g0 + rl));
    load_group(s0, w0);
    store_group(g0, s0, w0, false);
  }
  if (win1) {
    s1 = slot_source(a, qi, b, slot_of(8 * g1 + rl));
    load_group(s1, w1);
    store_group(g1, s1, w1, false);
  }

  const bool early = a.early != 0;
  if (!early) {
    griddep_wait();  // the selected ids are the previous kernel's output
    griddep_launch();
    if (warp == 0) {
      tc::tmem_alloc(&tmem_base, 512);
      tc::tmem_relinquish();
    }
  }
  // ---------------- the selected entries
  if (!win0) s0 = slot_source(a, qi, b, slot_of(8 * g0 + rl));
  if (has1 && !win1) s1 = slot_source(a, qi, b, slot_of(8 * g1 + rl));
  if (kMainFp4) {  // both groups' rows in flight at once (20 registers each)
    if (!win0) load_group(s0, w0);
    if (has1 && !win1) load_group(s1, w1);
    if (!win0) store_group(g0, s0, w0, true);
    if (has1 && !win1) store_group(g1, s1, w1, true);
  } else {         // 1 KB bf16 rows: one group at a time
    if (!win0) {
      load_group(s0, w0);
      store_group(g0, s0, w0, true);
    }
    if (has1 && !win1) {
      load_group(s1, w1);
      store_group(g1, s1, w1, true);
    }
  }
  if (early) {  // the rows are gathered: now the previous kernel's completion
    griddep_wait();
    griddep_launch();
    if (warp == 0) {
      tc::tmem_alloc(&tmem_base, 512);
      tc::tmem_relinquish();
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = tmem_base;
  bool ok = true;

  // ---- S^T = C . Q^T: block 0 rows 0..127 -> columns 0..63; with R = 160
  // block 1 rows 32..159 -> columns 64..127 (lanes 96..127 hold rows 128..159)
  constexpr uint32_t kIdescS = tc::idesc_f16(128, kAllHeads, false, false, false, false);
  constexpr uint32_t kIdescO = tc::idesc_f16(128, kAllHeads, false, false, true, false);
  if (tid == 0) {
#pragma unroll 1
    for (int blk = 0; blk < (R > 128 ? 2 : 1); ++blk) {
      const uint32_t cb = tc::smem_u32(ctile) + (blk ? 4 * kDim * 16 : 0);  // row group 4 = row 32
#pragma unroll 4
      for (int ks = 0; ks < kDim / 16; ++ks) {
        const uint64_t ad = tc::sdesc(cb + ks * 256, 128, kDim * 16);
        const uint64_t bd = tc::sdesc(tc::smem_u32(qs) + ks * 256, 128, kDim * 16);
        tc::mma_ss(tb + 64 * blk, ad, bd, kIdescS, ks > 0 ? 1u : 0u);
      }
    }
    tc::mma_commit(&bar);
  }
  ok = tc::mbar_wait(&bar, 0) && ok;
  tc::fence_after_sync();

  // ---- partial softmax over the CTA's rows: thread (r, p) holds row r of
  // block 0 and, in lane quarter 3 with R = 160, row 128 + (r - 96), for
  // heads 16p .. 16p + 15
  const float sc2 = a.scale * kLog2e;
  const bool extra = R > 128 && quad == 3;
  const bool valid0 = (vmask[r >> 5] >> (r & 31)) & 1u;
  const int r1 = 128 + (r - 96);
  const bool valid1 = extra && ((vmask[r1 >> 5] >> (r1 & 31)) & 1u);
  float v[16], v1[16];
  {
    uint32_t wv[16];
    tc::tmem_ld16(tc::taddr(tb, lane_base, 16 * p), wv);
    tc::tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = valid0 ? __uint_as_float(wv[j]) * sc2 : -INFINITY;
    if (R > 128) {
      tc::tmem_ld16(tc::taddr(tb, lane_base, 64 + 16 * p), wv);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) v1[j] = valid1 ? __uint_as_float(wv[j]) * sc2 : -INFINITY;
    }
  }
  float* red_m = scr;                    // [4][64]
  float* red_s = scr + 4 * kAllHeads;    // [4][64]
  float* mx = scr + 8 * kAllHeads;       // [64]
  tc::fence_before_sync();
  __syncthreads();  // every S read from tensor memory: Q's space becomes P^T and scratch
  tc::fence_after_sync();
  {
    float vm[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) vm[j] = R > 128 ? fmaxf(v[j], v1[j]) : v[j];
    const float wm = warp_reduce16<true>(vm);
    if ((lane & 1) == 0) red_m[quad * kAllHeads + 16 * p + (lane >> 1)] = wm;
  }
  __syncthreads();
  if (tid < kAllHeads)
    mx[tid] = fmaxf(fmaxf(red_m[tid], red_m[kAllHeads + tid]), fmaxf(red_m[2 * kAllHeads + tid], red_m[3 * kAllHeads + tid]));
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float mh = mx[16 * p + j];
    v[j] = (valid0 && mh != -INFINITY) ? exp2f(v[j] - mh) : 0.0f;
    *reinterpret_cast<__half*>(pt + tc::kmajor_off(16 * p + j, r, R)) = __float2half_rn(v[j]);
    if (R > 128) {
      v1[j] = (valid1 && mh != -INFINITY) ? exp2f(v1[j] - mh) : 0.0f;
      if (extra) *reinterpret_cast<__half*>(pt + tc::kmajor_off(16 * p + j, r1, R)) = __float2half_rn(v1[j]);
      v[j] += v1[j];
    }
  }
  {
    const float ws = warp_reduce16<false>(v);
    if ((lane & 1) == 0) red_s[quad * kAllHeads + 16 * p + (lane >> 1)] = ws;
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  float m_own = 0.0f, l_own = 0.0f;
  if (tid < kAllHeads) {
    m_own = mx[tid];
    l_own = (red_s[tid] + red_s[kAllHeads + tid]) + (red_s[2 * kAllHeads + tid] + red_s[3 * kAllHeads + tid]);
  }

  // ---- O^T[c] = C[:, chunk c]^T . P^T (C read MN-major)
  if (tid == 0) {
    if (ok) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t cbase = tc::smem_u32(ctile) + c * 16 * 128;
#pragma unroll 2
        for (int ks = 0; ks < R / 16; ++ks) {
          const uint64_t ad = tc::sdesc(cbase + ks * 2 * (kDim * 16), kDim * 16, 128);
          const uint64_t bd = tc::sdesc(tc::smem_u32(pt) + ks * 256, 128, (R / 8) * 128);
          tc::mma_ss(tb + 128 + 64 * c, ad, bd, kIdescO, ks > 0 ? 1u : 0u);
        }
      }
    }
    tc::mma_commit(&bar);
  }
  ok = tc::mbar_wait(&bar, 1) && ok;
  tc::fence_after_sync();
  // ---- this tile's unscaled partial output into its own shared memory (Q,
  // P^T and C are free once its MMAs are done), [chunk][head][channel]: a
  // warp's stores are 128 contiguous bytes
  float* stg = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t wv[16];
    tc::tmem_ld16(tc::taddr(tb, lane_base, 128 + 64 * c + 16 * p), wv);
    tc::tmem_wait_ld();
    float* dst = stg + (c * kAllHeads + 16 * p) * 128 + r;
#pragma unroll
    for (int j = 0; j < 16; ++j) dst[128 * j] = __uint_as_float(wv[j]);
  }
  if (tid < kAllHeads) {
    m_all[0][tid] = m_own;  // this CTA's (max, sum) per head, read by the cluster below
    l_all[0][tid] = l_own;
  }
  tc::fence_before_sync();
  tc::cluster_sync();  // every CTA's partial output and (max, sum) are in place
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tb, 512);
  if (!ok && tid == 0) report(a.status, CSA2_ERR_TIMEOUT);
  if (rflag) report(a.status, CSA2_ERR_RANGE);

  // ---- per-head factors of every tile: 2^(m_t - M) / L
  if (tid < kAllHeads) {
    float mk[NC], lk[NC];
#pragma unroll
    for (int k2 = 0; k2 < NC; ++k2) {
      mk[k2] = tc::ld_dsmem(tc::map_rank(tc::smem_u32(&m_all[0][tid]), k2));
      lk[k2] = tc::ld_dsmem(tc::map_rank(tc::smem_u32(&l_all[0][tid]), k2));
    }
    float M = -INFINITY;
#pragma unroll
    for (int k2 = 0; k2 < NC; ++k2) M = fmaxf(M, mk[k2]);
    float L = 0.0f;
#pragma unroll
    for (int k2 = 0; k2 < NC; ++k2)
      if (mk[k2] != -INFINITY) L += exp2f(mk[k2] - M) * lk[k2];
#pragma unroll
    for (int k2 = 0; k2 < NC; ++k2)
      fac_s[k2][tid] = (ok && L > 0.0f && mk[k2] != -INFINITY) ? exp2f(mk[k2] - M) / L : 0.0f;
    if (t == 0 && a.lse)
      a.lse[(int64_t)qi * kHeads + tid] = L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
  __syncthreads();
  // ---- the pieces this CTA owns (piece i = chunk i / 4, heads 16 (i % 4)..;
  // owner i mod NC): every tile's part pulled with 16-byte distributed loads,
  // all issued before the sums, weighted and summed in tile order
  const uint32_t stg_addr = tc::smem_u32(stg);
  for (int piece = t; piece < 16; piece += NC) {
    const int c = piece >> 2, h = 16 * (piece & 3) + (tid >> 5), ch4 = 4 * (tid & 31);
    const uint32_t off = 4u * (uint32_t)((c * kAllHeads + h) * 128 + ch4);
    float4 v[NC];
#pragma unroll
    for (int k2 = 0; k2 < NC; ++k2) v[k2] = tc::ld_dsmem_v4(tc::map_rank(stg_addr + off, k2));
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int k2 = 0; k2 < NC; ++k2) {
      const float f = fac_s[k2][h];
      acc.x = fmaf(f, v[k2].x, acc.x);
      acc.y = fmaf(f, v[k2].y, acc.y);
      acc.z = fmaf(f, v[k2].z, acc.z);
      acc.w = fmaf(f, v[k2].w, acc.w);
    }
    *reinterpret_cast<float4*>(a.out + ((int64_t)qi * kHeads + h) * kDim + 128 * c + ch4) = acc;
  }
  tc::cluster_sync();  // no CTA leaves while another still reads its shared memory
}

template <int kDtype, bool kSwaFp8>
cudaError_t launch_rows(const AttArgs& a, int Q, cudaStream_t stream) {
  const int n_tiles = a.tiles_main + a.tiles_win;
  auto kern = attend_rows_kernel<kDtype, kSwaFp8>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRowSmem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_tiles, Q);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kRowSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = n_tiles;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // whether this cluster shape can be scheduled at all, asked once per shape
  // (per instantiation: the function-local table is one per template)
  static int schedulable[kRowMaxTiles + 1] = {};  // 0 unknown, 1 yes, -1 no
  if (schedulable[n_tiles] == 0) {
    int clusters = 0;
    const bool yes = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters >= 1;
    (void)cudaGetLastError();
    schedulable[n_tiles] = yes ? 1 : -1;
  }
  if (schedulable[n_tiles] < 0) return cudaErrorNotSupported;
  return launch_k(kern, cfg.gridDim, cfg.blockDim, kRowSmem, stream, n_tiles, a);
}

// Clusters of the query-cluster kernel that fit on the device at once (0:
// not schedulable), asked once per instantiation.
template <int kDtype, bool kSwaFp8, int NC>
int qc_clusters() {
  static int cached = -1;
  if (cached < 0) {
    auto kern = attend_qc_kernel<kDtype, kSwaFp8, NC>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQcSmem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NC, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kQcSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = NC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) clusters = 0;
    (void)cudaGetLastError();
    cached = clusters;
  }
  return cached;
}

// Query-cluster attention for 4 or 5 row tiles: five CTAs of 128 rows per
// query when the batch fits one wave that way beside one more CTA per query
// (the selection that precedes a decode attention holds one SM per query
// while this kernel's CTAs start), else four of 160 rows when those fit one
// wave, else whichever shape takes fewer waves.  cudaErrorNotSupported when
// neither shape can run.
template <int kDtype, bool kSwaFp8>
cudaError_t launch_qc(const AttArgs& a, int Q, cudaStream_t stream) {
  const int c5 = qc_clusters<kDtype, kSwaFp8, 5>(), c4 = qc_clusters<kDtype, kSwaFp8, 4>();
  if (c5 < 1 && c4 < 1) return cudaErrorNotSupported;
  int64_t w5 = c5 > 0 ? (Q + c5 - 1) / c5 : INT64_MAX, w4 = c4 > 0 ? (Q + c4 - 1) / c4 : INT64_MAX;
  if (w5 == 1 && w4 == 1 && 6 * (int64_t)Q > num_sms()) w5 = 2;  // five beside the selection do not fit
  if (w4 < w5) {
    auto kern = attend_qc_kernel<kDtype, kSwaFp8, 4>;
    return launch_k(kern, dim3(4, Q), dim3(kThreads), kQcSmem, stream, 4, a);
  }
  auto kern = attend_qc_kernel<kDtype, kSwaFp8, 5>;
  return launch_k(kern, dim3(5, Q), dim3(kThreads), kQcSmem, stream, 5, a);
}

template <int kDtype>
cudaError_t launch_split(const AttArgs& a, int Q, cudaStream_t stream) {
  const int n_tiles = a.tiles_main + a.tiles_win;
  auto kern = attend_split_kernel<kDtype>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSplitSmem);
  if (n_tiles > 8) cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return launch_k(kern, dim3(n_tiles * (kHeads / kSplitHG), Q), dim3(kThreads), kSplitSmem, stream, n_tiles, a);
}

template <int kDtype, int HG>
size_t att_smem(int n_tiles, int stages = 2) {
  const int nslot = n_tiles * 128;
  return (size_t)stages * kStageBytes + 2 * kCBytes + std::max(HG * kDim * 2, nslot * HG * 2) + nslot * 4;
}

template <int kDtype, int HG, int kStages>
cudaError_t launch_hgs(const AttArgs& a, int Q, cudaStream_t stream) {
  const size_t smem = att_smem<kDtype, HG>(a.tiles_main + a.tiles_win, kStages);
  auto kern = attend_tc_kernel<kDtype, HG, kStages>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return launch_k(kern, dim3(kHeads / HG, Q), dim3(kThreads), smem, stream, 0, a);
}

constexpr size_t kSmemLimit = 225 * 1024;  // dynamic, leaving room for static shared memory

template <int kDtype, int HG>
cudaError_t launch_hg(const AttArgs& a, int Q, cudaStream_t stream) {
  // three staging units in flight when they fit, else two
  if (att_smem<kDtype, HG>(a.tiles_main + a.tiles_win, 3) <= kSmemLimit) return launch_hgs<kDtype, HG, 3>(a, Q, stream);
  return launch_hgs<kDtype, HG, 2>(a, Q, stream);
}

template <int kDtype>
cudaError_t launch_dtype(const AttArgs& a, int Q, int num_sms, cudaStream_t stream) {
  const int nt = a.tiles_main + a.tiles_win;
  // widest head group that fits TMEM (512 columns) and shared memory, preferring
  // more CTAs when there are few query tokens
  const bool few = (int64_t)Q * 2 < 2 * num_sms;
  const bool fit64 = nt * 64 <= 512 && att_smem<kDtype, 64>(nt) <= kSmemLimit;
  const bool fit32 = nt * 32 <= 512 && att_smem<kDtype, 32>(nt) <= kSmemLimit;
  if (!few && fit64) return launch_hg<kDtype, 64>(a, Q, stream);
  if ((int64_t)Q * 4 >= 2 * num_sms && fit32) return launch_hg<kDtype, 32>(a, Q, stream);
  if (nt * 16 <= 512 && att_smem<kDtype, 16>(nt) <= kSmemLimit) return launch_hg<kDtype, 16>(a, Q, stream);
  return cudaErrorInvalidConfiguration;
}

}  // namespace

bool attend_rows_path(int topk, int window) { return (topk + 127) / 128 + (window + 127) / 128 <= kRowMaxTiles; }

bool attend_tc_supported(int topk, int window) {
  const int nt = (topk + 127) / 128 + (window + 127) / 128;
  return nt * 16 <= 512 && att_smem<CSA2_CACHE_FP4, 16>(nt) <= kSmemLimit;
}

cudaError_t launch_attend(const csa2_cfg& cfg, int B, int Tq, const uint16_t* q, const csa2_cache& main_c,
                          const int32_t* n_entries, const int32_t* topk, const void* swa, int S,
                          const int32_t* swa_len, const int64_t* swa_pos0, const int64_t* q_pos,
                          float scale, float* out, float* lse, int32_t* status, bool ids_early,
                          cudaStream_t stream) {
  const int Q = B * Tq;
  if (Q == 0) return cudaSuccess;
  const bool fp8 = (cfg.formats & CSA2_FMT_SWA_FP8) != 0;
  AttArgs a{Tq, cfg.topk, cfg.window, S, (cfg.topk + 127) / 128, (cfg.window + 127) / 128, q, view_of(main_c),
            n_entries, (int64_t)main_c.max_pages * kPage, topk,
            fp8 ? nullptr : static_cast<const uint16_t*>(swa), fp8 ? static_cast<const uint8_t*>(swa) : nullptr,
            swa_len, swa_pos0, q_pos, scale, out, lse, status, ids_early ? 1 : 0};
  // up to six row tiles: one CTA per (query, tile) for every head, the
  // query's tiles in one cluster; more: split by head groups (bf16 window
  // rows only)
  const int n_tiles = a.tiles_main + a.tiles_win;
  if (n_tiles == 4 || n_tiles == 5) {
    cudaError_t e;
    if (cfg.cache_dtype == CSA2_CACHE_FP4)
      e = fp8 ? launch_qc<CSA2_CACHE_FP4, true>(a, Q, stream) : launch_qc<CSA2_CACHE_FP4, false>(a, Q, stream);
    else
      e = fp8 ? launch_qc<CSA2_CACHE_BF16, true>(a, Q, stream) : launch_qc<CSA2_CACHE_BF16, false>(a, Q, stream);
    if (e != cudaErrorNotSupported) return e;
  }
  if (n_tiles <= kRowMaxTiles) {
    cudaError_t e;
    if (cfg.cache_dtype == CSA2_CACHE_FP4)
      e = fp8 ? launch_rows<CSA2_CACHE_FP4, true>(a, Q, stream) : launch_rows<CSA2_CACHE_FP4, false>(a, Q, stream);
    else
      e = fp8 ? launch_rows<CSA2_CACHE_BF16, true>(a, Q, stream) : launch_rows<CSA2_CACHE_BF16, false>(a, Q, stream);
    if (e != cudaErrorNotSupported || fp8) return e;
  }
  if (fp8) return cudaErrorNotSupported;
  if ((int64_t)Q * 4 * n_tiles <= 8 * (int64_t)num_sms() && n_tiles <= 16) {
    cudaError_t e = cfg.cache_dtype == CSA2_CACHE_FP4 ? launch_split<CSA2_CACHE_FP4>(a, Q, stream)
                                                      : launch_split<CSA2_CACHE_BF16>(a, Q, stream);
    if (e == cudaSuccess) return e;
    (void)cudaGetLastError();  // cluster shape not schedulable here: use the per-query kernel
  }
  if (cfg.cache_dtype == CSA2_CACHE_FP4) return launch_dtype<CSA2_CACHE_FP4>(a, Q, num_sms(), stream);
  return launch_dtype<CSA2_CACHE_BF16>(a, Q, num_sms(), stream);
}

}  // namespace csa2
