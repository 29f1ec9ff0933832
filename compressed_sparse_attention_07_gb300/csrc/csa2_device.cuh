// Device-side helpers shared by the CSA2 kernels: status reporting, paged
// cache addressing, FP4 (E2M1 + E4M3 per 16 channels) decode / encode.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa2.h"

namespace csa2 {

constexpr int kDim = 512;       // latent channels
constexpr int kRope = 64;       // RoPE'd leading channels
constexpr int kHeads = 64;      // main query heads
constexpr int kIdxHeads = 32;   // indexer heads
constexpr int kIdxDim = 128;    // indexer channels
constexpr int kPage = CSA2_PAGE_ENTRIES;
constexpr int kHsiBlock = 8;

// Page strides in bytes.
constexpr int kMainFp4Data = kPage * kDim / 2;      // 16384
constexpr int kMainFp4Scales = kPage * kDim / 16;   // 2048
constexpr int kIdxFp4Data = kPage * kIdxDim / 2;    // 4096
constexpr int kIdxFp4Scales = kPage * kIdxDim / 16; // 512
constexpr int kIdxS32Scales = kPage * kIdxDim / 32; // 256 (68-byte indexer entries)
constexpr int kMainBf16Data = kPage * kDim * 2;     // 65536
constexpr int kIdxBf16Data = kPage * kIdxDim * 2;   // 16384
constexpr int kSwaFp8Row = kDim + kDim / 32;        // 528: MXFP8 window row (elements + E8M0 scales)

struct CacheView {
  uint8_t* data;
  uint8_t* scales;
  const int32_t* block_table;
  int32_t max_pages;
  int32_t num_pages;
};

__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// Page holding entry j of sequence b, or -1 (status set) when the block
// table points outside the page pool.
__device__ __forceinline__ int64_t page_of(const CacheView& c, int b, int64_t j, int32_t* status) {
  int64_t slot = j / kPage;
  if (slot < 0 || slot >= c.max_pages) {
    report(status, CSA2_ERR_BAD_INDEX);
    return -1;
  }
  int32_t p = __ldg(c.block_table + (int64_t)b * c.max_pages + slot);
  if (p < 0 || p >= c.num_pages) {
    report(status, CSA2_ERR_BAD_PAGE);
    return -1;
  }
  return p;
}

// Entries visible to a query at position t: r*j + r - 1 <= t and j < n.
__device__ __forceinline__ int64_t visible_entries(int64_t t, int r, int64_t n) {
  if (t < r - 1) return 0;
  int64_t v = (t - (r - 1)) / r + 1;
  return v < n ? v : n;
}

// E2M1 magnitude index m = (e1 e0 mant): 0, .5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ float e2m1_to_float(uint32_t code) {
  uint32_t e = (code >> 1) & 3u, m = code & 1u;
  float mag = (e == 0) ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * (float)(1u << (e - 1));
  return (code & 8u) ? -mag : mag;
}

// E4M3 (no infinities; the all-ones pattern is NaN, never produced here).
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  uint32_t e = (byte >> 3) & 15u, m = byte & 7u;
  float mag = (e == 0) ? (float)m * 0.001953125f                       // m * 2^-9
                       : __int_as_float((int)((e + 120u) << 23 | (m << 20)));  // (1+m/8) 2^(e-7)
  return (byte & 0x80u) ? -mag : mag;
}

// Non-negative E4M3 value of code c in 0..126.
__device__ __forceinline__ float e4m3_pos(int c) { return e4m3_to_float((uint32_t)c); }

// Scale code for a 16-channel group: the E4M3 code nearest to amax / 6, ties
// to the even code, saturating at 448 (code 126).  Decided by comparing amax
// with 6 * midpoint, which is exact in fp32, so amax / 6 is never rounded.
__device__ __forceinline__ int e4m3_scale_code(float amax) {
  // count thresholds t_c = 6 * (v_c + v_{c+1}) / 2 below amax (ties: odd c counts)
  int lo = 0, hi = 126;  // answer in [lo, hi]
  while (lo < hi) {
    int c = (lo + hi) >> 1;  // is the answer > c ?  <=> amax passes threshold c
    float t = 3.0f * (e4m3_pos(c) + e4m3_pos(c + 1));
    bool up = (amax > t) || (amax == t && (c & 1));
    if (up) lo = c + 1; else hi = c;
  }
  return lo;
}

// E2M1 code of x / s (s > 0): round to nearest, ties to the even magnitude
// index, saturating at 6; decided by |x| against s * midpoint (exact).
__device__ __forceinline__ uint32_t e2m1_code(float x, float s) {
  if (!(s > 0.0f)) return 0u;
  float a = fabsf(x);
  const float mid[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
  uint32_t m = 0;
#pragma unroll
  for (int k = 0; k < 7; ++k) {
    float t = s * mid[k];
    m += (a > t) || (a == t && (k & 1));
  }
  if (m == 0) return 0u;
  return (x < 0.0f) ? (m | 8u) : m;
}

// Score bit pattern marking a non-candidate position (a NaN never produced
// by the scoring) and the monotone unsigned key of a score: larger score ->
// larger key; the non-candidate pattern maps to key 0.
// Programmatic dependent launch: wait until the previous kernel on the
// stream has completed and its writes are visible; let the next kernel's
// grid be scheduled (it waits for this one in turn).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

constexpr uint32_t kScoreInvalid = 0xFFFFFFFFu;
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  if (u == kScoreInvalid) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

}  // namespace csa2
