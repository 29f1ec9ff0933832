// a1 -- CSA2 compressor: merge r tokens per entry with per-channel weights,
// RoPE at the entry's last covered position, encode into the paged main
// cache, project the stored entry to indexer K and encode that too (FP4
// with one E4M3 scale per 16 channels, or per 32 for the 68-byte indexer
// entry of hn.213312.xyz sec. 3.1).
// (DeepSeek-V4.1 Flash, hn.213312.xyz sec. 2.3.1 and sec. 2.4.4; 36kr "CSA2",
// "FP4 and Bounded Replay".)  Four CTAs per new entry: each merges, rotates
// and encodes the entry (the first one stores it) and projects it onto 32 of
// the 128 indexer channels, so each reads a quarter of W_idx.  The step moves
// a few KB per entry: latency-bound and kept simple.
#include <cmath>

#include "internal.h"

namespace csa2 {
namespace {

// RoPE inverse frequencies theta^(-2i/64), formed on the host in fp64.
struct RopeFreqs {
  double f[kRope / 2];
};

template <int kDtype, bool kIdxS32>
__global__ void __launch_bounds__(256) compress_kernel(int T, int r, RopeFreqs rf, const uint16_t* __restrict__ x,
                                                       const int64_t* __restrict__ pos0,
                                                       const float* __restrict__ merge_w,
                                                       const uint16_t* __restrict__ w_idx, CacheView mc,
                                                       CacheView ic, int32_t* n_entries, int32_t* status) {
  __shared__ float e_s[kDim];          // the stored (decoded) entry
  __shared__ float kpart[32][32];  // projection partial sums: 32 row slices x this CTA's 32 columns
  const int m = blockIdx.x, b = blockIdx.y, sx = blockIdx.z, t = threadIdx.x;
  griddep_wait();  // every input may be the previous kernel's output
  griddep_launch();
  // the W_idx rows this thread needs (16 independent 8-byte loads of this
  // CTA's 32 columns), issued first: their latency overlaps the merge
  const int kg = t & 7, rs = t >> 3;
  uint2 wv[16];
  {
    const uint2* w2 = reinterpret_cast<const uint2*>(w_idx) + 8 * sx + kg;  // row c at + c * 32
#pragma unroll
    for (int i = 0; i < 16; ++i) wv[i] = __ldg(w2 + (rs * 16 + i) * (kIdxDim / 4));
  }
  const int64_t j = pos0[b] / r + m;
  // both block-table lookups early, off the critical path of the projection
  const int64_t page = page_of(mc, b, j, status);
  const int64_t ipage = page_of(ic, b, j, status);

  // merge: thread t owns channels 2t and 2t+1
  float v0 = 0.0f, v1 = 0.0f;
  for (int i = 0; i < r; ++i) {
    const uint16_t* xr = x + ((int64_t)b * T + (int64_t)m * r + i) * kDim;
    uint32_t pair = __ldg(reinterpret_cast<const uint32_t*>(xr) + t);
    float x0 = __uint_as_float(pair << 16), x1 = __uint_as_float(pair & 0xFFFF0000u);
    float w0 = __ldg(merge_w + i * kDim + 2 * t), w1 = __ldg(merge_w + i * kDim + 2 * t + 1);
    v0 = (i == 0) ? w0 * x0 : fmaf(w0, x0, v0);
    v1 = (i == 0) ? w1 * x1 : fmaf(w1, x1, v1);
  }
  // RoPE on the pair (2t, 2t+1) for the first 64 channels: the angle p * f is
  // formed and reduced modulo 2 pi in fp64 (Cody-Waite, 2 pi split so that
  // k * hi is exact), then rotated with fp32 sincos of the reduced angle.
  if (t < kRope / 2) {
    const double ang = (double)(r * j + r - 1) * rf.f[t];
    const double kk = rint(ang * 0.15915494309189535);      // 1 / (2 pi)
    double red = fma(-kk, 6.28318530717958623, ang);          // 2 pi, high part
    red = fma(-kk, 2.4492935982947064e-16, red);              // 2 pi, low part
    float s, c;
    sincosf((float)red, &s, &c);
    float a = v0, bb = v1;
    v0 = fmaf(a, c, -(bb * s));
    v1 = fmaf(a, s, bb * c);
  }

  const int slot = (int)(j % kPage);
  if (kDtype == CSA2_CACHE_FP4) {
    float amax = fmaxf(fabsf(v0), fabsf(v1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    int sc = e4m3_scale_code(amax);
    float s = e4m3_pos(sc);
    uint32_t c0 = e2m1_code(v0, s), c1 = e2m1_code(v1, s);
    if (page >= 0 && sx == 0) {
      mc.data[page * kMainFp4Data + slot * (kDim / 2) + t] = (uint8_t)(c0 | (c1 << 4));
      if ((t & 7) == 0) mc.scales[page * kMainFp4Scales + slot * (kDim / 16) + (t >> 3)] = (uint8_t)sc;
    }
    e_s[2 * t] = e2m1_to_float(c0) * s;
    e_s[2 * t + 1] = e2m1_to_float(c1) * s;
  } else {
    __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
    uint32_t packed = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
    if (page >= 0 && sx == 0)
      reinterpret_cast<uint32_t*>(mc.data + page * kMainBf16Data + slot * (kDim * 2))[t] = packed;
    e_s[2 * t] = __bfloat162float(h0);
    e_s[2 * t + 1] = __bfloat162float(h1);
  }
  __syncthreads();

  // indexer K = stored entry . W_idx: thread t owns columns 4*(t%32)..+3 over
  // the 64-row slice t/32 (each warp reads whole 256-byte rows); the 8 slice
  // sums are added in slice order.
  {
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float e = e_s[rs * 16 + i];
      acc[0] = fmaf(e, __uint_as_float(wv[i].x << 16), acc[0]);
      acc[1] = fmaf(e, __uint_as_float(wv[i].x & 0xFFFF0000u), acc[1]);
      acc[2] = fmaf(e, __uint_as_float(wv[i].y << 16), acc[2]);
      acc[3] = fmaf(e, __uint_as_float(wv[i].y & 0xFFFF0000u), acc[3]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) kpart[rs][4 * kg + q] = acc[q];
  }
  __syncthreads();
  if (t < 32) {
    float kv = kpart[0][t];
#pragma unroll
    for (int q = 1; q < 32; ++q) kv += kpart[q][t];
    const int col = 32 * sx + t;  // indexer channel
    if (kDtype == CSA2_CACHE_FP4) {
      float amax = fabsf(kv);
#pragma unroll
      for (int o = 1; o < (kIdxS32 ? 32 : 16); o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      int sc = e4m3_scale_code(amax);
      uint32_t code = e2m1_code(kv, e4m3_pos(sc));
      uint32_t hi = __shfl_xor_sync(0xffffffffu, code, 1);
      if (ipage >= 0 && (t & 1) == 0) {
        int bi = col >> 1;  // byte index 0..63 -> 16-byte chunk bi/16
        ic.data[ipage * kIdxFp4Data + ((bi >> 4) * kPage + slot) * 16 + (bi & 15)] = (uint8_t)(code | (hi << 4));
      }
      if (kIdxS32) {
        if (ipage >= 0 && (col & 31) == 0) ic.scales[ipage * kIdxS32Scales + slot * (kIdxDim / 32) + (col >> 5)] = (uint8_t)sc;
      } else if (ipage >= 0 && (col & 15) == 0) {
        ic.scales[ipage * kIdxFp4Scales + slot * (kIdxDim / 16) + (col >> 4)] = (uint8_t)sc;
      }
    } else {
      uint16_t h = __bfloat16_as_ushort(__float2bfloat16_rn(kv));
      if (ipage >= 0) {
        int byte = 2 * col;  // chunk byte/16
        *reinterpret_cast<uint16_t*>(ic.data + ipage * kIdxBf16Data + ((byte >> 4) * kPage + slot) * 16 +
                                     (byte & 15)) = h;
      }
    }
  }
  if (m == gridDim.x - 1 && t == 0 && sx == 0) n_entries[b] = (int32_t)(j + 1);
}

}  // namespace

cudaError_t launch_compress(const csa2_cfg& cfg, int B, int T, const uint16_t* x, const int64_t* pos0,
                            const float* merge_w, const uint16_t* w_idx, const csa2_cache& main_c,
                            const csa2_cache& idx_c, int32_t* n_entries, int32_t* status,
                            cudaStream_t stream) {
  const int M = T / cfg.ratio;
  if (M == 0 || B == 0) return cudaSuccess;
  dim3 grid(M, B, 4);  // 4 CTAs per entry: 32 indexer channels each
  RopeFreqs rf;
  for (int i = 0; i < kRope / 2; ++i) rf.f[i] = std::pow(cfg.rope_theta, -2.0 * i / kRope);
  if (idx_dtype(cfg) == CSA2_CACHE_FP4_S32)
    return launch_k(compress_kernel<CSA2_CACHE_FP4, true>, grid, dim3(256), 0, stream, 0, T, cfg.ratio, rf, x, pos0,
                    merge_w, w_idx, view_of(main_c), view_of(idx_c), n_entries, status);
  if (cfg.cache_dtype == CSA2_CACHE_FP4)
    return launch_k(compress_kernel<CSA2_CACHE_FP4, false>, grid, dim3(256), 0, stream, 0, T, cfg.ratio, rf, x, pos0,
                    merge_w, w_idx, view_of(main_c), view_of(idx_c), n_entries, status);
  return launch_k(compress_kernel<CSA2_CACHE_BF16, false>, grid, dim3(256), 0, stream, 0, T, cfg.ratio, rf, x, pos0, merge_w,
                  w_idx, view_of(main_c), view_of(idx_c), n_entries, status);
}

}  // namespace csa2
