// a2 -- decode entries of a paged cache (main KV or indexer K, FP4 or bf16)
// to fp32, exactly (E2M1 x E4M3 per 16 channels, hn.213312.xyz sec. 2.4.4;
// per 32 channels for the 68-byte indexer entry, sec. 3.1).
#include "internal.h"

namespace csa2 {
namespace {

template <int kDtype>
__global__ void __launch_bounds__(128) gather_dequant_kernel(CacheView c, int channels, int n, const int32_t* ids,
                                                             float* out, int32_t* status) {
  griddep_wait();
  griddep_launch();
  const int i = blockIdx.x, b = blockIdx.y;
  const int32_t id = ids[(int64_t)b * n + i];
  float* o = out + ((int64_t)b * n + i) * channels;
  const int64_t page = id >= 0 ? page_of(c, b, id, status) : -1;
  const int slot = id >= 0 ? id % kPage : 0;
  for (int ch = threadIdx.x; ch < channels; ch += blockDim.x) {
    float v = 0.0f;
    if (page >= 0) {
      if (kDtype == CSA2_CACHE_FP4_S32) {
        const int byte = ch >> 1;
        const uint8_t code_b = c.data[page * kIdxFp4Data + ((byte >> 4) * kPage + slot) * 16 + (byte & 15)];
        const uint8_t sc = c.scales[page * kIdxS32Scales + slot * (kIdxDim / 32) + (ch >> 5)];
        v = e2m1_to_float((ch & 1) ? (code_b >> 4) : (code_b & 15u)) * e4m3_to_float(sc);
      } else if (kDtype == CSA2_CACHE_FP4) {
        const int byte = ch >> 1;
        uint8_t code_b, sc;
        if (channels == kDim) {
          code_b = c.data[page * kMainFp4Data + slot * (kDim / 2) + byte];
          sc = c.scales[page * kMainFp4Scales + slot * (kDim / 16) + (ch >> 4)];
        } else {
          code_b = c.data[page * kIdxFp4Data + ((byte >> 4) * kPage + slot) * 16 + (byte & 15)];
          sc = c.scales[page * kIdxFp4Scales + slot * (kIdxDim / 16) + (ch >> 4)];
        }
        v = e2m1_to_float((ch & 1) ? (code_b >> 4) : (code_b & 15u)) * e4m3_to_float(sc);
      } else {
        const uint16_t* p = (channels == kDim)
                                ? reinterpret_cast<const uint16_t*>(c.data + page * kMainBf16Data + slot * (kDim * 2)) + ch
                                : reinterpret_cast<const uint16_t*>(c.data + page * kIdxBf16Data +
                                                                    (((2 * ch) >> 4) * kPage + slot) * 16 + ((2 * ch) & 15));
        v = bf16_bits_to_float(*p);
      }
    }
    o[ch] = v;
  }
}

}  // namespace

cudaError_t launch_gather_dequant(const csa2_cache& c, int cache_dtype, int B, int n, const int32_t* ids,
                                  float* out, int32_t* status, cudaStream_t stream) {
  if (B == 0 || n == 0) return cudaSuccess;
  dim3 grid(n, B);
  if (cache_dtype == CSA2_CACHE_FP4_S32)
    return launch_k(gather_dequant_kernel<CSA2_CACHE_FP4_S32>, grid, dim3(128), 0, stream, 0, view_of(c), c.channels,
                    n, ids, out, status);
  if (cache_dtype == CSA2_CACHE_FP4)
    return launch_k(gather_dequant_kernel<CSA2_CACHE_FP4>, grid, dim3(128), 0, stream, 0, view_of(c), c.channels, n,
                    ids, out, status);
  return launch_k(gather_dequant_kernel<CSA2_CACHE_BF16>, grid, dim3(128), 0, stream, 0, view_of(c), c.channels, n,
                  ids, out, status);
}

// FP8 window rows (hn.213312.xyz sec. 2.4.4: the SWA KV stays FP8) in the
// OCP MXFP8 layout: one 528-byte row per token, E4M3 elements and one E8M0
// scale per 32 channels.  One CTA of 128 threads per row; thread t encodes
// channels 4t..4t+3, eight threads per 32-channel block.
namespace {

__global__ void __launch_bounds__(128) swa_encode_kernel(int T, int S, const uint16_t* __restrict__ x,
                                                         const int64_t* __restrict__ row0, uint8_t* rows,
                                                         int32_t* status) {
  // no early launch of the next kernel: the attention reads window rows
  // before it waits for its predecessor, so a kernel that writes them lets
  // its successor start only when it has completed
  griddep_wait();
  const int i = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const int64_t r0 = __ldg(row0 + b);
  if (r0 < 0 || r0 + T > S) {
    if (i == 0 && t == 0) report(status, CSA2_ERR_BAD_INDEX);
    return;
  }
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(x + ((int64_t)b * T + i) * kDim) + t);
  float v[4] = {__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                __uint_as_float(w.y & 0xFFFF0000u)};
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  // scale exponent floor(log2 amax) - 8 (E4M3's top binade is 2^8), read off
  // the bits: normal values by their exponent field, subnormal ones by the
  // position of the leading mantissa bit
  int sb = 0;
  const uint32_t ab = __float_as_uint(amax);
  if (ab != 0u) {
    const int e = (int)(ab >> 23);
    const int fl = e != 0 ? e - 127 : (31 - __clz((int)(ab & 0x7FFFFFu))) - 149;
    sb = min(max(fl - 8 + 127, 0), 254);
  }
  const float inv = __uint_as_float((uint32_t)(254 - sb) << 23);  // 2^(127 - sb), exact
  uint32_t packed = 0;
#pragma unroll
  for (int k = 0; k < 4; k += 2) {
    uint16_t p;
    // the upper source lands in the upper byte: channel 4t+k in the low byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(p) : "f"(v[k + 1] * inv), "f"(v[k] * inv));
    uint32_t q = p;
    if ((q & 0xFFu) == 0x80u) q &= 0xFF00u;  // a value that rounds to zero gets +0
    if ((q & 0xFF00u) == 0x8000u) q &= 0x00FFu;
    packed |= q << (8 * k);
  }
  uint8_t* row = rows + ((int64_t)b * S + r0 + i) * kSwaFp8Row;
  reinterpret_cast<uint32_t*>(row)[t] = packed;
  if ((t & 7) == 0) row[kDim + (t >> 3)] = (uint8_t)sb;
}

}  // namespace

cudaError_t launch_swa_encode(int B, int T, const uint16_t* x, const int64_t* row0, void* rows, int S,
                              int32_t* status, cudaStream_t stream) {
  if (B == 0 || T == 0) return cudaSuccess;
  return launch_k(swa_encode_kernel, dim3(T, B), dim3(128), 0, stream, 0, T, S, x, row0,
                  static_cast<uint8_t*>(rows), status);
}

}  // namespace csa2
