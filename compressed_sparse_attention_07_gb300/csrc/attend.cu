// a2 -- decode entries of a paged cache (main KV or indexer K, FP4 or bf16)
// to fp32, exactly (E2M1 x E4M3 per 16 channels; hn.213312.xyz sec. 2.4.4).
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
      if (kDtype == CSA2_CACHE_FP4) {
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
  if (cache_dtype == CSA2_CACHE_FP4)
    return launch_k(gather_dequant_kernel<CSA2_CACHE_FP4>, grid, dim3(128), 0, stream, 0, view_of(c), c.channels, n,
                    ids, out, status);
  return launch_k(gather_dequant_kernel<CSA2_CACHE_BF16>, grid, dim3(128), 0, stream, 0, view_of(c), c.channels, n,
                  ids, out, status);
}

}  // namespace csa2
