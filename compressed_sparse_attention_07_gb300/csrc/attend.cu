// a7 -- CSA2 sparse attention: per query token, one softmax per head over
// the selected main-KV entries together with the layer's sliding-window rows;
// the same 512-channel latent is key and value.
// (DeepSeek-V4.1 Flash, hn.213312.xyz sec. 2.2.2 and 3.3.1; 36kr "CSA2".)
#include "internal.h"

namespace csa2 {
namespace {

constexpr int kAttThreads = 256;
constexpr int kHeadsPerCta = 8;
constexpr int kTileRows = 32;
constexpr int kTileStride = kDim + 1;  // conflict-free column walks

struct AttendArgs {
  int Tq, k, W, S;
  const uint16_t* q;
  CacheView mc;
  const int32_t* n_entries;
  int64_t capacity;
  const int32_t* topk;
  const uint16_t* swa;
  const int32_t* swa_len;
  const int64_t* swa_pos0;
  const int64_t* q_pos;
  float scale;
  float* out;
  float* lse;
  int32_t* status;
};

// Row source of slot i: >= 0 main entry id, <= -2 window row (-2 - row), -1 none.
__device__ __forceinline__ int64_t slot_source(const AttendArgs& a, int qi, int b, int i) {
  if (i < a.k) {
    int32_t id = __ldg(a.topk + (int64_t)qi * a.k + i);
    if (id < 0) return -1;
    if (id >= __ldg(a.n_entries + b) || id >= a.capacity) {
      report(a.status, CSA2_ERR_BAD_INDEX);
      return -1;
    }
    return id;
  }
  const int64_t t = __ldg(a.q_pos + qi);
  const int64_t pos = t - a.W + 1 + (i - a.k);
  const int64_t p0 = __ldg(a.swa_pos0 + b);
  int64_t len = __ldg(a.swa_len + b);
  len = len < a.S ? len : a.S;
  if (pos < 0 || pos < p0 || pos >= p0 + len) return -1;
  return -2 - (pos - p0);
}

// Decode rows [s0, s0 + 32) of the slot list into tile (fp32); 8 threads per row.
template <int kDtype>
__device__ void load_tile(const AttendArgs& a, int qi, int b, int s0, int nslots, const int64_t* src, float* tile) {
  const int r = threadIdx.x >> 3, part = threadIdx.x & 7;  // part covers channels [64*part, 64*part+64)
  const int i = s0 + r;
  float* row = tile + r * kTileStride + 64 * part;
  const int64_t sidx = (i < nslots) ? src[i] : -1;
  if (sidx == -1) {
    for (int c = 0; c < 64; ++c) row[c] = 0.0f;
    return;
  }
  if (sidx <= -2) {  // window row, bf16
    const uint16_t* wr = a.swa + ((int64_t)b * a.S + (-2 - sidx)) * kDim + 64 * part;
    const uint4* w4 = reinterpret_cast<const uint4*>(wr);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      uint4 x = __ldg(w4 + v);
      uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        row[8 * v + 2 * q] = __uint_as_float(w[q] << 16);
        row[8 * v + 2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
      }
    }
    return;
  }
  const int64_t page = page_of(a.mc, b, sidx, a.status);
  if (page < 0) {
    for (int c = 0; c < 64; ++c) row[c] = 0.0f;
    return;
  }
  const int slot = (int)(sidx % kPage);
  if (kDtype == CSA2_CACHE_FP4) {
    const uint4* c4 = reinterpret_cast<const uint4*>(a.mc.data + page * kMainFp4Data + slot * (kDim / 2) + 32 * part);
    uint32_t sc = __ldg(reinterpret_cast<const uint32_t*>(a.mc.scales + page * kMainFp4Scales + slot * (kDim / 16) + 4 * part));
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      uint4 x = __ldg(c4 + v);
      uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int c = 32 * v + 8 * q + n;  // channel within this part
          float s = e4m3_to_float((sc >> (8 * (c >> 4))) & 0xFFu);
          row[c] = e2m1_to_float((w[q] >> (4 * n)) & 15u) * s;
        }
      }
    }
  } else {
    const uint4* w4 = reinterpret_cast<const uint4*>(a.mc.data + page * kMainBf16Data + slot * (kDim * 2) + 128 * part);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      uint4 x = __ldg(w4 + v);
      uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        row[8 * v + 2 * q] = __uint_as_float(w[q] << 16);
        row[8 * v + 2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
      }
    }
  }
}

template <int kDtype>
__global__ void __launch_bounds__(kAttThreads) attend_kernel(AttendArgs a) {
  extern __shared__ __align__(16) float smem[];
  const int nslots = a.k + a.W;
  float* qs = smem;                                   // [8][512]
  float* tile = qs + kHeadsPerCta * kDim;             // [32][513]
  float* logits = tile + kTileRows * kTileStride;     // [8][nslots]
  int64_t* src = reinterpret_cast<int64_t*>(logits + kHeadsPerCta * nslots);  // [nslots], 8-byte aligned
  __shared__ float inv_sum[kHeadsPerCta];

  const int hg = blockIdx.x, qi = blockIdx.y, b = qi / a.Tq;
  const int tid = threadIdx.x;
  for (int i = tid; i < kHeadsPerCta * kDim; i += kAttThreads)
    qs[i] = bf16_bits_to_float(__ldg(a.q + ((int64_t)qi * kHeads + hg * kHeadsPerCta) * kDim + i));
  for (int i = tid; i < nslots; i += kAttThreads) src[i] = slot_source(a, qi, b, i);
  __syncthreads();

  // logits: thread (h, row) per tile
  const int h = tid >> 5, rr = tid & 31;
  for (int s0 = 0; s0 < nslots; s0 += kTileRows) {
    load_tile<kDtype>(a, qi, b, s0, nslots, src, tile);
    __syncthreads();
    const float* row = tile + rr * kTileStride;
    const float* qh = qs + h * kDim;
    float d = 0.0f;
#pragma unroll 8
    for (int c = 0; c < kDim; ++c) d = fmaf(qh[c], row[c], d);
    const int i = s0 + rr;
    if (i < nslots) logits[h * nslots + i] = (src[i] == -1) ? -INFINITY : d * a.scale;
    __syncthreads();
  }

  // softmax per head: warp h
  {
    const int lane = tid & 31;
    float* lh = logits + h * nslots;
    float mx = -INFINITY;
    for (int i = lane; i < nslots; i += 32) mx = fmaxf(mx, lh[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.0f;
    for (int i = lane; i < nslots; i += 32) {
      float p = (mx == -INFINITY) ? 0.0f : __expf(lh[i] - mx);
      lh[i] = p;
      sum += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      inv_sum[h] = sum > 0.0f ? 1.0f / sum : 0.0f;
      if (a.lse) a.lse[(int64_t)qi * kHeads + hg * kHeadsPerCta + h] = sum > 0.0f ? mx + logf(sum) : -INFINITY;
    }
  }
  __syncthreads();

  // out = sum_e p_e c_e: thread t owns channels t and t + 256 for the 8 heads
  float acc[kHeadsPerCta][2];
#pragma unroll
  for (int hh = 0; hh < kHeadsPerCta; ++hh) acc[hh][0] = acc[hh][1] = 0.0f;
  for (int s0 = 0; s0 < nslots; s0 += kTileRows) {
    load_tile<kDtype>(a, qi, b, s0, nslots, src, tile);
    __syncthreads();
    const int nr = min(kTileRows, nslots - s0);
    for (int r2 = 0; r2 < nr; ++r2) {
      const float c0 = tile[r2 * kTileStride + tid], c1 = tile[r2 * kTileStride + tid + 256];
#pragma unroll
      for (int hh = 0; hh < kHeadsPerCta; ++hh) {
        const float p = logits[hh * nslots + s0 + r2];
        acc[hh][0] = fmaf(p, c0, acc[hh][0]);
        acc[hh][1] = fmaf(p, c1, acc[hh][1]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int hh = 0; hh < kHeadsPerCta; ++hh) {
    float* o = a.out + ((int64_t)qi * kHeads + hg * kHeadsPerCta + hh) * kDim;
    o[tid] = acc[hh][0] * inv_sum[hh];
    o[tid + 256] = acc[hh][1] * inv_sum[hh];
  }
}

template <int kDtype>
__global__ void __launch_bounds__(128) gather_dequant_kernel(CacheView c, int channels, int n, const int32_t* ids,
                                                             float* out, int32_t* status) {
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

cudaError_t launch_attend(const csa2_cfg& cfg, int B, int Tq, const uint16_t* q, const csa2_cache& main_c,
                          const int32_t* n_entries, const int32_t* topk, const uint16_t* swa, int S,
                          const int32_t* swa_len, const int64_t* swa_pos0, const int64_t* q_pos,
                          float scale, float* out, float* lse, int32_t* status, cudaStream_t stream) {
  const int Q = B * Tq;
  if (Q == 0) return cudaSuccess;
  AttendArgs a{Tq, cfg.topk, cfg.window, S, q, view_of(main_c), n_entries, (int64_t)main_c.max_pages * kPage,
               topk, swa, swa_len, swa_pos0, q_pos, scale, out, lse, status};
  const int nslots = cfg.topk + cfg.window;
  size_t smem = sizeof(float) * ((size_t)kHeadsPerCta * kDim + (size_t)kTileRows * kTileStride +
                                 (size_t)kHeadsPerCta * nslots) +
                sizeof(int64_t) * nslots;
  dim3 grid(kHeads / kHeadsPerCta, Q);
  if (cfg.cache_dtype == CSA2_CACHE_FP4) {
    cudaFuncSetAttribute(attend_kernel<CSA2_CACHE_FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attend_kernel<CSA2_CACHE_FP4><<<grid, kAttThreads, smem, stream>>>(a);
  } else {
    cudaFuncSetAttribute(attend_kernel<CSA2_CACHE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attend_kernel<CSA2_CACHE_BF16><<<grid, kAttThreads, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_gather_dequant(const csa2_cache& c, int cache_dtype, int B, int n, const int32_t* ids,
                                  float* out, int32_t* status, cudaStream_t stream) {
  if (B == 0 || n == 0) return cudaSuccess;
  dim3 grid(n, B);
  if (cache_dtype == CSA2_CACHE_FP4)
    gather_dequant_kernel<CSA2_CACHE_FP4><<<grid, 128, 0, stream>>>(view_of(c), c.channels, n, ids, out, status);
  else
    gather_dequant_kernel<CSA2_CACHE_BF16><<<grid, 128, 0, stream>>>(view_of(c), c.channels, n, ids, out, status);
  return cudaGetLastError();
}

}  // namespace csa2
