// Device helpers shared by the indexer scoring kernels: FP4 (E2M1) and E4M3
// decoding to f16 pairs, and the construction of the query tile (Q_idx of one
// query, 32 heads x 128 channels, f16 or bf16, K-major core matrices) that
// the tensor core reads as the B operand.
#pragma once

#include "csa2_device.cuh"
#include "tc.cuh"

namespace csa2 {
namespace score {

// Two E4M3 scale bytes (low byte first) -> one f16 pair (exact).
__device__ __forceinline__ uint32_t e4m3_pair(uint32_t two) {
  uint32_t f;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f) : "h"((uint16_t)(two & 0xFFFFu)));
  return f;
}

// Two E4M3 scale bytes (low byte first) -> each as a broadcast f16x2 (exact).
__device__ __forceinline__ void e4m3_pair_bcast(uint32_t two, uint32_t& lo2, uint32_t& hi2) {
  uint32_t f;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f) : "h"((uint16_t)(two & 0xFFFFu)));
  asm("prmt.b32 %0, %1, 0, 0x1010;" : "=r"(lo2) : "r"(f));
  asm("prmt.b32 %0, %1, 0, 0x3232;" : "=r"(hi2) : "r"(f));
}

// Four bytes of packed E2M1 pairs -> four f16x2 (element 2i of a byte in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

// Two fp32 lanes at once (the packed f32x2 FMA-pipe instructions): a + b,
// and a * b + c, each lane rounded as its scalar form.
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  uint64_t ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Eight channels of one indexer query row (bf16 bits in w[4], channels
// 2j / 2j+1 in the low / high half of w[j]) made into the tensor core's
// operand type: f16 (exact for |x| in [2^-17, 65504]) or kept bf16.  With
// q_fp4 the row is first encoded like a cache entry (E4M3 scale nearest
// amax / 6 per 16 channels, E2M1 codes, both by exact comparisons) and read
// back; the 16-channel group is this lane's 8 channels and its neighbour
// lane's (lane ^ 1), whose maximum is shared by one shuffle.  Returns
// nonzero when a bf16 value made into f16 was outside the f16 range (or not
// finite): the caller reports CSA2_ERR_RANGE.
template <bool kBf16>
__device__ __forceinline__ uint32_t q_operand8(uint32_t (&w)[4], bool q_fp4) {
  uint32_t bad = 0;
  if (q_fp4) {
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(w[j] << 16);
      f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const float sc = e4m3_pos(e4m3_scale_code(amax));
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = e2m1_to_float(e2m1_code(f[j], sc)) * sc;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (kBf16) {
        w[j] = (__float_as_uint(f[2 * j]) >> 16) | (__float_as_uint(f[2 * j + 1]) & 0xFFFF0000u);
      } else {
        const __half2 h2 = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
        w[j] = *reinterpret_cast<const uint32_t*>(&h2);
      }
    }
  } else if (!kBf16) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h2 = __floats2half2_rn(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
      w[j] = *reinterpret_cast<const uint32_t*>(&h2);
      bad |= ((w[j] & 0x7C007C00u) + 0x04000400u) & 0x80008000u;  // an infinite or NaN half
    }
  }
  return bad;
}

}  // namespace score
}  // namespace csa2
