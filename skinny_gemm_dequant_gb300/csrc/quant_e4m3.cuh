// 1x128 E4M3 activation quantisation of one 128-element group held by a warp (4 consecutive
// values per lane): the UE8M0 scale 2^e is the smallest power of two with amax <= 448 * 2^e
// (e >= -127), the codes are round-to-nearest-even E4M3 of x * 2^-e, saturating.  Used by every
// launch that quantises activations for the block-scaled tensor-core GEMM.
#pragma once
#include "common.cuh"

namespace ql {

// two fp32 -> two E4M3 codes (v0 in the low byte), round to nearest even, saturating
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float v0, float v1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(v1), "f"(v0));
  return r;
}

// the lane's 4 codes packed (value 0 in the low byte) and the group's scale byte 127 + e
__device__ __forceinline__ uint32_t e4m3_group_encode(const float (&f)[4], uint32_t& scale_byte) {
  float amax = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
  amax = warp_max(amax);
  int e = 0;
  if (amax > 0.f) {
    // start two below the answer and step up: smallest e with amax <= 448 * 2^e (exact tests)
    const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
    e = ex - 9;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (amax > ldexpf(448.0f, e)) ++e;
  }
  e = max(e, -127);
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, e in [-127, 126]
  const uint32_t c01 = f32x2_to_e4m3x2(f[0] * inv, f[1] * inv);
  const uint32_t c23 = f32x2_to_e4m3x2(f[2] * inv, f[3] * inv);
  scale_byte = (uint32_t)(127 + e);
  return (c01 & 0xFFFFu) | (c23 << 16);
}

}  // namespace ql
