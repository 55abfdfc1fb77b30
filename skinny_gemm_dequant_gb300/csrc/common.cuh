// Shared device helpers of the sm_103a quantized linear kernels: raw loads, format
// conversions, the legacy-path tensor-core fragment MMA, PDL controls, bounded waits.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qlinear.h"

namespace ql {

// ------------------------------------------------------------------ status word
// workspace[0..255] : [0] status flags, [1] reserved, [16..63] split-K tile counters
// (tile counters grow beyond 64 entries into the op-specific region when needed).
struct DevStatus {
  uint32_t flags;
};

__device__ __forceinline__ void raise_flag(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// ------------------------------------------------------------------ loads
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  // weights are read exactly once: do not allocate them in L1
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// ------------------------------------------------------------------ bf16 / fp16 helpers
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// fp32 -> bf16, round to nearest even (NaN kept quiet)
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// the two FP8 pairs of a word (bytes 0,1 -> lo, bytes 2,3 -> hi), exact: the word is split into
// its 16-bit halves as registers, not by masking and shifting
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h0;\n\tcvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
__device__ __forceinline__ void e5m2x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e5m2x2 %0, h0;\n\tcvt.rn.f16x2.e5m2x2 %1, h1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// the four E2M1 pairs of a word (byte i -> o[i], low nibble -> low lane), exact.  Unpacking the
// word into byte registers first costs about a third less than shifting out each byte
// (measured on GB300: 8 codes per word, 304 CTAs x 256 threads).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// four signed int8 (one word) to two exact f16x2: lanes (b0,b1) and (b2,b3).
// 0x6400 | u is the f16 value 1024 + u for u in [0,255]; with u = b + 128 (xor 0x80)
// subtracting 1152 returns b exactly.
__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x7170;" : "=r"(a) : "r"(u), "r"(0x64646464u));   // bytes 0,1
  asm("prmt.b32 %0, %1, %2, 0x7372;" : "=r"(b) : "r"(u), "r"(0x64646464u));   // bytes 2,3
  const uint32_t bias = 0x64806480u;                                            // 1152, 1152
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

// UE8M0 byte -> fp32 2^(b-127); b = 0 gives the fp32 subnormal 2^-127, b = 255 NaN
__device__ __forceinline__ float ue8m0_to_f32(uint32_t b) {
  b &= 0xFFu;
  if (b == 0) return __uint_as_float(0x00400000u);
  if (b == 255) return __uint_as_float(0x7FC00000u);
  return __uint_as_float(b << 23);
}

// two UE8M0 bytes (low byte -> .x) to exact fp32 2^(b-127) (b = 0: 2^-127, b = 255: NaN) through
// the hardware's ue8m0x2 -> bf16x2 conversion: bf16 keeps fp32's exponent range, so both are exact
__device__ __forceinline__ float2 ue8m0x2_to_f32x2(uint32_t two_bytes) {
  uint32_t r;
  asm("cvt.rn.bf16x2.ue8m0x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two_bytes));
  return make_float2(__uint_as_float(r << 16), __uint_as_float(r & 0xFFFF0000u));
}

// ------------------------------------------------------------------ warp MMA (f16 -> f32)
// D[16x8] += A[16x16] * B[16x8]; A row-major fragments a0..a3, B "col" fragments b0,b1.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  // a pure register operation: not volatile, so the compiler may schedule it around loads
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D[16x8] += A[16x16] * B[16x8] on bf16 operands (f32 accumulate)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

// the MoE expert activation: silu(alpha * min(g, limit)) * clamp(u, -limit, limit); limit =
// +infinity and alpha = 1 give the plain silu(g) * u (fminf / fmaxf against infinity are exact)
__device__ __forceinline__ float swiglu_f32(float g, float u, float alpha, float limit) {
  return silu_f32(alpha * fminf(g, limit)) * fminf(fmaxf(u, -limit), limit);
}

}  // namespace ql
