// Activation quantisation prologues.
//
//  * INT8, dynamic per token ([Z100] §二.2.1, the "scaled_int8_quant" step in front of the
//    sdot4 GEMV): x_s = amax/127, x_q = clamp(rint(x/x_s), -127, 127), IEEE fp32 divisions.
//  * E4M3, dynamic per token and per 128-K group with a UE8M0 scale ([DSV4] §3.3 quant_config:
//    activation_scheme dynamic, fmt e4m3, scale_fmt ue8m0): scale 2^e with e the smallest
//    integer such that amax <= 448 * 2^e (so no code saturates), codes rounded to nearest even.
// Both kernels trigger the dependent GEMM launch at entry (programmatic dependent launch), so
// the GEMM starts streaming its weights while the activations are being quantised.
#include "internal.h"
#include "quant_e4m3.cuh"

namespace ql {

__global__ void __launch_bounds__(256) quant_int8_kernel(const uint16_t* __restrict__ x, int K, int64_t ldx,
                                                         int8_t* __restrict__ xq, float* __restrict__ xs,
                                                         int8_t* xq_dbg, float* xs_dbg) {
  pdl_launch_dependents();
  const int m = blockIdx.x;
  const uint16_t* xr = x + (int64_t)m * ldx;
  __shared__ float s_red[8];
  float amax = 0.f;
  for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? s_red[threadIdx.x] : 0.f;
    v = warp_max(v);
    if (threadIdx.x == 0) s_red[0] = v;
  }
  __syncthreads();
  amax = s_red[0];
  const float s = __fdiv_rn(amax, 127.0f);
  int8_t* qr = xq + (int64_t)m * K;
  for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float xv = (i & 1) ? __uint_as_float(w[i >> 1] & 0xFFFF0000u) : __uint_as_float(w[i >> 1] << 16);
      int q = 0;
      if (s > 0.f) {
        float r = rintf(__fdiv_rn(xv, s));
        r = fminf(fmaxf(r, -127.f), 127.f);
        q = (int)r;
      }
      packed[i >> 2] |= ((uint32_t)(q & 0xFF)) << (8 * (i & 3));
    }
    *reinterpret_cast<uint2*>(qr + k) = make_uint2(packed[0], packed[1]);
    if (xq_dbg) *reinterpret_cast<uint2*>(xq_dbg + (int64_t)m * K + k) = make_uint2(packed[0], packed[1]);
  }
  if (threadIdx.x == 0) {
    xs[m] = s;
    if (xs_dbg) xs_dbg[m] = s;
  }
}

// one warp per (token, 128-group); lane holds 4 consecutive values
__global__ void __launch_bounds__(256) quant_e4m3_kernel(const uint16_t* __restrict__ x, int M, int K, int64_t ldx,
                                                         uint8_t* __restrict__ q, int64_t ldq,
                                                         uint8_t* __restrict__ s, int64_t lds, int s_transposed,
                                                         uint8_t* q_dbg, uint8_t* s_dbg) {
  pdl_launch_dependents();
  const int ng = K / 128;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= M * ng) return;
  const int m = gw / ng, gi = gw % ng;
  const int k = gi * 128 + lane * 4;
  const uint2 v = *reinterpret_cast<const uint2*>(x + (int64_t)m * ldx + k);
  const float f[4] = {__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                      __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u)};
  uint32_t sb;
  const uint32_t codes = e4m3_group_encode(f, sb);
  *reinterpret_cast<uint32_t*>(q + (int64_t)m * ldq + k) = codes;
  if (q_dbg) *reinterpret_cast<uint32_t*>(q_dbg + (int64_t)m * K + k) = codes;
  if (lane == 0) {
    const uint8_t b = (uint8_t)sb;
    if (s_transposed) s[(int64_t)gi * lds + m] = b;
    else s[(int64_t)m * lds + gi] = b;
    if (s_dbg) s_dbg[(int64_t)m * ng + gi] = b;
  }
}

cudaError_t launch_quant_int8(const uint16_t* x, int M, int K, int64_t ldx, int8_t* xq, float* xs,
                              int8_t* xq_dbg, float* xs_dbg, cudaStream_t st) {
  quant_int8_kernel<<<M, 256, 0, st>>>(x, K, ldx, xq, xs, xq_dbg, xs_dbg);
  return cudaGetLastError();
}

cudaError_t launch_quant_e4m3(const uint16_t* x, int M, int K, int64_t ldx, uint8_t* q, int64_t ldq,
                              uint8_t* s, int64_t lds, int s_transposed, uint8_t* q_dbg, uint8_t* s_dbg,
                              cudaStream_t st) {
  const int warps = M * (K / 128);
  quant_e4m3_kernel<<<(warps + 7) / 8, 256, 0, st>>>(x, M, K, ldx, q, ldq, s, lds, s_transposed, q_dbg, s_dbg);
  return cudaGetLastError();
}

}  // namespace ql
