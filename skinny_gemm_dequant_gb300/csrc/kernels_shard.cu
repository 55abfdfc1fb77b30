// Kernels around the collective steps of a sharded (tensor-parallel) linear layer:
//  * the per-token amax of a K shard of x: a row-parallel INT8 layer takes the maximum over
//    the shards (all-reduce MAX) before any shard quantises, so every shard's codes are the
//    unsharded layer's codes ([Z100] §二.2.1: x_s = max|x| / 127 over the token's whole row);
//  * the INT8 epilogue from int32 sums already added over the shards (all-reduce SUM, exact):
//    y = bf16((acc * x_s) * w_s) (+ bias after the cast), x_s = amax / 127 (IEEE division);
//  * the single bf16 rounding (+ bias after the cast) of fp32 partial sums added over shards.
#include "internal.h"

namespace ql {

__global__ void __launch_bounds__(256) token_amax_kernel(const uint16_t* __restrict__ x, int K, int64_t ldx,
                                                         float* __restrict__ amax_out) {
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
  if (threadIdx.x == 0) {
    float v = s_red[0];
    for (int i = 1; i < 8; ++i) v = fmaxf(v, s_red[i]);
    amax_out[m] = v;
  }
}

__global__ void __launch_bounds__(256) int8_epilogue_kernel(const int32_t* __restrict__ acc, int M, int N,
                                                            const float* __restrict__ amax,
                                                            const float* __restrict__ w_s, int w_s_len,
                                                            const uint16_t* __restrict__ bias, uint16_t* y,
                                                            int64_t ldy) {
  const int64_t total = (int64_t)M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(i / N), n = (int)(i - (int64_t)m * N);
    const float xs = __fdiv_rn(amax[m], 127.0f);
    uint16_t yb = f32_to_bf16_rn(__fmul_rn(__fmul_rn((float)acc[i], xs), w_s[w_s_len > 1 ? n : 0]));
    if (bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + bf16_bits_to_f32(bias[n]));
    y[(int64_t)m * ldy + n] = yb;
  }
}

__global__ void __launch_bounds__(256) finish_f32_kernel(const float* __restrict__ y32, int M, int N, int64_t ld32,
                                                         const uint16_t* __restrict__ bias, uint16_t* y,
                                                         int64_t ldy) {
  const int64_t total = (int64_t)M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(i / N), n = (int)(i - (int64_t)m * N);
    uint16_t yb = f32_to_bf16_rn(y32[(int64_t)m * ld32 + n]);
    if (bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + bf16_bits_to_f32(bias[n]));
    y[(int64_t)m * ldy + n] = yb;
  }
}

static unsigned elementwise_grid(int64_t total) {
  const int64_t b = (total + 255) / 256;
  return (unsigned)(b < kNumSMs * 8 ? (b > 0 ? b : 1) : kNumSMs * 8);
}

cudaError_t launch_token_amax(const uint16_t* x, int M, int K, int64_t ldx, float* amax, cudaStream_t st) {
  token_amax_kernel<<<M, 256, 0, st>>>(x, K, ldx, amax);
  return cudaGetLastError();
}

cudaError_t launch_int8_epilogue(const int32_t* acc, int M, int N, const float* amax, const float* w_s, int w_s_len,
                                 const uint16_t* bias, uint16_t* y, int64_t ldy, cudaStream_t st) {
  int8_epilogue_kernel<<<elementwise_grid((int64_t)M * N), 256, 0, st>>>(acc, M, N, amax, w_s, w_s_len, bias, y, ldy);
  return cudaGetLastError();
}

cudaError_t launch_finish_f32(const float* y32, int M, int N, int64_t ld32, const uint16_t* bias, uint16_t* y,
                              int64_t ldy, cudaStream_t st) {
  finish_f32_kernel<<<elementwise_grid((int64_t)M * N), 256, 0, st>>>(y32, M, N, ld32, bias, y, ldy);
  return cudaGetLastError();
}

}  // namespace ql
