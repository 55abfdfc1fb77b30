// Grouped MoE for batches of more than 16 tokens on the tcgen05 path ([DSV4] §0.3, the grouped
// batch MoE, with the 1x128 E4M3 activations of the block-scaled GEMM at both expert GEMMs):
//   routing (a warp per token) -> dispatch (one CTA: offsets, dispatch rows, the tile list of
//   the grouped GEMMs) -> x quantised per 128-K group, written to each of its token's dispatch
//   rows -> grouped gate_up GEMM (fp32 gate/up rows per pair) -> h = bf16(swiglu(g, u))
//   quantised per 128-K group into the down GEMM's dispatch rows -> grouped down GEMM (fp32 o
//   rows per pair) -> the weighted combine.
// Within one expert the order of its dispatch rows changes no result: every output element is
// its own dot product over the same K order.
#include "internal.h"
#include "quant_e4m3.cuh"
#include "route.cuh"

namespace ql {

// ------------------------------------------------------------------ routing
// One warp per token (E <= 1024), routed by route_token_warp.
__global__ void __launch_bounds__(256) moe_route_many_kernel(const MoeGroupArgs a) {
  const int m = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (m >= a.M) return;
  const int E = a.E, topk = a.topk;
  int my_e = -1;
  float my_w = 0.f;
  if (a.logits) {
    route_token_warp(a.logits + (int64_t)m * E, E, topk, a.renorm != 0, my_e, my_w);
  } else if (lane < topk) {
    my_e = a.ids_in[(int64_t)m * topk + lane];
    my_w = a.w_in[(int64_t)m * topk + lane];
    if (my_e < 0 || my_e >= E) {
      raise_flag(a.status, 2u);
      my_e = -1;  // not dispatched; the combine skips it
    }
  }
  if (lane < topk) {
    const int64_t pi = (int64_t)m * topk + lane;
    a.ids[pi] = my_e;
    a.wts[pi] = my_w;
    if (a.ids_dbg) a.ids_dbg[pi] = my_e;
    if (a.w_dbg) a.w_dbg[pi] = my_w;
    if (my_e >= 0) atomicAdd(&a.counts[my_e], 1);
  }
}

// ------------------------------------------------------------------ dispatch
// exclusive scan of one int per thread over a block of 1024 threads
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) s_warp[w] = inc;
  __syncthreads();
  if (w == 0) {
    int t = s_warp[lane], ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += u;
    }
    s_warp[lane] = ti - t;  // exclusive offset of each warp
  }
  __syncthreads();
  const int r = s_warp[w] + inc - v;
  __syncthreads();  // s_warp is reused by the next scan
  return r;
}

// One CTA of 1024 threads (E <= 1024): offsets[e] = first dispatch row of expert e, the tile
// list (expert, first row, rows) of up to tt rows each in increasing expert order, the dispatch
// row of every routed pair and the pair of every dispatch row.
__global__ void __launch_bounds__(1024) moe_dispatch_kernel(const MoeGroupArgs a) {
  __shared__ int s_warp[32];
  __shared__ int s_cur[1024];
  const int e = threadIdx.x, E = a.E, tt = a.tt;
  const int c = e < E ? a.counts[e] : 0;
  const int off = block_exclusive_scan(c, s_warp);
  const int nt = (c + tt - 1) / tt;
  const int t_off = block_exclusive_scan(nt, s_warp);
  if (e < E) {
    a.offsets[e] = off;
    s_cur[e] = off;
    for (int i = 0; i < nt; ++i) a.tiles[t_off + i] = make_int4(e, off + i * tt, min(tt, c - i * tt), 0);
  }
  if (e == E - 1) {
    a.offsets[E] = off + c;
    *a.ntiles = t_off + nt;
  }
  __syncthreads();
  const int P = a.M * a.topk;
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int x = a.ids[p];
    int pos = -1;
    if (x >= 0) {
      pos = atomicAdd(&s_cur[x], 1);
      a.pairs[pos] = p;
    }
    a.pos_of_pair[p] = pos;
  }
}

// ------------------------------------------------------------------ activations of gate_up
// a warp per (token, 128-group): the group's E4M3 codes and UE8M0 scale, written to each
// dispatch row of the token's routed pairs
__global__ void __launch_bounds__(256) moe_quant_scatter_kernel(const MoeGroupArgs a) {
  const int H = a.H, ng = H / 128;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (gw >= a.M * ng) return;
  const int m = gw / ng, gi = gw - m * ng;
  const int k = gi * 128 + lane * 4;
  const uint2 v = *reinterpret_cast<const uint2*>(a.x + (int64_t)m * a.ldx + k);
  const float f[4] = {__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                      __uint_as_float(v.y & 0xFFFF0000u)};
  uint32_t sb;
  const uint32_t codes = e4m3_group_encode(f, sb);
  for (int j = 0; j < a.topk; ++j) {
    const int pos = a.pos_of_pair[(int64_t)m * a.topk + j];
    if (pos < 0) continue;
    *reinterpret_cast<uint32_t*>(a.q_gu + (int64_t)pos * H + k) = codes;
    if (lane == 0) a.s_gu[(int64_t)pos * ng + gi] = (uint8_t)sb;
  }
}

// ------------------------------------------------------------------ activations of down
// a warp per (dispatch row, 128-group of I): h = bf16(swiglu(g, u)) from the pair's fp32 gate and
// up sums, then the group's E4M3 codes and UE8M0 scale in the same row of the down GEMM's input
__global__ void __launch_bounds__(256) moe_h_quant_kernel(const MoeGroupArgs a) {
  const int I = a.I, ng = I / 128;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int rows = a.offsets[a.E];  // dispatch rows in use
  if (gw >= rows * ng) return;
  const int r = gw / ng, gi = gw - r * ng;
  const int pair = a.pairs[r];
  const int k = gi * 128 + lane * 4;
  const float* gp = a.gu + (int64_t)pair * 2 * I;
  const float4 g = *reinterpret_cast<const float4*>(gp + k);
  const float4 u = *reinterpret_cast<const float4*>(gp + I + k);
  const float gv[4] = {g.x, g.y, g.z, g.w}, uv[4] = {u.x, u.y, u.z, u.w};
  uint16_t hb[4];
  float f[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    hb[i] = f32_to_bf16_rn(swiglu_f32(gv[i], uv[i], a.act_alpha, a.act_limit));
    f[i] = bf16_bits_to_f32(hb[i]);
  }
  if (a.h_dbg)
    *reinterpret_cast<uint2*>(a.h_dbg + (int64_t)pair * I + k) =
        make_uint2((uint32_t)hb[0] | ((uint32_t)hb[1] << 16), (uint32_t)hb[2] | ((uint32_t)hb[3] << 16));
  uint32_t sb;
  const uint32_t codes = e4m3_group_encode(f, sb);
  *reinterpret_cast<uint32_t*>(a.q_dn + (int64_t)r * I + k) = codes;
  if (lane == 0) a.s_dn[(int64_t)r * ng + gi] = (uint8_t)sb;
}

// ------------------------------------------------------------------ launches
cudaError_t launch_moe_grouped_prologue(const MoeGroupArgs& a, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(a.counts, 0, (size_t)a.E * 4, st);
  if (e != cudaSuccess) return e;
  moe_route_many_kernel<<<(a.M + 7) / 8, 256, 0, st>>>(a);
  moe_dispatch_kernel<<<1, 1024, 0, st>>>(a);
  const int warps = a.M * (a.H / 128);
  moe_quant_scatter_kernel<<<(warps + 7) / 8, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_moe_h_quant(const MoeGroupArgs& a, cudaStream_t st) {
  const int warps = a.M * a.topk * (a.I / 128);  // bound: every pair dispatched
  moe_h_quant_kernel<<<(warps + 7) / 8, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace ql
