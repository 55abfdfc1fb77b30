// MoE decode helpers: softmax top-k routing with grouped dispatch, and the weighted combine.
//
// Routing ([DSV4] §0.1, the M=1 routing fast path "Q1", and §0.3 grouped batch MoE): per token
// p = softmax(logits), the topk experts with the largest logits (equal logits: lower expert id
// first), weights p[ids] (renormalised on request), by route_token_warp.  Dispatch groups the
// (token, slot) pairs by expert (increasing id, stable in pair order) and lists the distinct
// experts in increasing id; the expert GEMMs work on one slot per distinct expert.
#include "internal.h"
#include "route.cuh"

namespace ql {

constexpr int kRouteThreads = 512;  // one warp per token, M <= 16

__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(const MoeRouteArgs r) {
  __shared__ int s_ids[256];
  __shared__ int s_cnt[1025];
  const int M = r.M, E = r.E, topk = r.topk;
  const int P = M * topk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (r.logits) {
    if (warp < M) {  // a warp per token
      const int m = warp;
      int id = -1;
      float w = 0.f;
      route_token_warp(r.logits + (int64_t)m * E, E, topk, r.renorm != 0, id, w);
      if (lane < topk) {
        const int p = m * topk + lane;
        s_ids[p] = id;
        r.ids[p] = id;
        r.wts[p] = w;
        if (r.ids_dbg) r.ids_dbg[p] = id;
        if (r.w_dbg) r.w_dbg[p] = w;
      }
    }
  } else {
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
      int e = r.ids_in[p];
      if (e < 0 || e >= E) {
        raise_flag(r.status, 2u);
        e = -1;
      }
      s_ids[p] = e;
      r.ids[p] = e;
      r.wts[p] = r.w_in[p];
      if (r.ids_dbg) r.ids_dbg[p] = e;
      if (r.w_dbg) r.w_dbg[p] = r.w_in[p];
    }
  }
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  // dispatch: pairs grouped by expert (increasing id), stable in pair order; distinct experts
  // listed in increasing id
  for (int p = threadIdx.x; p < P; p += blockDim.x)
    if (s_ids[p] >= 0) atomicAdd(&s_cnt[s_ids[p]], 1);
  __syncthreads();
  if (warp == 0) {
    // exclusive scans of the counts (offsets) and of the used flags (slots), E/32 per lane
    const int per = (E + 31) / 32, e0 = lane * per;
    int c = 0, u = 0;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      c += s_cnt[e];
      u += s_cnt[e] > 0;
    }
    int ci = c, ui = u;  // inclusive warp scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int cv = __shfl_up_sync(0xffffffffu, ci, o), uv = __shfl_up_sync(0xffffffffu, ui, o);
      if (lane >= o) {
        ci += cv;
        ui += uv;
      }
    }
    int run = ci - c, nu = ui - u;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      const int n = s_cnt[e];
      r.offsets[e] = run;
      if (n > 0) r.uniq[nu++] = e;
      s_cnt[e] = run;  // now the expert's first dispatch position
      run += n;
    }
    if (lane == 31) {
      r.offsets[E] = run;
      *r.nuniq = nu;
    }
  }
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int e = s_ids[p];
    if (e < 0) continue;
    int rank = 0;  // earlier pairs of the same expert
    for (int q = 0; q < p; ++q) rank += s_ids[q] == e;
    r.pairs[s_cnt[e] + rank] = p;
  }
  __syncthreads();
  pdl_launch_dependents();
}

cudaError_t launch_moe_route(const MoeRouteArgs& r, cudaStream_t st) {
  moe_route_kernel<<<1, kRouteThreads, 0, st>>>(r);
  return cudaGetLastError();
}

// y[m, n] = bf16( sum_j w[m,j] * o[m*topk + j, n] ), summed in slot order
__global__ void __launch_bounds__(256) moe_combine_kernel(const float* __restrict__ o, const int32_t* __restrict__ ids,
                                                          const float* __restrict__ w, int topk, int H,
                                                          uint16_t* __restrict__ y) {
  pdl_wait();
  const int m = blockIdx.y;
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= H) return;
  float acc = 0.f;
  for (int j = 0; j < topk; ++j) {
    const int p = m * topk + j;
    if (ids[p] >= 0) acc = fmaf(w[p], o[(int64_t)p * H + n], acc);
  }
  y[(int64_t)m * H + n] = f32_to_bf16_rn(acc);
}

cudaError_t launch_moe_combine(const float* o, const int32_t* ids, const float* w, int M, int topk, int H,
                               uint16_t* y, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((H + 255) / 256, M, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_combine_kernel, o, ids, w, topk, H, y);
}

}  // namespace ql
