// Host-side declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "skinny.cuh"

namespace ql {

constexpr int kNumSMs = 152;  // GB300: 2 dies x 76 SMs (checked against the device at launch)

// launch helpers (return the CUDA error of the launch)
cudaError_t launch_quant_int8(const uint16_t* x, int M, int K, int64_t ldx, int8_t* xq, float* xs,
                              int8_t* xq_dbg, float* xs_dbg, cudaStream_t st);
cudaError_t launch_quant_e4m3(const uint16_t* x, int M, int K, int64_t ldx, uint8_t* q, int64_t ldq,
                              uint8_t* s, int64_t lds, int s_transposed, uint8_t* q_dbg, uint8_t* s_dbg,
                              cudaStream_t st);
cudaError_t launch_skinny(int fmt, int mt, int epi, const SkinnyArgs& a, dim3 grid, cudaStream_t st, bool pdl);

struct MoeRouteArgs {
  const uint16_t* logits;
  const int32_t* ids_in;
  const float* w_in;
  int M, E, topk, renorm;
  int32_t* ids;
  float* wts;
  int32_t* offsets;
  int32_t* pairs;
  int32_t* uniq;
  int32_t* nuniq;
  int32_t* ids_dbg;
  float* w_dbg;
  uint32_t* status;
};
cudaError_t launch_moe_route(const MoeRouteArgs& r, cudaStream_t st);
cudaError_t launch_moe_combine(const float* o, const int32_t* ids, const float* w, int M, int topk, int H,
                               uint16_t* y, cudaStream_t st);

// persistent TMA-fed skinny GEMM (skinny2.cuh); its activation image is written kXCopies times
constexpr int kXCopies = 2;
struct Skinny2Plan {
  int mt, mp;             // token tiles of 8, padded token rows
  int64_t nb;             // 128-row blocks
  int nk;                 // units per row block
  int64_t kpad;           // K rounded up to whole units (row length of the activation image)
  int64_t total;          // nb * nk
  int grid;               // CTAs (one per SM)
  int64_t units_per_cta;
  size_t fp8_scale_bytes; // shared memory for the FP8 block-scale rows
};
Skinny2Plan skinny2_plan(int fmt, int64_t M, int64_t N, int64_t K, int block_n, int64_t slots = 1);
// bytes at the start of every workspace that must be zero before a call (the status word, the
// counters and the split-K tickets); the kernels leave them zero
size_t workspace_zero_bytes();
struct Skinny2Args;
cudaError_t launch_skinny2(int fmt, const Skinny2Plan& p, const Skinny2Args& a, const uint8_t* w, int64_t ldw,
                           cudaStream_t st);
// the two MXFP4 expert GEMVs of the MoE (kind: S2_MOE_GU or S2_MOE_DN, skinny2.cuh)
cudaError_t launch_moe2(int kind, const Skinny2Plan& p, const Skinny2Args& a, const uint8_t* w, int64_t ldw,
                        int64_t w_estride, int experts, cudaStream_t st);

// grouped MoE for M > 16 (kernels_moe_grouped.cu): routing, dispatch and the activation launches
struct MoeGroupArgs {
  const uint16_t* logits;  // bf16 [M, E] or null
  const int32_t* ids_in;   // given routing [M, topk] or null
  const float* w_in;
  int M, E, topk, renorm;
  int32_t* ids;  // [M * topk], -1 for a pair that is not dispatched
  float* wts;
  int32_t* counts;  // [E], zeroed by the prologue
  int32_t* ids_dbg;
  float* w_dbg;
  uint32_t* status;
  int tt;            // rows per tile of the grouped GEMMs
  int32_t* offsets;  // [E + 1]
  int4* tiles;       // [tiles bound]
  int32_t* ntiles;
  int32_t* pairs;        // dispatch row -> pair
  int32_t* pos_of_pair;  // pair -> dispatch row (-1: none)
  const uint16_t* x;     // bf16 [M, ldx]
  int64_t ldx;
  int H, I;
  uint8_t* q_gu;  // E4M3 [M * topk, H] by dispatch row
  uint8_t* s_gu;  // UE8M0 [M * topk, H / 128]
  float* gu;      // fp32 [M * topk, 2I] by pair
  uint8_t* q_dn;  // E4M3 [M * topk, I] by dispatch row
  uint8_t* s_dn;  // UE8M0 [M * topk, I / 128]
  uint16_t* h_dbg;  // bf16 [M * topk, I] by pair, or null
  float act_alpha, act_limit;
};
cudaError_t launch_moe_grouped_prologue(const MoeGroupArgs& a, cudaStream_t st);
cudaError_t launch_moe_h_quant(const MoeGroupArgs& a, cudaStream_t st);

// split-K choice of the skinny kernel (shared by the workspace query and the launch)
struct SplitK {
  int ks, kc;
};
SplitK skinny_split(int fmt, int mt, int64_t row_blocks, int64_t K);
size_t skinny_smem(int fmt, int mt, int kc);

uint32_t wait_limit();

// sharded-layer kernels (kernels_shard.cu)
cudaError_t launch_token_amax(const uint16_t* x, int M, int K, int64_t ldx, float* amax, cudaStream_t st);
cudaError_t launch_int8_epilogue(const int32_t* acc, int M, int N, const float* amax, const float* w_s, int w_s_len,
                                 const uint16_t* bias, uint16_t* y, int64_t ldy, cudaStream_t st);
cudaError_t launch_finish_f32(const float* y32, int M, int N, int64_t ld32, const uint16_t* bias, uint16_t* y,
                              int64_t ldy, cudaStream_t st);

// Raise a kernel's dynamic shared-memory limit to the device's opt-in maximum minus its static
// shared memory.  Done once per kernel, before any launch, so calls made during CUDA-graph
// capture only enqueue work.
template <class F>
cudaError_t raise_smem_limit(F* kfn) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kfn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
  // prefer the largest shared-memory carveout, so kernels sized for several CTAs per SM get them
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return e;
}

}  // namespace ql
