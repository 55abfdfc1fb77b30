// Instantiations and launch of the skinny weight-streaming GEMM (see skinny.cuh).
#include <atomic>

#include "internal.h"

namespace ql {

size_t skinny_smem(int fmt, int mt, int kc) {
  switch (fmt) {
    case FMT_INT8: return mt == 1 ? skinny_smem_bytes<FMT_INT8, 1>(kc) : skinny_smem_bytes<FMT_INT8, 2>(kc);
    case FMT_FP8: return mt == 1 ? skinny_smem_bytes<FMT_FP8, 1>(kc) : skinny_smem_bytes<FMT_FP8, 2>(kc);
    default: return mt == 1 ? skinny_smem_bytes<FMT_MXFP4, 1>(kc) : skinny_smem_bytes<FMT_MXFP4, 2>(kc);
  }
}

// K split: enough CTAs to keep about two resident per SM, and an activation tile that fits
// in ~96 KB of shared memory.  kc is a multiple of the per-CTA K step (chunk x K slices).
SplitK skinny_split(int fmt, int mt, int64_t row_blocks, int64_t K) {
  const int chunk = (fmt == FMT_MXFP4) ? 128 : 64;
  const int xpad = (fmt == FMT_MXFP4) ? 32 : 8;
  const int64_t kstep = (int64_t)chunk * SK_KW;
  const int64_t budget = 96 * 1024;
  int64_t max_kc = (budget / (8 * mt * 2) - xpad) / kstep * kstep;
  if (max_kc < kstep) max_kc = kstep;
  const int64_t target = 2 * kNumSMs;
  int64_t ks_occ = (target + row_blocks - 1) / row_blocks;
  int64_t ks_mem = (K + max_kc - 1) / max_kc;
  int64_t ks = ks_occ > ks_mem ? ks_occ : ks_mem;
  const int64_t ks_max = (K + kstep - 1) / kstep;
  if (ks > ks_max) ks = ks_max;
  if (ks < 1) ks = 1;
  int64_t kc = ((K + ks - 1) / ks + kstep - 1) / kstep * kstep;
  if (kc > max_kc) kc = max_kc;
  ks = (K + kc - 1) / kc;
  return SplitK{(int)ks, (int)kc};
}

template <int FMT, int MT, int EPI>
static cudaError_t launch_one(const SkinnyArgs& a, dim3 grid, cudaStream_t st, bool pdl) {
  auto kfn = skinny_gemm_kernel<FMT, MT, EPI>;
  const size_t smem = skinny_smem_bytes<FMT, MT>(a.kc);
  // raise the dynamic shared-memory limit once (to the largest size seen), so that calls made
  // during CUDA-graph capture only enqueue the launch
  static std::atomic<int> attr_set{0};
  if (!attr_set.load()) {
    cudaError_t err = raise_smem_limit(kfn);
    if (err != cudaSuccess) return err;
    attr_set.store(1);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(SK_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kfn, a);
}

cudaError_t launch_skinny(int fmt, int mt, int epi, const SkinnyArgs& a, dim3 grid, cudaStream_t st, bool pdl) {
#define QL_CASE(F, E)                                                               \
  if (fmt == F && epi == E) {                                                       \
    return mt == 1 ? launch_one<F, 1, E>(a, grid, st, pdl) : launch_one<F, 2, E>(a, grid, st, pdl); \
  }
  QL_CASE(FMT_INT8, EPI_INT8)
  QL_CASE(FMT_FP8, EPI_LINEAR)
  QL_CASE(FMT_MXFP4, EPI_LINEAR)
  QL_CASE(FMT_MXFP4, EPI_GATEUP)
  QL_CASE(FMT_MXFP4, EPI_DOWN)
#undef QL_CASE
  return cudaErrorInvalidValue;
}

}  // namespace ql
