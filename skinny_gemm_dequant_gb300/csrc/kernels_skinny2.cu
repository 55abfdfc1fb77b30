// Plan and launch of the persistent TMA-fed skinny GEMM (skinny2_kernel.cuh): work split, tensor
// maps of the weights and of the activation image, shared-memory ring depth.  Dense linear layers
// and the two MXFP4 expert GEMVs of the MoE go through the same kernel.
#include <atomic>

#include <cudaTypedefs.h>

#include "internal.h"
#include "skinny2_kernel.cuh"

namespace ql {

// ------------------------------------------------------------------ plan + launch

// slots: 1 for a dense layer; for the MoE the most distinct experts a call can route to (the
// device knows the actual count and splits the units by it)
Skinny2Plan skinny2_plan(int fmt, int64_t M, int64_t N, int64_t K, int block_n, int64_t slots) {
  Skinny2Plan p;
  p.mt = M <= 8 ? 1 : (M <= 16 ? 2 : 4);  // 8-token MMA tiles (4: INT8 only)
  p.mp = 8 * p.mt;
  const int kpu = fmt == FMT_MXFP4 ? S2Traits<FMT_MXFP4>::KPU
                                   : (fmt == FMT_BF16 ? S2Traits<FMT_BF16>::KPU : S2Traits<FMT_INT8>::KPU);  // K per unit
  p.nb = (N + S2_ROWS - 1) / S2_ROWS;
  p.nk = (int)((K + kpu - 1) / kpu);
  p.kpad = (int64_t)p.nk * kpu;
  p.total = slots * p.nb * p.nk;
  const int64_t sms = (int64_t)kNumSMs * s2_ctas_per_sm(fmt, p.mt);  // fixed: workspace query and launch agree
  p.grid = (int)(p.total < sms ? p.total : sms);
  p.units_per_cta = (p.total + p.grid - 1) / p.grid;
  p.fp8_scale_bytes = 0;
  if (fmt == FMT_FP8) {
    const int64_t nrb = p.units_per_cta / p.nk + 2;
    const int64_t nbr = S2_ROWS / block_n + 2;
    p.fp8_scale_bytes = (size_t)(nrb * nbr * ((K + 127) / 128 * 2 + 2));
  }
  return p;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::atomic<int> done{0};
  if (!done.load()) {
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(q);
    done.store(1);
  }
  return fn;
}

// 3D / 4D views: dims d[0..], byte strides st[1..] of dims 1.., box b[], 128-byte swizzle
static bool mapnd(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank, const uint64_t* d,
                  const uint64_t* st, const uint32_t* b) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5], es[5];
  for (int i = 0; i < rank; ++i) {
    dims[i] = d[i];
    box[i] = b[i];
    es[i] = 1;
    if (i > 0) strides[i - 1] = st[i - 1];
  }
  return fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool map2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// w_estride: bytes between experts' weight matrices (MoE; a dense layer has one "expert")
template <int FMT, int MT, int KIND>
static cudaError_t launch2(const Skinny2Plan& p, Skinny2Args a, const uint8_t* w, int64_t ldw, int64_t w_estride,
                           int experts, cudaStream_t st) {
  using Tr = S2Traits<FMT>;
  constexpr uint32_t STAGE = s2_stage_bytes<FMT, MT>();
  constexpr int Mp = 8 * MT;
  // behind the ring: FP8 block-scale rows (dense FP8) or the routing (MoE gate_up)
  const size_t extra = p.fp8_scale_bytes + (KIND == S2_MOE_GU ? s2_route_bytes(a.M * a.topk, a.E) : 0);
  const size_t fixed = 1024 + extra + 256;  // alignment slack, extra, static
  // per CTA: the SM's 228 KB less 1 KB reserved per resident CTA, capped by the opt-in limit
  const int optin = s2_ctas_per_sm(FMT, MT) == 1 ? 227 * 1024 : (228 * 1024) / s2_ctas_per_sm(FMT, MT) - 1024;
  int S = (int)((optin - fixed) / (STAGE + 16));
  if (S > 8) S = 8;
  if (S < 2) return cudaErrorInvalidValue;
  // local activations: weight-only stages plus the CTA's image of its own K units; taken only
  // when the ring keeps at least the depth of the shared-image layout
  size_t local_bytes = 0;
  uint32_t stage_bytes = STAGE;
  if (KIND == S2_DENSE_LOCAL) {
    const int64_t slots = p.units_per_cta < p.nk ? p.units_per_cta : p.nk;
    if (slots * (Tr::KPU / 8) > 1024) return cudaErrorNotSupported;  // s2_local_image holds <= 4 vectors a thread
    const size_t lb = ((size_t)slots * Tr::NXB * a.M * 128 + 127) & ~size_t(127);
    const uint32_t sb = S2_ROWS * S2_WB + Tr::SCB;
    int SL = (optin > (int)(fixed + lb)) ? (int)((optin - fixed - lb) / (sb + 16)) : 0;
    if (SL > 8) SL = 8;
    if (SL < S || SL < 3) return cudaErrorNotSupported;  // the caller takes the shared image
    S = SL;
    local_bytes = lb;
    stage_bytes = sb;
  }
  a.local_bytes = (int)local_bytes;
  a.stages = S;
  a.bk_shift = 0;
  while (a.block_k > 0 && (1 << a.bk_shift) < a.block_k) ++a.bk_shift;
  a.nk = p.nk;
  a.nb = (int)p.nb;
  a.total = p.total;
  const uint64_t wbytes = FMT == FMT_MXFP4 ? (uint64_t)a.K / 2 : (FMT == FMT_BF16 ? (uint64_t)a.K * 2 : (uint64_t)a.K);
  a.wbytes = (int)wbytes;
  const size_t smem = 1024 + (size_t)S * stage_bytes + (size_t)S * 16 + local_bytes + extra;
  CUtensorMap tw, tw2, tx;
  // whole 128-byte chunks as the third dimension (a box of 2 chunks is one 32 KB TMA operation),
  // experts as the fourth
  const uint64_t nfull = wbytes / 128 > 0 ? wbytes / 128 : 1;
  {
    const uint64_t d[4] = {128, (uint64_t)a.N, nfull, (uint64_t)experts};
    const uint64_t st[3] = {(uint64_t)ldw, 128, (uint64_t)w_estride};
    const uint32_t b[4] = {128, S2_ROWS, S2_CHUNKS, 1};
    if (!mapnd(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, 4, d, st, b)) return cudaErrorInvalidValue;
  }
  if (!map2d(&tw2, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, wbytes, (uint64_t)a.N, (uint64_t)ldw, 128, S2_ROWS))
    return cudaErrorInvalidValue;
  a.xcopies = kXCopies;
  a.kpad = p.kpad;
  if (FMT == FMT_BF16) {
    // the caller's x [M][ldx] bf16: boxes of 64 columns x Mp rows, zeros past K and past M
    if (!map2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.ldx * 2, 64,
               (uint32_t)Mp))
      return cudaErrorInvalidValue;
  } else {
    // image [copies][img_rows][kpad] f16 seen as {64, img_rows, copies, kpad/64}; a box covers
    // Mp rows (rows past img_rows read as zeros)
    const uint64_t d[4] = {64, (uint64_t)a.img_rows, (uint64_t)kXCopies, (uint64_t)(p.kpad / 64)};
    const uint64_t st[3] = {(uint64_t)p.kpad * 2, (uint64_t)a.img_rows * p.kpad * 2, 128};
    const uint32_t b[4] = {64, (uint32_t)Mp, 1, (uint32_t)Tr::NXB};
    if (!mapnd(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.x16, 4, d, st, b)) return cudaErrorInvalidValue;
  }
  auto kfn = skinny2_kernel<FMT, MT, KIND>;
  static std::atomic<int> attr{0};
  if (!attr.load()) {
    cudaError_t e = raise_smem_limit(kfn);
    if (e != cudaSuccess) return e;
    attr.store(1);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
  cfg.blockDim = dim3(S2_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kfn, tw, tw2, tx, a);
}

cudaError_t launch_skinny2(int fmt, const Skinny2Plan& p, const Skinny2Args& a, const uint8_t* w, int64_t ldw,
                           cudaStream_t st) {
  const int64_t es = (int64_t)a.N * ldw;  // one expert
  if (a.local && p.mt == 1 && fmt != FMT_BF16) {
    // every CTA builds its own activation image, when the ring keeps its depth beside it
    cudaError_t e = cudaErrorNotSupported;
    if (fmt == FMT_INT8) e = launch2<FMT_INT8, 1, S2_DENSE_LOCAL>(p, a, w, ldw, es, 1, st);
    else if (fmt == FMT_FP8) e = launch2<FMT_FP8, 1, S2_DENSE_LOCAL>(p, a, w, ldw, es, 1, st);
    else if (fmt == FMT_F8E4C) e = launch2<FMT_F8E4C, 1, S2_DENSE_LOCAL>(p, a, w, ldw, es, 1, st);
    else if (fmt == FMT_F8E5C) e = launch2<FMT_F8E5C, 1, S2_DENSE_LOCAL>(p, a, w, ldw, es, 1, st);
    else if (fmt == FMT_MXFP4) e = launch2<FMT_MXFP4, 1, S2_DENSE_LOCAL>(p, a, w, ldw, es, 1, st);
    if (e != cudaErrorNotSupported) return e;
  }
  if (fmt == FMT_INT8)
    return p.mt == 1   ? launch2<FMT_INT8, 1, S2_DENSE>(p, a, w, ldw, es, 1, st)
           : p.mt == 2 ? launch2<FMT_INT8, 2, S2_DENSE>(p, a, w, ldw, es, 1, st)
                       : launch2<FMT_INT8, 4, S2_DENSE>(p, a, w, ldw, es, 1, st);
  if (fmt == FMT_FP8)
    return p.mt == 1 ? launch2<FMT_FP8, 1, S2_DENSE>(p, a, w, ldw, es, 1, st)
                     : launch2<FMT_FP8, 2, S2_DENSE>(p, a, w, ldw, es, 1, st);
  if (fmt == FMT_BF16)
    return p.mt == 1 ? launch2<FMT_BF16, 1, S2_DENSE>(p, a, w, ldw, es, 1, st)
                     : launch2<FMT_BF16, 2, S2_DENSE>(p, a, w, ldw, es, 1, st);
  if (fmt == FMT_F8E4C)
    return p.mt == 1 ? launch2<FMT_F8E4C, 1, S2_DENSE>(p, a, w, ldw, es, 1, st)
                     : launch2<FMT_F8E4C, 2, S2_DENSE>(p, a, w, ldw, es, 1, st);
  if (fmt == FMT_F8E5C)
    return p.mt == 1 ? launch2<FMT_F8E5C, 1, S2_DENSE>(p, a, w, ldw, es, 1, st)
                     : launch2<FMT_F8E5C, 2, S2_DENSE>(p, a, w, ldw, es, 1, st);
  return p.mt == 1 ? launch2<FMT_MXFP4, 1, S2_DENSE>(p, a, w, ldw, es, 1, st)
                   : launch2<FMT_MXFP4, 2, S2_DENSE>(p, a, w, ldw, es, 1, st);
}

cudaError_t launch_moe2(int kind, const Skinny2Plan& p, const Skinny2Args& a, const uint8_t* w, int64_t ldw,
                        int64_t w_estride, int experts, cudaStream_t st) {
  if (kind == S2_MOE_GU)
    return p.mt == 1 ? launch2<FMT_MXFP4, 1, S2_MOE_GU>(p, a, w, ldw, w_estride, experts, st)
                     : launch2<FMT_MXFP4, 2, S2_MOE_GU>(p, a, w, ldw, w_estride, experts, st);
  return p.mt == 1 ? launch2<FMT_MXFP4, 1, S2_MOE_DN>(p, a, w, ldw, w_estride, experts, st)
                   : launch2<FMT_MXFP4, 2, S2_MOE_DN>(p, a, w, ldw, w_estride, experts, st);
}

}  // namespace ql
