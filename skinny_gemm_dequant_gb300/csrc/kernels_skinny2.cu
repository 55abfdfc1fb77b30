// Launch of the persistent TMA-fed skinny GEMM (skinny2.cuh) and its activation prologues.
//
// Prologues (one CTA per padded token row, run once per call, chained to the GEMM by
// programmatic dependent launch so the GEMM's weight loads start while they run):
//  * INT8: dynamic per-token quantisation ([Z100] §二.2.1): x_s = amax/127 and
//    x_q = clamp(rint(x/x_s)) with IEEE divisions; the GEMM reads the codes as an exact f16
//    image [rows][K] (rows past M are zero).
//  * bf16 activations (FP8 block and MXFP4 weights): an f16 image scaled per token by 2^-p,
//    p chosen from the token's amax so the image stays inside the f16 range with its full
//    significand; the GEMM multiplies results back by 2^p.
#include <atomic>

#include <cudaTypedefs.h>

#include "internal.h"
#include "skinny2.cuh"

namespace ql {

__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float u = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    u = warp_max(u);
    if (threadIdx.x == 0) red[0] = u;
  }
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

constexpr int kProThreads = 512;
constexpr int kProVec = 8;  // 16-byte vectors held per thread: one pass for K <= 512*8*8

__device__ __forceinline__ float bf16x2_absmax(uint32_t w) {
  return fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xFFFF0000u)));
}

// INT8: x_s = amax/127, codes rint(x/x_s) clamped to +-127 (IEEE divisions), written as an
// exact f16 image; one CTA per padded token row, the row read once into registers
__global__ void __launch_bounds__(kProThreads) prologue_int8_kernel(const uint16_t* __restrict__ x, int M, int K,
                                                                    int64_t ldx, uint16_t* __restrict__ x16,
                                                                    float* __restrict__ xs, int8_t* xq_dbg,
                                                                    float* xs_dbg) {
  pdl_launch_dependents();
  __shared__ float red[kProThreads / 32];
  const int m = blockIdx.x;
  uint16_t* out = x16 + ((int64_t)blockIdx.y * gridDim.x + m) * K;  // copy blockIdx.y
  const bool first = blockIdx.y == 0;
  const int nvec = K / 8;
  if (m >= M) {
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) *reinterpret_cast<uint4*>(out + 8 * v) = make_uint4(0, 0, 0, 0);
    return;
  }
  pdl_wait();  // the activations may come from the kernel before this call
  const uint16_t* xr = x + (int64_t)m * ldx;
  const bool one_pass = nvec <= kProVec * (int)blockDim.x;
  uint4 v[kProVec];
  float amax = 0.f;
  if (one_pass) {
#pragma unroll
    for (int j = 0; j < kProVec; ++j) {
      const int i = threadIdx.x + j * blockDim.x;
      v[j] = i < nvec ? *reinterpret_cast<const uint4*>(xr + 8 * i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kProVec; ++j)
      amax = fmaxf(amax, fmaxf(fmaxf(bf16x2_absmax(v[j].x), bf16x2_absmax(v[j].y)),
                               fmaxf(bf16x2_absmax(v[j].z), bf16x2_absmax(v[j].w))));
  } else {
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
      const uint4 u = *reinterpret_cast<const uint4*>(xr + 8 * i);
      amax = fmaxf(amax, fmaxf(fmaxf(bf16x2_absmax(u.x), bf16x2_absmax(u.y)), fmaxf(bf16x2_absmax(u.z), bf16x2_absmax(u.w))));
    }
  }
  amax = block_max(amax, red);
  const float s = __fdiv_rn(amax, 127.0f);
  auto quant = [&](const uint4 u, int i) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float qv[8];
    uint32_t qb[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float xv = (e & 1) ? __uint_as_float(w[e >> 1] & 0xFFFF0000u) : __uint_as_float(w[e >> 1] << 16);
      float q = 0.f;
      if (s > 0.f) q = fminf(fmaxf(rintf(__fdiv_rn(xv, s)), -127.f), 127.f);
      qv[e] = q;
      qb[e >> 2] |= ((uint32_t)((int)q & 0xFF)) << (8 * (e & 3));
    }
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = pack_f16x2(qv[2 * j], qv[2 * j + 1]);  // exact: |q| <= 127
    *reinterpret_cast<uint4*>(out + 8 * i) = make_uint4(h[0], h[1], h[2], h[3]);
    if (xq_dbg && first) *reinterpret_cast<uint2*>(xq_dbg + (int64_t)m * K + 8 * i) = make_uint2(qb[0], qb[1]);
  };
  if (one_pass) {
#pragma unroll
    for (int j = 0; j < kProVec; ++j) {
      const int i = threadIdx.x + j * blockDim.x;
      if (i < nvec) quant(v[j], i);
    }
  } else {
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) quant(*reinterpret_cast<const uint4*>(xr + 8 * i), i);
  }
  if (threadIdx.x == 0 && first) {
    xs[m] = s;
    if (xs_dbg) xs_dbg[m] = s;
  }
}

// bf16 activations: f16 image scaled by 2^-p per token (scaled amax in [2^14, 2^15))
__global__ void __launch_bounds__(kProThreads) prologue_bf16_kernel(const uint16_t* __restrict__ x, int M, int K,
                                                                    int64_t ldx, uint16_t* __restrict__ x16,
                                                                    float* __restrict__ tokscale) {
  pdl_launch_dependents();
  __shared__ float red[kProThreads / 32];
  const int m = blockIdx.x;
  uint16_t* out = x16 + ((int64_t)blockIdx.y * gridDim.x + m) * K;  // copy blockIdx.y
  const bool first = blockIdx.y == 0;
  const int nvec = K / 8;
  if (m >= M) {
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) *reinterpret_cast<uint4*>(out + 8 * v) = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0 && first) tokscale[m] = 1.f;
    return;
  }
  pdl_wait();
  const uint16_t* xr = x + (int64_t)m * ldx;
  const bool one_pass = nvec <= kProVec * (int)blockDim.x;
  uint4 v[kProVec];
  float amax = 0.f;
  if (one_pass) {
#pragma unroll
    for (int j = 0; j < kProVec; ++j) {
      const int i = threadIdx.x + j * blockDim.x;
      v[j] = i < nvec ? *reinterpret_cast<const uint4*>(xr + 8 * i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kProVec; ++j)
      amax = fmaxf(amax, fmaxf(fmaxf(bf16x2_absmax(v[j].x), bf16x2_absmax(v[j].y)),
                               fmaxf(bf16x2_absmax(v[j].z), bf16x2_absmax(v[j].w))));
  } else {
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
      const uint4 u = *reinterpret_cast<const uint4*>(xr + 8 * i);
      amax = fmaxf(amax, fmaxf(fmaxf(bf16x2_absmax(u.x), bf16x2_absmax(u.y)), fmaxf(bf16x2_absmax(u.z), bf16x2_absmax(u.w))));
    }
  }
  amax = block_max(amax, red);
  int p = 0;
  if (amax > 0.f) p = max((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127, -126) - 14;
  p = max(-100, min(100, p));
  const float inv = __uint_as_float((uint32_t)(127 - p) << 23);  // 2^-p
  auto conv = [&](const uint4 u, int i) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      h[j] = pack_f16x2(__uint_as_float(w[j] << 16) * inv, __uint_as_float(w[j] & 0xFFFF0000u) * inv);
    *reinterpret_cast<uint4*>(out + 8 * i) = make_uint4(h[0], h[1], h[2], h[3]);
  };
  if (one_pass) {
#pragma unroll
    for (int j = 0; j < kProVec; ++j) {
      const int i = threadIdx.x + j * blockDim.x;
      if (i < nvec) conv(v[j], i);
    }
  } else {
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) conv(*reinterpret_cast<const uint4*>(xr + 8 * i), i);
  }
  if (threadIdx.x == 0 && first) tokscale[m] = __uint_as_float((uint32_t)(127 + p) << 23);
}

cudaError_t launch_prologue_int8(const uint16_t* x, int M, int Mp, int K, int64_t ldx, uint16_t* x16, float* xs,
                                 int8_t* xq_dbg, float* xs_dbg, cudaStream_t st) {
  prologue_int8_kernel<<<dim3(Mp, kXCopies), kProThreads, 0, st>>>(x, M, K, ldx, x16, xs, xq_dbg, xs_dbg);
  return cudaGetLastError();
}

cudaError_t launch_prologue_bf16(const uint16_t* x, int M, int Mp, int K, int64_t ldx, uint16_t* x16, float* tokscale,
                                 cudaStream_t st) {
  prologue_bf16_kernel<<<dim3(Mp, kXCopies), kProThreads, 0, st>>>(x, M, K, ldx, x16, tokscale);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ plan + launch

Skinny2Plan skinny2_plan(int fmt, int64_t M, int64_t N, int64_t K, int block_n) {
  Skinny2Plan p;
  p.mt = M <= 8 ? 1 : 2;
  p.mp = 8 * p.mt;
  const int kpu = fmt == FMT_MXFP4 ? 256 : 128;
  p.nb = (N + S2_ROWS - 1) / S2_ROWS;
  p.nk = (int)((K + kpu - 1) / kpu);
  p.total = p.nb * p.nk;
  const int64_t sms = kNumSMs;  // fixed here so the workspace query and the launch agree
  p.grid = (int)(p.total < sms ? p.total : sms);
  // partial slots: the most CTAs any row block is spread over
  int maxseg = 1;
  for (int64_t rb = 0; rb < p.nb; ++rb) {
    const int64_t a = rb * p.nk, b = rb * p.nk + p.nk - 1;
    const int64_t ca = ((a + 1) * p.grid + p.total - 1) / p.total - 1;
    const int64_t cb = ((b + 1) * p.grid + p.total - 1) / p.total - 1;
    if (cb - ca + 1 > maxseg) maxseg = (int)(cb - ca + 1);
  }
  p.maxseg = maxseg;
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

template <int FMT, int MT>
static cudaError_t launch2(const Skinny2Plan& p, Skinny2Args a, const uint8_t* w, int64_t ldw, const uint16_t* x16,
                           cudaStream_t st) {
  constexpr uint32_t STAGE = s2_stage_bytes<FMT, MT>();
  const size_t fixed = 1024 + s2_xchg_bytes<MT>() + p.fp8_scale_bytes + 256;
  const int optin = 227 * 1024;
  int S = (int)((optin - fixed - 64) / (STAGE + 16));
  if (S > 12) S = 12;
  a.stages = S;
  a.nk = p.nk;
  a.total = p.total;
  a.maxseg = p.maxseg;
  const size_t smem = 1024 + (size_t)S * STAGE + (size_t)S * 16 + s2_xchg_bytes<MT>() + p.fp8_scale_bytes;
  CUtensorMap tw, tx;
  const uint64_t kbytes = FMT == FMT_MXFP4 ? (uint64_t)a.K / 2 : (uint64_t)a.K;
  if (!map2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, kbytes, (uint64_t)a.N, (uint64_t)ldw, S2_WB, S2_ROWS))
    return cudaErrorInvalidValue;
  a.xcopies = kXCopies;
  if (!map2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16, (uint64_t)a.K, (uint64_t)(8 * MT * kXCopies), (uint64_t)a.K * 2,
             64, 8 * MT))
    return cudaErrorInvalidValue;
  auto kfn = skinny2_kernel<FMT, MT>;
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
  return cudaLaunchKernelEx(&cfg, kfn, tw, tx, a);
}

cudaError_t launch_skinny2(int fmt, const Skinny2Plan& p, const Skinny2Args& a, const uint8_t* w, int64_t ldw,
                           const uint16_t* x16, cudaStream_t st) {
  if (fmt == FMT_INT8) return p.mt == 1 ? launch2<FMT_INT8, 1>(p, a, w, ldw, x16, st) : launch2<FMT_INT8, 2>(p, a, w, ldw, x16, st);
  if (fmt == FMT_FP8) return p.mt == 1 ? launch2<FMT_FP8, 1>(p, a, w, ldw, x16, st) : launch2<FMT_FP8, 2>(p, a, w, ldw, x16, st);
  return p.mt == 1 ? launch2<FMT_MXFP4, 1>(p, a, w, ldw, x16, st) : launch2<FMT_MXFP4, 2>(p, a, w, ldw, x16, st);
}

}  // namespace ql
