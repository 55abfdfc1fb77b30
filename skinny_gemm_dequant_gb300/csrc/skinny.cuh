// Skinny (M <= 16 tokens) weight-streaming GEMM for INT8, FP8-block and MXFP4 weights.
//
// Dataflow per warp: 16 weight rows x a K range.  Each thread streams 16-byte vectors of two
// rows (g and g+8 of the warp tile) straight from HBM into registers (the weights are used
// once, so they are not staged through shared memory), dequantises them in registers to
// f16 pairs and feeds the warp-level tensor-core MMA m16n8k16 with the weights as the A
// operand (16 rows) and the activations as B (8 tokens per tile).  Within a 64-K chunk the
// K index is permuted so that each thread's 16 contiguous weight bytes are its own MMA
// k-slots; the activations in shared memory are read with the same permutation, so the dot
// products are unchanged (a sum over k does not depend on the order of its terms).
//
// Scales (the scale-folding identity of the Z100 record, §二.2.4: a scale may be applied to
// a partial sum over its block before the reduction):
//   INT8  : f16 products of integers are exact and every 64-K partial (< 2^21) is an exact
//           fp32 integer, converted to int32 and summed exactly; (acc*x_s)*w_s at the end.
//   FP8   : each 64-K chunk lies in one 128x128 block; the chunk's fp32 partial is folded
//           into the accumulator with that block's UE8M0 scale.
//   MXFP4 : the four threads of a quad exchange words (a 4x4 transpose) so that every MMA
//           pair covers exactly one 32-K scale group of its rows; the group's partial is
//           folded with the per-row UE8M0 scale.
// Split-K across CTAs writes fp32/int32 partials to the workspace; the last CTA of a row
// block (atomic ticket) sums them in split order, so results are deterministic.
#pragma once
#include "common.cuh"

namespace ql {

// BF16 and the per-channel FP8 formats (E4M3 / E5M2 codes, fp32 scale per channel or tensor)
// run on the persistent kernel only
enum Fmt { FMT_INT8 = 0, FMT_FP8 = 1, FMT_MXFP4 = 2, FMT_BF16 = 3, FMT_F8E4C = 4, FMT_F8E5C = 5 };
enum Epi { EPI_INT8 = 0, EPI_LINEAR = 1, EPI_GATEUP = 2, EPI_DOWN = 3 };
enum XKind { X_INT8 = 0, X_BF16 = 1 };

constexpr int SK_THREADS = 256;
constexpr int SK_RW = 4;  // row tiles (16 rows each) per CTA
constexpr int SK_KW = 2;  // K slices per CTA
constexpr int SK_ROWS = 16 * SK_RW;

struct SkinnyArgs {
  const uint8_t* w;      // weight rows [rows, ldw] bytes (MoE: expert 0; + e * w_estride)
  int64_t ldw;           // bytes per weight row
  int64_t w_estride;     // bytes between experts (MoE)
  const uint8_t* wsb;    // FP8: UE8M0 grid [ceil(N/bn), lds]; MXFP4: UE8M0 [rows, lds]
  int64_t lds;           // scale row length in bytes
  int64_t s_estride;     // bytes between experts' scales (MoE)
  int block_n, block_k;  // FP8 block sizes
  const float* w_scale;  // INT8 per-channel (len N) or per-tensor (len 1) scales
  int w_scale_len;
  const void* x;         // INT8: int8 [M, ldx]; else bf16 [M, ldx] (MoE down: h [pairs, ldx])
  int64_t ldx;
  const float* x_s;      // INT8 per-token scales [M]
  int M, N, K;           // N = weight rows of one matrix (MoE gate_up: 2I)
  uint16_t* y;           // bf16 output [M, ldy]
  int64_t ldy;
  const uint16_t* bias;
  int32_t* acc_out;      // INT8 debug [M, N]
  int ks, kc;            // K splits and K elements per split
  void* part;            // partials [gridDim.z][ks][16][N] (fp32 or int32 bits)
  unsigned* counters;    // tickets, one per (blockIdx.z, blockIdx.x)
  // MoE
  const int32_t* offsets;   // [E+1]
  const int32_t* pairs;     // [M*topk] sorted by expert
  const int32_t* uniq;      // [E] distinct expert ids, increasing
  const int32_t* nuniq;     // [1]
  int topk, I;
  uint16_t* h;              // gate_up result [M*topk, I]
  uint16_t* h_dbg;          // optional copy
  float act_alpha, act_limit;  // expert activation silu(alpha * min(g, limit)) * clamp(u, +-limit)
  float* o;                 // down result [M*topk, N]
  int pdl;
};

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<FMT_INT8> {
  static constexpr int CHUNK = 64;  // K per quad iteration (4 threads x 16 bytes)
  static constexpr int XPAD = 8;    // f16 elements of row padding (rows 16 B mod 128 apart)
};
template <>
struct FmtTraits<FMT_FP8> {
  static constexpr int CHUNK = 64;
  static constexpr int XPAD = 8;
};
template <>
struct FmtTraits<FMT_MXFP4> {
  static constexpr int CHUNK = 128;  // 4 threads x 16 bytes x 2 codes
  static constexpr int XPAD = 32;    // rows 64 B mod 128 apart
};

__device__ __forceinline__ void quad_transpose(uint32_t (&w)[4], int t) {
  {
    const bool hi = t & 2;
    uint32_t s0 = hi ? w[0] : w[2];
    uint32_t s1 = hi ? w[1] : w[3];
    uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 2);
    uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 2);
    if (hi) { w[0] = r0; w[1] = r1; } else { w[2] = r0; w[3] = r1; }
  }
  {
    const bool odd = t & 1;
    uint32_t s0 = odd ? w[0] : w[1];
    uint32_t s1 = odd ? w[2] : w[3];
    uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 1);
    uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
    if (odd) { w[0] = r0; w[2] = r1; } else { w[1] = r0; w[3] = r1; }
  }
}

// Dynamic shared memory: x tile [16*MT][kc + XPAD] f16, then the K-slice reduction buffer.
template <int FMT, int MT>
__host__ __device__ constexpr size_t skinny_smem_bytes(int kc) {
  return (size_t)8 * MT * (kc + FmtTraits<FMT>::XPAD) * 2 +
         (size_t)(SK_KW - 1) * SK_RW * 32 * 4 * MT * 4 + 64 * 4;
}

template <int FMT, int MT, int EPI>
__global__ void __launch_bounds__(SK_THREADS, 2) skinny_gemm_kernel(const __grid_constant__ SkinnyArgs a) {
  using Tr = FmtTraits<FMT>;
  constexpr int CHUNK = Tr::CHUNK;
  constexpr int U = 4;  // chunks in flight per warp
  constexpr bool kMoE = (EPI == EPI_GATEUP || EPI == EPI_DOWN);
  constexpr bool kInt = (FMT == FMT_INT8);

  extern __shared__ __align__(16) uint8_t smem[];
  const int kc = a.kc;
  const int xstride = kc + Tr::XPAD;  // f16 elements per token row
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  float* red = reinterpret_cast<float*>(smem + (size_t)8 * MT * xstride * 2);
  float* tokscale = red + (SK_KW - 1) * SK_RW * 32 * 4 * MT;  // [16] per-token 2^p
  __shared__ int s_tok[16];       // activation row of each MMA column
  __shared__ int s_pair[16];      // MoE pair index of each column
  __shared__ int s_ntok;
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int rw = warp % SK_RW, kw = warp / SK_RW;

  // -------------------------------------------------------------- work assignment
  const uint8_t* W = a.w;
  const uint8_t* WS = a.wsb;
  int expert = 0;
  if constexpr (kMoE) {
    if (a.pdl) pdl_wait();
    const int slot = blockIdx.z;
    if (slot >= *a.nuniq) return;
    expert = a.uniq[slot];
    W += (int64_t)expert * a.w_estride;
    WS += (int64_t)expert * a.s_estride;
  }
  const int N = a.N, K = a.K;
  int row0;  // first row of this warp's 16-row tile
  if constexpr (EPI == EPI_GATEUP) {
    // CTA covers intermediate [i0, i0+32): warps rw 0,1 -> gate rows, rw 2,3 -> up rows
    const int i0 = blockIdx.x * 32;
    row0 = (rw < 2) ? (i0 + rw * 16) : (a.I + i0 + (rw - 2) * 16);
  } else {
    row0 = blockIdx.x * SK_ROWS + rw * 16;
  }
  const int ra = min(row0 + g, N - 1), rb = min(row0 + g + 8, N - 1);
  const int kbeg = blockIdx.y * kc;
  const int kend = min(K, kbeg + kc);
  const int nchunk = (kend - kbeg + CHUNK - 1) / CHUNK;

  // -------------------------------------------------------------- weight prefetch
  // bytes of one K element: 1 (INT8/FP8) or 1/2 (MXFP4)
  auto wbyte = [&](int k) -> int64_t { return (FMT == FMT_MXFP4) ? (k >> 1) : k; };
  const uint8_t* pa = W + (int64_t)ra * a.ldw;
  const uint8_t* pb = W + (int64_t)rb * a.ldw;
  const int tstep = (FMT == FMT_MXFP4) ? 32 : 16;  // K elements covered by one thread vector
  uint4 wa[U], wb[U];
  auto issue = [&](int slot, int ci) {
    const int c = kbeg + ci * CHUNK + t * tstep;
    if (ci < nchunk && c < kend) {
      wa[slot] = ldg_stream(pa + wbyte(c));
      wb[slot] = ldg_stream(pb + wbyte(c));
    } else {
      wa[slot] = make_uint4(0, 0, 0, 0);
      wb[slot] = make_uint4(0, 0, 0, 0);
    }
  };
#pragma unroll
  for (int u = 0; u < U; ++u) issue(u, kw + u * SK_KW);

  if constexpr (!kMoE) {
    if (a.pdl) pdl_wait();  // activations come from the previous kernel
  }

  // -------------------------------------------------------------- token columns
  if (threadIdx.x < 16) {
    int tok = -1, pr = -1;
    if constexpr (kMoE) {
      const int beg = a.offsets[expert], cnt = a.offsets[expert + 1] - beg;
      if ((int)threadIdx.x < cnt) {
        pr = a.pairs[beg + threadIdx.x];
        tok = (EPI == EPI_GATEUP) ? pr / a.topk : pr;
      }
      if (threadIdx.x == 0) s_ntok = cnt;
    } else {
      if ((int)threadIdx.x < a.M) tok = threadIdx.x;
      if (threadIdx.x == 0) s_ntok = a.M;
    }
    s_tok[threadIdx.x] = tok;
    s_pair[threadIdx.x] = pr;
  }
  __syncthreads();
  const int ntok = s_ntok;

  // -------------------------------------------------------------- stage activations (f16)
  const int ntrow = 8 * MT;
  if constexpr (kInt) {
    // int8 codes -> f16 (exact); 16 codes per thread step
    const int vec_per_row = kc / 16;
    for (int idx = threadIdx.x; idx < ntrow * vec_per_row; idx += SK_THREADS) {
      const int r = idx / vec_per_row, v = idx % vec_per_row;
      const int k = kbeg + v * 16;
      const int tok = s_tok[r];
      uint4 q = make_uint4(0, 0, 0, 0);
      if (tok >= 0 && k < kend)
        q = *reinterpret_cast<const uint4*>(static_cast<const int8_t*>(a.x) + (int64_t)tok * a.ldx + k);
      uint32_t o[8];
      s8x4_to_f16x2x2(q.x, o[0], o[1]);
      s8x4_to_f16x2x2(q.y, o[2], o[3]);
      s8x4_to_f16x2x2(q.z, o[4], o[5]);
      s8x4_to_f16x2x2(q.w, o[6], o[7]);
      uint4* dst = reinterpret_cast<uint4*>(xs + r * xstride + v * 16);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    if (threadIdx.x < 16) tokscale[threadIdx.x] = 1.0f;
  } else {
    // bf16 -> f16 with a per-token power-of-two prescale 2^-p chosen from this slice's
    // amax (scaled amax in [2^14, 2^15)), so f16 neither overflows nor loses the large
    // values' bits; partial sums are multiplied back by 2^p.
    const uint16_t* xb = static_cast<const uint16_t*>(a.x);
    for (int r = warp; r < ntrow; r += SK_THREADS / 32) {
      const int tok = s_tok[r];
      float m = 0.f;
      if (tok >= 0) {
        for (int k = kbeg + lane * 8; k < kend; k += 32 * 8) {
          const uint4 v = *reinterpret_cast<const uint4*>(xb + (int64_t)tok * a.ldx + k);
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            m = fmaxf(m, fabsf(__uint_as_float(wv[i] << 16)));
            m = fmaxf(m, fabsf(__uint_as_float(wv[i] & 0xFFFF0000u)));
          }
        }
      }
      m = warp_max(m);
      if (lane == 0) {
        int p = 0;
        if (m > 0.f) {
          const int ex = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;  // floor(log2 m) for normals
          p = max(ex, -126) - 14;
        }
        p = max(-100, min(100, p));
        tokscale[r] = __uint_as_float((uint32_t)(127 + p) << 23);  // 2^p
      }
    }
    __syncthreads();
    const int vec_per_row = kc / 8;
    for (int idx = threadIdx.x; idx < ntrow * vec_per_row; idx += SK_THREADS) {
      const int r = idx / vec_per_row, v = idx % vec_per_row;
      const int k = kbeg + v * 8;
      const int tok = s_tok[r];
      uint4 o = make_uint4(0, 0, 0, 0);
      if (tok >= 0 && k < kend) {
        const uint4 q = *reinterpret_cast<const uint4*>(xb + (int64_t)tok * a.ldx + k);
        const float inv = 1.0f / tokscale[r];  // exact: power of two
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
        uint32_t ov[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          ov[i] = pack_f16x2(__uint_as_float(wv[i] << 16) * inv, __uint_as_float(wv[i] & 0xFFFF0000u) * inv);
        o = make_uint4(ov[0], ov[1], ov[2], ov[3]);
      }
      *reinterpret_cast<uint4*>(xs + r * xstride + v * 8) = o;
    }
  }
  __syncthreads();

  // -------------------------------------------------------------- main loop
  float blk[MT][4];
  float accf[MT][4];
  int32_t acci[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) { accf[m][i] = 0.f; acci[m][i] = 0; }

  const uint8_t* WSa = nullptr;  // MXFP4 per-row scale rows
  const uint8_t* WSb = nullptr;
  if constexpr (FMT == FMT_MXFP4) {
    WSa = WS + (int64_t)ra * a.lds;
    WSb = WS + (int64_t)rb * a.lds;
  }
  const uint8_t* WSf = nullptr;  // FP8 scale row of this warp's n-block
  if constexpr (FMT == FMT_FP8) WSf = WS + (int64_t)(min(row0, N - 1) / a.block_n) * a.lds;

  auto compute = [&](const uint4 va, const uint4 vb, const int ci) {
    const int cl = ci * CHUNK;  // chunk start relative to kbeg
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) blk[m][i] = 0.f;
    if constexpr (FMT == FMT_MXFP4) {
      uint32_t A[4] = {va.x, va.y, va.z, va.w};
      uint32_t B[4] = {vb.x, vb.y, vb.z, vb.w};
      quad_transpose(A, t);
      quad_transpose(B, t);
      const int kgrp = (kbeg + cl) >> 5;  // first 32-group of the chunk
      uint32_t sa4 = 0, sb4 = 0;
      if (kgrp + 4 <= (K >> 5)) {
        sa4 = ldg_u32(WSa + kgrp);
        sb4 = ldg_u32(WSb + kgrp);
      } else {  // ragged K tail: only the groups below K/32 exist
        for (int q = 0; q < 4 && kgrp + q < (K >> 5); ++q) {
          sa4 |= (uint32_t)WSa[kgrp + q] << (8 * q);
          sb4 |= (uint32_t)WSb[kgrp + q] << (8 * q);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t xf[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + (g + 8 * m) * xstride + cl + 32 * q + 8 * t);
          xf[m][0] = xv.x; xf[m][1] = xv.y; xf[m][2] = xv.z; xf[m][3] = xv.w;
        }
        uint32_t wa[4], wb[4];  // bytes 0..3 of rows g and g+8 as f16 pairs
        e2m1x8_to_f16x2x4(A[q], wa);
        e2m1x8_to_f16x2x4(B[q], wb);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int m = 0; m < MT; ++m)
            mma_f16_16816(blk[m], wa[2 * h], wb[2 * h], wa[2 * h + 1], wb[2 * h + 1], xf[m][2 * h], xf[m][2 * h + 1]);
        const float sa = ue8m0_to_f32(sa4 >> (8 * q));
        const float sb = ue8m0_to_f32(sb4 >> (8 * q));
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          accf[m][0] = fmaf(blk[m][0], sa, accf[m][0]);
          accf[m][1] = fmaf(blk[m][1], sa, accf[m][1]);
          accf[m][2] = fmaf(blk[m][2], sb, accf[m][2]);
          accf[m][3] = fmaf(blk[m][3], sb, accf[m][3]);
          blk[m][0] = blk[m][1] = blk[m][2] = blk[m][3] = 0.f;
        }
      }
    } else {
      const uint32_t A[4] = {va.x, va.y, va.z, va.w};
      const uint32_t B[4] = {vb.x, vb.y, vb.z, vb.w};
      uint32_t xf[MT][8];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const uint4* xp = reinterpret_cast<const uint4*>(xs + (g + 8 * m) * xstride + cl + 16 * t);
        const uint4 x0 = xp[0], x1 = xp[1];
        xf[m][0] = x0.x; xf[m][1] = x0.y; xf[m][2] = x0.z; xf[m][3] = x0.w;
        xf[m][4] = x1.x; xf[m][5] = x1.y; xf[m][6] = x1.z; xf[m][7] = x1.w;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t a0, a1, a2, a3;
        if constexpr (FMT == FMT_INT8) {
          s8x4_to_f16x2x2(A[j], a0, a2);
          s8x4_to_f16x2x2(B[j], a1, a3);
        } else {
          e4m3x4_to_f16x2x2(A[j], a0, a2);
          e4m3x4_to_f16x2x2(B[j], a1, a3);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) mma_f16_16816(blk[m], a0, a1, a2, a3, xf[m][2 * j], xf[m][2 * j + 1]);
      }
      if constexpr (FMT == FMT_INT8) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int i = 0; i < 4; ++i) acci[m][i] += __float2int_rn(blk[m][i]);
      } else {
        const float s = ue8m0_to_f32(WSf[(kbeg + cl) / a.block_k]);
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int i = 0; i < 4; ++i) accf[m][i] = fmaf(blk[m][i], s, accf[m][i]);
      }
    }
  };

  // U chunks stay in flight: chunk (base+u) is consumed from slot u, which is then refilled
  // with chunk (base+u+U); slots are compile-time indices, so the buffers stay in registers.
  for (int base = 0; kw + base * SK_KW < nchunk; base += U) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int ci = kw + (base + u) * SK_KW;
      if (ci < nchunk) {
        const uint4 va = wa[u], vb = wb[u];
        issue(u, ci + U * SK_KW);
        compute(va, vb, ci);
      }
    }
  }
  pdl_launch_dependents();

  // -------------------------------------------------------------- reduce the K slices of the CTA
  // accumulator element i of tile m: row (i < 2 ? g : g + 8), column 2t + (i & 1) + 8m
  float res[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) res[m][i] = kInt ? __int_as_float(acci[m][i]) : accf[m][i];
  if (kw > 0) {
    float* dst = red + ((kw - 1) * SK_RW + rw) * 32 * 4 * MT + lane * 4 * MT;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[m * 4 + i] = res[m][i];
  }
  __syncthreads();
  if (kw == 0) {
#pragma unroll
    for (int s = 1; s < SK_KW; ++s) {
      const float* src = red + ((s - 1) * SK_RW + rw) * 32 * 4 * MT + lane * 4 * MT;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (kInt) res[m][i] = __int_as_float(__float_as_int(res[m][i]) + __float_as_int(src[m * 4 + i]));
          else res[m][i] += src[m * 4 + i];
        }
    }
    if (!kInt) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) res[m][i] *= tokscale[2 * t + (i & 1) + 8 * m];
    }
  }

  // -------------------------------------------------------------- split-K across CTAs
  if (a.ks > 1) {
    if (kw == 0) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = row0 + g + (i >= 2 ? 8 : 0);
          const int col = 2 * t + (i & 1) + 8 * m;
          if (row < N && col < 16)
            reinterpret_cast<float*>(a.part)[(((int64_t)blockIdx.z * a.ks + blockIdx.y) * 16 + col) * N + row] = res[m][i];
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned prev = atomicAdd(&a.counters[blockIdx.z * gridDim.x + blockIdx.x], 1u);
      s_last = (prev == (unsigned)a.ks - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (kw == 0) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = row0 + g + (i >= 2 ? 8 : 0);
          const int col = 2 * t + (i & 1) + 8 * m;
          float s = 0.f;
          int si = 0;
          if (row < N && col < 16) {
            for (int sp = 0; sp < a.ks; ++sp) {
              const float v = __ldcg(reinterpret_cast<const float*>(a.part) +
                                     (((int64_t)blockIdx.z * a.ks + sp) * 16 + col) * N + row);
              if (kInt) si += __float_as_int(v); else s += v;
            }
          }
          res[m][i] = kInt ? __int_as_float(si) : s;
        }
    }
    if (threadIdx.x == 0) a.counters[blockIdx.z * gridDim.x + blockIdx.x] = 0;  // leave the ticket ready for the next call
  }

  // -------------------------------------------------------------- epilogues
  if constexpr (EPI == EPI_GATEUP) {
    // up-row warps hand their results to the gate-row warps of the same intermediate rows
    float* xch = red;  // reuse: [2][32][4*MT]
    __syncthreads();
    if (kw == 0 && rw >= 2) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) xch[((rw - 2) * 32 + lane) * 4 * MT + m * 4 + i] = res[m][i];
    }
    __syncthreads();
    if (kw == 0 && rw < 2) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int irow = row0 + g + (i >= 2 ? 8 : 0);  // intermediate index
          const int col = 2 * t + (i & 1) + 8 * m;
          if (col < ntok && irow < a.I) {
            const float gv = res[m][i];
            const float uv = xch[(rw * 32 + lane) * 4 * MT + m * 4 + i];
            const uint16_t hb = f32_to_bf16_rn(swiglu_f32(gv, uv, a.act_alpha, a.act_limit));
            const int pr = s_pair[col];
            a.h[(int64_t)pr * a.I + irow] = hb;
            if (a.h_dbg) a.h_dbg[(int64_t)pr * a.I + irow] = hb;
          }
        }
    }
  } else if (kw == 0) {
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = row0 + g + (i >= 2 ? 8 : 0);
        const int col = 2 * t + (i & 1) + 8 * m;
        if (row >= N || col >= ntok) continue;
        if constexpr (EPI == EPI_DOWN) {
          a.o[(int64_t)s_pair[col] * N + row] = res[m][i];
        } else if constexpr (EPI == EPI_INT8) {
          const int32_t acc = __float_as_int(res[m][i]);
          if (a.acc_out) a.acc_out[(int64_t)col * N + row] = acc;
          const float ws = a.w_scale[a.w_scale_len > 1 ? row : 0];
          float v = __fmul_rn(__fmul_rn((float)acc, a.x_s[col]), ws);
          uint16_t yb = f32_to_bf16_rn(v);
          if (a.bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + bf16_bits_to_f32(a.bias[row]));
          a.y[(int64_t)col * a.ldy + row] = yb;
        } else {
          uint16_t yb = f32_to_bf16_rn(res[m][i]);
          if (a.bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + bf16_bits_to_f32(a.bias[row]));
          a.y[(int64_t)col * a.ldy + row] = yb;
        }
      }
  }
}

}  // namespace ql
