// INT8 W8A8 GEMM for M = 17..256 tokens on the 5th-generation tensor cores (tcgen05).
//
// Formula ([Z100] §二.2.1, INT8 W8A8 with dynamic per-token activation quantisation, and the
// epilogue order of §二.2):
//   x_s[m] = max_k |x[m,k]| / 127,  x_q[m,k] = rint(x[m,k] / x_s[m]) clamped to [-127, 127]
//   acc[m,n] = sum_k x_q[m,k] w[n,k]   (exact, int32)
//   y[m,n] = bf16((acc * x_s[m]) * w_s[n])  (+ bias, added after the cast)
//
// sm_103a has no integer tcgen05 MMA.  Every int8 value is exact in f16 and every product of two
// is exact in fp32, so the contraction runs as kind::f16 with fp32 accumulation in tensor memory.
// fp32 holds the integers below 2^24 exactly, and a group of 512 K adds at most
// 512 * 127 * 127 < 2^23 to an output, so the MMAs accumulate one 512-K group at a time into one
// of two tensor-memory buffers while drain warps move the other buffer into int32 registers.
//
// Mapping (swap-AB, as the block-scaled GEMM): the MMA's A operand is a 128-row weight tile, the
// tokens (16..128 per CTA) are its N dimension.  Roles in a CTA of 16 warps:
//   warp 0      : TMA producer: int8 weight tile 128 x 64 K and the f16 activation-code tile;
//   warp 1      : tensor-memory allocation and the single MMA-issuing thread;
//   warps 4..7  : widen the int8 weight tile to the 128-byte-swizzled f16 tile the MMA reads;
//   warps 8..15 : drain each finished 512-K group to int32 (two warps per tensor-memory lane
//                 quadrant, half of the token columns each), then the epilogue.
// Split K: when the 128-row x token tiles alone would leave most SMs idle (fewer than half the
// SMs), blockIdx.z splits K into ks ranges of whole 512-K groups.  Each CTA stores its int32
// sums in its own slot of the workspace and counts in on the tile's ticket; the CTA that completes
// the count adds the ks slots (exact integers: the order does not matter) and runs the epilogue.
// Every mbarrier wait is bounded; a wait that runs out raises QL_DEV_TIMEOUT in the status word,
// the other roles stop, copies and MMAs still in flight are waited for, and tensor memory is
// freed before the CTA exits.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <mutex>

#include "gemm_i8_tcgen05.h"
#include "internal.h"
#include "tc_ptx.cuh"

namespace ql {
namespace tc {

constexpr int kI8Threads = 512;
constexpr int kI8BlockK = 64;          // K per stage: one 128-byte row of the f16 tile
constexpr int kI8GroupStages = 8;      // stages per accumulation group (512 K)
constexpr uint32_t kI8TmemCols = 256;  // two accumulators of up to 128 token columns
constexpr uint32_t kI8A8Bytes = 128 * kI8BlockK;       // int8 weight tile (8 KB)
constexpr uint32_t kI8A16Bytes = 128 * kI8BlockK * 2;  // f16 weight tile (16 KB)
constexpr uint32_t kI8DrainLimit = 1u << 22;

struct I8Params {
  int M, N, K, nk, tt, stages;
  int ks;               // K splits (gridDim.z)
  int32_t* part;        // [ks][M][N] int32 partial sums (ks > 1)
  unsigned* tickets;    // [tiles] arrival counts (ks > 1); zero between calls
  const float* w_s;
  int w_s_len;
  const float* x_s;
  const uint16_t* bias;
  uint16_t* y;
  int64_t ldy;
  int32_t* acc_out;
  uint32_t* status;
  uint32_t wait_limit;
  int tma_y;  // 1: the output tile leaves through shared memory and one TMA store (tmY)
};

// ------------------------------------------------------------------ activation quantisation
// One CTA per token: amax, x_s = amax / 127 and the codes rint(x / x_s) (IEEE fp32 divisions),
// written as exact f16 values into the image [M][kpad] (zeros past K) that the GEMM reads.
__global__ void __launch_bounds__(256) quant_i8_image_kernel(const uint16_t* __restrict__ x, int K, int64_t ldx,
                                                             int kpad, uint16_t* __restrict__ img,
                                                             float* __restrict__ xs, int8_t* xq_dbg, float* xs_dbg,
                                                             const float* __restrict__ amax_in) {
  pdl_launch_dependents();  // the GEMM may start and prefetch its weights
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
  amax = fmaxf(fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3])),
               fmaxf(fmaxf(s_red[4], s_red[5]), fmaxf(s_red[6], s_red[7])));
  if (amax_in) amax = amax_in[m];  // a K shard: the whole row's amax, from the caller
  const float s = __fdiv_rn(amax, 127.0f);
  uint16_t* ir = img + (int64_t)m * kpad;
  for (int k = threadIdx.x * 8; k < kpad; k += blockDim.x * 8) {
    uint32_t h[4] = {0u, 0u, 0u, 0u};
    uint32_t packed[2] = {0u, 0u};
    if (k < K) {  // K % 16 == 0: a group of 8 is either inside K or past it
      const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float qv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float xv = (i & 1) ? __uint_as_float(w[i >> 1] & 0xFFFF0000u) : __uint_as_float(w[i >> 1] << 16);
        float q = 0.f;
        if (s > 0.f) q = fminf(fmaxf(rintf(__fdiv_rn(xv, s)), -127.f), 127.f);
        qv[i] = q;
        packed[i >> 2] |= ((uint32_t)((int)q & 0xFF)) << (8 * (i & 3));
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = pack_f16x2(qv[2 * j], qv[2 * j + 1]);  // exact: |q| <= 127
      if (xq_dbg) *reinterpret_cast<uint2*>(xq_dbg + (int64_t)m * K + k) = make_uint2(packed[0], packed[1]);
    }
    *reinterpret_cast<uint4*>(ir + k) = make_uint4(h[0], h[1], h[2], h[3]);
  }
  if (threadIdx.x == 0) {
    xs[m] = s;
    if (xs_dbg) xs_dbg[m] = s;
  }
}

// ------------------------------------------------------------------ the GEMM
// Shared memory per stage: int8 weight tile [128][64] (plain rows) | f16 weight tile [128][64]
// (128-byte swizzle) | f16 activation tile [tt][64] (128-byte swizzle), every part 1 KB aligned.
// kSplit: K split over blockIdx.z (p.ks > 1); the unsplit kernel keeps the whole K and no slots
template <bool kSplit>
__global__ void __launch_bounds__(kI8Threads, 1)
    i8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmY, const __grid_constant__ I8Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  const uint32_t b_bytes = (uint32_t)p.tt * kI8BlockK * 2;
  const uint32_t stage = kI8A8Bytes + kI8A16Bytes + b_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * stage);
  uint64_t* tma_full = bars;           // [S] TMA bytes landed
  uint64_t* conv_full = bars + S;      // [S] f16 weight tile written (4 converter warps)
  uint64_t* empty = bars + 2 * S;      // [S] the stage's MMAs have finished (commit)
  uint64_t* acc_full = bars + 3 * S;   // [2] an accumulation group is complete (commit)
  uint64_t* acc_empty = bars + 3 * S + 2;  // [2] the drain warps have read a buffer (8 warps)
  uint64_t* done = bars + 3 * S + 4;   // every MMA has finished (abort path)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_last;
  __shared__ float s_xs[128];  // the token tile's x_s, for the epilogue

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * 128;
  const int t0 = blockIdx.y * p.tt;
  // this CTA's K range: groups [g0, g1) of the call's 512-K groups, stages [kt0, kt0 + nk)
  const int groups_all = (p.nk + kI8GroupStages - 1) / kI8GroupStages;
  const int kz = kSplit ? (int)blockIdx.z : 0;
  const int g0 = (int)((int64_t)kz * groups_all / p.ks), g1 = (int)((int64_t)(kz + 1) * groups_all / p.ks);
  const int kt0 = kSplit ? g0 * kI8GroupStages : 0;
  const int nk = kSplit ? min(g1 * kI8GroupStages, p.nk) - kt0 : p.nk;
  const int ngroups = (nk + kI8GroupStages - 1) / kI8GroupStages;
  const uint32_t lim = p.wait_limit;
  volatile int* abort = &s_abort;
  auto stage_ptr = [&](int s) { return smem + (size_t)s * stage; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&tma_full[s], 1);
      mbar_init(&conv_full[s], 4);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    s_abort = 0;
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kI8TmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  auto fail = [&]() {
    atomicOr(p.status, (uint32_t)QL_DEV_TIMEOUT);
    *abort = 1;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- TMA producer
      const int pre = nk < S ? nk : S;
      for (int kt = 0; kt < pre; ++kt) {  // weights do not depend on the previous kernel
        mbar_arrive_expect_tx(&tma_full[kt], kI8A8Bytes + b_bytes);
        tma_load_2d(stage_ptr(kt), &tmA, (kt0 + kt) * kI8BlockK, n0, &tma_full[kt]);
      }
      pdl_wait();  // activation codes come from the quantisation kernel
      for (int kt = 0; kt < pre; ++kt)
        tma_load_2d(stage_ptr(kt) + kI8A8Bytes + kI8A16Bytes, &tmB, (kt0 + kt) * kI8BlockK, t0, &tma_full[kt]);
      int issued = pre;
      // slot and phase kept incrementally: one thread runs this loop, so its instruction count
      // per stage paces the ring (no divisions by the runtime stage count)
      int s = pre == S ? 0 : pre;
      uint32_t ph = 0;  // parity of the slot's previous use
      for (int kt = pre; kt < nk; ++kt) {
        if (!mbar_wait(&empty[s], ph, lim, abort)) {
          fail();
          break;
        }
        mbar_arrive_expect_tx(&tma_full[s], kI8A8Bytes + b_bytes);
        tma_load_2d(stage_ptr(s), &tmA, (kt0 + kt) * kI8BlockK, n0, &tma_full[s]);
        tma_load_2d(stage_ptr(s) + kI8A8Bytes + kI8A16Bytes, &tmB, (kt0 + kt) * kI8BlockK, t0, &tma_full[s]);
        issued = kt + 1;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (*abort) {
        // no copy may land after the CTA exits: wait for the last load of every stage
        for (int kt = issued - S < 0 ? 0 : issued - S; kt < issued; ++kt)
          mbar_wait(&tma_full[kt % S], (uint32_t)(kt / S) & 1, kI8DrainLimit, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      // descriptors built once and advanced by constants (the start-address field is address / 16)
      const uint32_t idesc = idesc_f16((uint32_t)p.tt);
      const uint64_t a_desc0 = smem_desc_sw128(smem_u32(smem + kI8A8Bytes));
      const uint64_t b_desc0 = smem_desc_sw128(smem_u32(smem + kI8A8Bytes + kI8A16Bytes));
      const uint32_t step = stage >> 4;
      // slot, parity and descriptor offset kept incrementally: this thread's instructions per
      // stage pace the tensor core (a division by the runtime stage count cost ~10 % of a call)
      int s = 0;
      uint32_t par = 0;
      uint64_t doff = 0;
      uint32_t ready = 0;  // bits 0 / 1: this stage's TMA / conversion barriers already seen complete
      for (int kt = 0; kt < nk; ++kt) {
        const int g = kt / kI8GroupStages;
        const bool first = kt % kI8GroupStages == 0;
        const uint32_t buf = tmem + (uint32_t)(g & 1) * 128u;
        // a group reuses the buffer of group g - 2 once the drain warps have read it
        if (first && g >= 2 && !mbar_wait(&acc_empty[g & 1], (uint32_t)((g >> 1) - 1) & 1, lim, abort)) {
          fail();
          break;
        }
        if ((!(ready & 1) && !mbar_wait(&tma_full[s], par, lim, abort)) ||
            (!(ready & 2) && !mbar_wait(&conv_full[s], par, lim, abort))) {
          fail();
          break;
        }
        tc_fence_after();
        const uint64_t ad = a_desc0 + doff, bd = b_desc0 + doff;
        // the next stage's slot and parity, whose barriers are tested while these MMAs issue
        const int sn = s + 1 == S ? 0 : s + 1;
        const uint32_t pn = s + 1 == S ? par ^ 1u : par;
        ready = mma4_f16_test2(buf, ad, bd, idesc, first ? 0u : 1u, smem_u32(&tma_full[sn]), smem_u32(&conv_full[sn]), pn);
        tc_commit(&empty[s]);
        if (kt % kI8GroupStages == kI8GroupStages - 1 || kt == nk - 1) tc_commit(&acc_full[g & 1]);
        doff += step;
        if (++s == S) {
          s = 0;
          par ^= 1u;
          doff = 0;
        }
      }
      tc_commit(done);
      if (*abort) mbar_wait(done, 0, kI8DrainLimit, nullptr);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ int8 -> f16 weight tile
    // each warp widens 32 rows per stage, 8 rows per pass: lane = (row within the pass, 16-byte
    // chunk); the f16 row is 128 bytes, chunk j of row r stored at chunk j ^ (r & 7)
    const int cw = warp - 4;
    int s = 0;
    uint32_t par = 0;
    for (int kt = 0; kt < nk; ++kt) {
      int got = 0;
      if (lane == 0) got = mbar_wait(&tma_full[s], par, lim, abort);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) fail();
        break;
      }
      const uint32_t a8 = smem_u32(stage_ptr(s)), a16 = a8 + kI8A8Bytes;
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {
        const int r = cw * 32 + pass * 8 + (lane >> 2), c = lane & 3;
        uint32_t w0, w1, w2, w3;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                     : "r"(a8 + (uint32_t)(r * kI8BlockK + c * 16)));
        uint32_t h[8];
        s8x4_to_f16x2x2(w0, h[0], h[1]);
        s8x4_to_f16x2x2(w1, h[2], h[3]);
        s8x4_to_f16x2x2(w2, h[4], h[5]);
        s8x4_to_f16x2x2(w3, h[6], h[7]);
        const uint32_t row = a16 + (uint32_t)(r * 128);
        const uint32_t c0 = (uint32_t)((2 * c) ^ (r & 7)), c1 = (uint32_t)((2 * c + 1) ^ (r & 7));
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(row + c0 * 16), "r"(h[0]), "r"(h[1]), "r"(h[2]),
                     "r"(h[3])
                     : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(row + c1 * 16), "r"(h[4]), "r"(h[5]), "r"(h[6]),
                     "r"(h[7])
                     : "memory");
      }
      // generic-proxy writes -> tensor-core (async-proxy) reads
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv_full[s]);
      if (++s == S) {
        s = 0;
        par ^= 1u;
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ drain + epilogue
    const int q = warp & 3;          // tensor-memory lane quadrant
    const int hcol = (warp - 8) >> 2;  // which half of the token columns
    const int half = p.tt / 2;       // 8..64 columns, a multiple of 8
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    int32_t sum[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) sum[i] = 0;
    bool ok = true;
    for (int g = 0; g < ngroups; ++g) {
      int got = 0;
      if (lane == 0) got = mbar_wait(&acc_full[g & 1], (uint32_t)(g >> 1) & 1, lim, abort);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) fail();
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t col0 = (uint32_t)(g & 1) * 128u + (uint32_t)(hcol * half);
      // two rounds of up to 32 columns: loads, one wait, then the exact conversions
#pragma unroll
      for (int rnd = 0; rnd < 2; ++rnd) {
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < 32; c += 8)
          if (rnd * 32 + c < half) {
            uint32_t r8[8];
            tmem_ld_x8(tmem + lane_base + col0 + (uint32_t)(rnd * 32 + c), r8);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[c + i] = r8[i];
          }
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (rnd * 32 + c < half) sum[rnd * 32 + c] += __float2int_rn(__uint_as_float(v[c]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[g & 1]);
    }
    const int n = n0 + 32 * q + lane;
    if constexpr (kSplit) {
      // split K: store this CTA's sums, count in, and let the CTA completing the count add all.
      // Every drain warp reaches both barriers, also after a timeout (its sums are then not
      // stored; the status word already reports the failure).
      int32_t* slot = p.part + (int64_t)kz * p.M * p.N;
      if (ok && n < p.N) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int t = t0 + hcol * half + c;
          if (c < half && t < p.M) slot[(int64_t)t * p.N + n] = sum[c];
        }
      }
      __threadfence();
      asm volatile("bar.sync 1, 256;" ::: "memory");  // the eight drain warps
      unsigned* ticket = p.tickets + blockIdx.y * gridDim.x + blockIdx.x;
      if (warp == 8 && lane == 0) s_last = atomicAdd(ticket, 1u) == (unsigned)(p.ks - 1);
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const bool last = s_last != 0;
      if (last) {
        __threadfence();  // the other slots were fenced before their counts
        if (ok && n < p.N) {
          // every slot from L2, this CTA's own included (stored and fenced above), 32 loads in
          // flight at a time (integer sums: any order is exact); the loads of one output at a
          // time took ~33 us at 5120x17408
#pragma unroll
          for (int c = 0; c < 64; ++c) sum[c] = 0;
          const int32_t* base = p.part + (int64_t)(t0 + hcol * half) * p.N + n;
          for (int z = 0; z < p.ks; ++z) {
            const int32_t* slot_z = base + (int64_t)z * p.M * p.N;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {  // 32 loads in flight at a time
              int32_t v[32];
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const int cc = 32 * hb + c;
                v[c] = (cc < half && t0 + hcol * half + cc < p.M) ? __ldcg(slot_z + (int64_t)cc * p.N) : 0;
              }
#pragma unroll
              for (int c = 0; c < 32; ++c) sum[32 * hb + c] += v[c];
            }
          }
        }
        if (warp == 8 && lane == 0) *ticket = 0;  // every split has counted in: ready for the next call
      }
      ok = ok && last;
    }
    // the tile's x_s into shared memory once, by every drain warp (also after a timeout: all of
    // them reach the barrier): read from global memory inside the output loop, each value waited
    // behind the previous outputs' stores, the loop took ~6 us
    pdl_wait();  // x_s comes from the quantisation kernel
    {
      const int i = threadIdx.x - 256;  // drain threads are 256..511
      if (i < p.tt) s_xs[i] = t0 + i < p.M ? p.x_s[t0 + i] : 0.f;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");  // the eight drain warps
    // with a TMA store, the tile [tt tokens][128 rows] of bf16 goes to shared memory first: the
    // stage ring is idle once the last group has drained (its loads were all consumed)
    uint16_t* tile = reinterpret_cast<uint16_t*>(smem);
    if (ok) {
      if (n < p.N || p.tma_y) {
        const float ws = (p.w_s && n < p.N) ? p.w_s[p.w_s_len > 1 ? n : 0] : 0.f;
        const float bias = (p.bias && n < p.N) ? bf16_bits_to_f32(p.bias[n]) : 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int tl = hcol * half + c, t = t0 + tl;
          if (c < half && t < p.M) {
            const int32_t a = sum[c];
            if (p.acc_out && n < p.N) p.acc_out[(int64_t)t * p.N + n] = a;
            if (!p.y) continue;  // a K shard: the int32 sums are the result
            uint16_t yb = f32_to_bf16_rn(__fmul_rn(__fmul_rn((float)a, s_xs[tl]), ws));
            if (p.bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + bias);
            if (p.tma_y)
              tile[tl * 128 + 32 * q + lane] = yb;
            else
              p.y[(int64_t)t * p.ldy + n] = yb;
          }
        }
      }
    }
    if (p.tma_y) {
      // every drain warp reaches the barrier; the store goes out only from a CTA holding the
      // finished sums (with split K: the one that added the splits) and without a timeout
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> TMA reads
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (threadIdx.x == 256 && (!kSplit || s_last) && !*abort) {
        tma_store_2d(&tmY, smem_u32(tile), n0, t0);
        bulk_commit_and_wait_all();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kI8TmemCols);
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 i8_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(q);
  });
  return fn;
}

static bool i8_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  auto fn = i8_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) fprintf(stderr, "qlinear: cuTensorMapEncodeTiled failed (%d)\n", (int)r);
  return r == CUDA_SUCCESS;
}

int64_t i8_kpad(int64_t K) { return (K + kI8BlockK - 1) / kI8BlockK * kI8BlockK; }

size_t i8_image_bytes(int64_t M, int64_t K) { return (size_t)M * i8_kpad(K) * 2; }

static int64_t i8_tile_tokens(int64_t M) {
  const int64_t mpad = (M + 15) / 16 * 16;
  return mpad < 128 ? mpad : 128;  // token columns per CTA; more tokens take more CTAs
}

// One CTA per SM at most (shared memory), so a call with few output tiles leaves SMs idle and
// one with a few more than the SMs runs a second, mostly empty wave: split K into whole 512-K
// groups (at most 8 splits, at most one per group) where that shortens the modelled launch.
int i8_splits(int64_t M, int64_t N, int64_t K) {
  const int64_t tiles = (N + 127) / 128 * ((M + i8_tile_tokens(M) - 1) / i8_tile_tokens(M));
  const int64_t stages = i8_kpad(K) / kI8BlockK;
  const int64_t groups = (stages + kI8GroupStages - 1) / kI8GroupStages;
  // the launch's modelled time: waves of CTAs (one per SM), each ~0.45 us per 64-K stage of its
  // range plus a fixed ~8 us (prologue, drain, epilogue), ~12 us with a split (its slots and the
  // reduction); fewer splits win unless more are 3 % faster.  For 5120 x 17408 at 256 tokens (80
  // tiles) it picks 3 splits in 2 waves over 1 split in 1 wave on 80 SMs
  int best = 1;
  double best_t = 1e30;
  for (int ks = 1; ks <= 8 && ks <= groups; ++ks) {
    const int64_t waves = (tiles * ks + kNumSMs - 1) / kNumSMs;
    const double t = (double)waves * (0.45 * (double)((stages + ks - 1) / ks) + (ks > 1 ? 12.0 : 8.0));
    if (t < 0.97 * best_t) {
      best = ks;
      best_t = t;
    }
  }
  return best;
}

size_t i8_part_bytes(int64_t M, int64_t N, int64_t K) {
  const int ks = i8_splits(M, N, K);
  return ks > 1 ? (size_t)ks * M * N * 4 : 0;
}

cudaError_t launch_i8_gemm(const I8GemmArgs& g, cudaStream_t st) {
  const int64_t kpad = i8_kpad(g.K);
  // activation codes (exact f16), per-token scales
  quant_i8_image_kernel<<<g.M, 256, 0, st>>>(g.x, g.K, g.ldx, (int)kpad, g.img, g.xs, g.xq_dbg, g.xs_dbg, g.amax_in);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  I8Params p = {};
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.nk = (int)(kpad / kI8BlockK);
  p.tt = (int)i8_tile_tokens(g.M);
  p.ks = i8_splits(g.M, g.N, g.K);
  p.part = g.part;
  p.tickets = g.tickets;
  const size_t stage = (size_t)kI8A8Bytes + kI8A16Bytes + (size_t)p.tt * kI8BlockK * 2;
  const size_t budget = 227 * 1024 - 1024 - 1024;  // alignment slack, static shared memory
  int S = (int)(budget / stage);
  if (S > 8) S = 8;
  p.stages = S;
  p.w_s = g.w_s;
  p.w_s_len = g.w_s_len;
  p.x_s = g.xs;
  p.bias = g.bias;
  p.y = g.y;
  p.ldy = g.ldy;
  p.acc_out = g.acc_out;
  p.status = g.status;
  p.wait_limit = g.wait_limit;

  CUtensorMap ta, tb;
  // weights: int8 [N][K] rows of ldw bytes, box 64 K x 128 rows, plain rows (the converter warps
  // read them); activation codes: f16 [M][kpad], box 64 K x tt rows, 128-byte swizzle
  if (!i8_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.w, (uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.ldw, kI8BlockK, 128,
              CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !i8_map(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g.img, (uint64_t)kpad, (uint64_t)g.M, (uint64_t)kpad * 2, kI8BlockK,
              (uint32_t)p.tt, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // the output: bf16 [M][ldy], stored a [tt][128] box per CTA when its rows can be TMA rows
  // (16-byte aligned base and row pitch), N is a multiple of 8 (a TMA store clips the inner
  // dimension at whole 16-byte chunks) and K is not split (measured: M = 128 / 256 at 17408x5120
  // -1.6 / -3.3 us a call; the split calls at 5120x17408 gain nothing from it); else the drain
  // warps store it element by element
  CUtensorMap ty = ta;
  p.tma_y = 0;
  if (g.y && p.ks == 1 && g.N % 8 == 0 && (reinterpret_cast<uintptr_t>(g.y) & 15) == 0 && (g.ldy * 2) % 16 == 0 &&
      i8_map(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.y, (uint64_t)g.N, (uint64_t)g.M, (uint64_t)g.ldy * 2, 128,
             (uint32_t)p.tt, CU_TENSOR_MAP_SWIZZLE_NONE))
    p.tma_y = 1;

  const size_t smem = 1024 + (size_t)S * stage + (size_t)(3 * S + 5) * 8;
  static std::atomic<int> attr{0};
  if (!attr.load()) {
    e = raise_smem_limit(i8_gemm_kernel<false>);
    if (e == cudaSuccess) e = raise_smem_limit(i8_gemm_kernel<true>);
    if (e != cudaSuccess) return e;
    attr.store(1);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((g.N + 127) / 128), (unsigned)((g.M + p.tt - 1) / p.tt), (unsigned)p.ks);
  cfg.blockDim = dim3(kI8Threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return p.ks > 1 ? cudaLaunchKernelEx(&cfg, i8_gemm_kernel<true>, ta, tb, ty, p)
                  : cudaLaunchKernelEx(&cfg, i8_gemm_kernel<false>, ta, tb, ty, p);
}

}  // namespace tc
}  // namespace ql
