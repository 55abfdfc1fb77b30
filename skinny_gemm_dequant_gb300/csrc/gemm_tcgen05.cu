// Block-scaled GEMM on the 5th-generation tensor cores (tcgen05) for batched decode/prefill
// (M >= 17 tokens) with 1x128 E4M3 activations, FP8-E4M3 or MXFP4 (E2M1) weights.
//
// Formula ([Z100] §二.2.4 / chapter 三 §2, block-scaled FP8):
//   y[m,n] = sum_kb a_s[m,kb] * w_s[n/128,kb] * sum_{k in kb} a[m,k] w[n,k]
// and for MXFP4 weights ([DSV4] §9.3) the weight scale is per row and per 32 K.  Every scale is
// a power of two (UE8M0), so applying them per 32-K MMA step inside the tensor core
// (kind::mxf8f6f4 .block_scale, one scale byte per row and per 32 K) gives exactly the formula.
//
// Mapping (swap-AB): the MMA's A operand is a 128-row weight tile, its N dimension is the token
// tile (16..256), so D[128 x tokens] lives in tensor memory, 1 fp32 column per token.
// Roles inside a CTA of 8 warps:
//   warp 0     : TMA producer (weights and activation codes, 128 K per stage, 128B swizzle);
//   warp 1     : tensor-memory allocation and the single MMA-issuing thread;
//   warps 4..7 : write the per-stage UE8M0 scale vectors into tensor memory (tcgen05.st),
//                then the epilogue (tcgen05.ld -> bf16 -> global).
// Every mbarrier wait is bounded; a wait that runs out raises QL_DEV_TIMEOUT in the status word,
// the other roles stop, copies and MMAs still in flight are waited for, and tensor memory is
// freed before the CTA exits.
#include <cudaTypedefs.h>

#include <cstdio>
#include <atomic>
#include <mutex>

#include "gemm_tcgen05.h"
#include "internal.h"
#include "tc_ptx.cuh"

namespace ql {
namespace tc {

constexpr int kThreads = 256;
constexpr int kBlockN = 128;  // weight rows per CTA (MMA M)
constexpr int kBlockK = 128;  // K elements per stage
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;  // scale vectors live after the (<= 256-column) accumulator
constexpr uint32_t kSfColResident = 128;  // resident scale vectors: after a <= 128-column accumulator
constexpr int kResidentFirst = 8;  // resident scales: stages written before the MMAs may start
#ifndef QL_RESIDENT_SCALES
#define QL_RESIDENT_SCALES 1  // 0: every call writes its scale vectors into the ring, stage by stage
#endif
constexpr uint32_t kDrainLimit = 1u << 22;

struct TcParams {
  int M, N, K;
  int tt, nsub, sub_n, stages;
  int fp4;
  const uint8_t* ws;
  int64_t lds;
  const uint8_t* as;
  int64_t las;
  uint16_t* y;
  int64_t ldy;
  const uint16_t* bias;
  uint32_t* status;
  uint32_t wait_limit;
  int sf_layout;  // 0: row r at (lane r % 32 of every quadrant, column r / 32); 1: (lane r, column 0)
  int staged;     // 1: every scale byte of the CTA is copied to shared memory once, at the start
  // 1 (staged, one token sub-tile of <= 128 columns, every stage's scale vectors fit in tensor
  // memory behind the accumulator): the scale writers put all of them in tensor memory before
  // the MMAs need them, instead of one ring slot per stage (which paced the MMAs: the writer
  // sharing a scheduler with the MMA-issuing warp fell ~0.45 us behind every stage)
  int resident;
  int tma_y;  // 1: the output tile leaves through shared memory and one TMA store (tmY)
  uint32_t sc_w_bytes;  // shared-memory bytes of the staged weight scales (16-byte multiple)
  // grouped (MoE) launches: blockIdx.y indexes a tile list built on the device
  int grouped;
  const int4* tiles;     // (expert, first dispatch row, rows, 0)
  const int* ntiles;
  const int32_t* pairs;  // dispatch row -> (token, slot) pair
  float* out;            // fp32 [pair][ld_out]
  int64_t ld_out;
  int64_t s_estride;     // bytes between two experts' weight-scale arrays
};

// Staged scales, behind the mbarriers:
//   weights, FP8: one byte per stage (the CTA's 128 rows share one 128x128 block row);
//   weights, FP4: one 32-bit word (4 x 32-K scale bytes) per row and stage, stage-major, the row
//                 index XORed with (stage & 31) so that both the staging writes (consecutive
//                 stages) and the per-stage reads (consecutive rows) hit 32 distinct banks;
//   activations: one byte per token of the tile and stage, stage-major.
__host__ __device__ constexpr uint32_t sc_w_bytes(int fp4, int nk) {
  return ((uint32_t)(fp4 ? nk * 128 * 4 : nk) + 15u) & ~15u;
}

__device__ __forceinline__ uint32_t rep4(uint32_t b) { return (b & 0xFFu) * 0x01010101u; }

__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmY, const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  const uint32_t a_bytes = kBlockN * kBlockK;          // 16 KB of A per stage (fp4 unpacked to bytes)
  const uint32_t b_bytes = (uint32_t)p.tt * kBlockK;   // tokens x 128 B
  // transaction bytes of the A load: packed fp4 counts the bytes read (8 KB), not the padded
  // shared-memory image it expands to
  const uint32_t a_tx = p.fp4 ? a_bytes / 2 : a_bytes;
  uint8_t* sA = smem;
  uint8_t* sB = smem + (size_t)S * a_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + (size_t)S * b_bytes);
  uint64_t* tma_full = bars;
  uint64_t* sf_full = bars + S;
  uint64_t* empty = bars + 2 * S;
  uint64_t* acc_full = bars + 3 * S;
  uint8_t* sc_w = reinterpret_cast<uint8_t*>(bars + 3 * S + 2);  // staged scales (p.staged)
  uint8_t* sc_a = sc_w + p.sc_w_bytes;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBlockN;
  int t0 = blockIdx.y * p.tt;
  int expert = 0, ntok = p.M - t0;  // token columns of this tile that hold real tokens
  if (p.grouped) {
    // the tile list comes from the dispatch launch; a CTA beyond its end has nothing to do
    pdl_wait();
    if ((int)blockIdx.y >= *p.ntiles) return;
    const int4 tl = p.tiles[blockIdx.y];
    expert = tl.x;
    t0 = tl.y;
    ntok = tl.z;
  }
  const uint8_t* wsc = p.ws + (int64_t)expert * p.s_estride;  // this expert's weight scales
  const int nk = p.K / kBlockK;
  const uint32_t lim = p.wait_limit;
  volatile int* abort = &s_abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&tma_full[s], 1);
      mbar_init(&sf_full[s], 4);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
    s_abort = 0;
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemCols);
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

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    // weight tile of stage kt: a 2D view, or (grouped) a 3D view with the expert outermost
    auto load_a = [&](uint8_t* dst, int kt, uint64_t* bar) {
      if (p.grouped)
        tma_load_3d(dst, &tmA, kt * kBlockK, n0, expert, bar);
      else
        tma_load_2d(dst, &tmA, kt * kBlockK, n0, bar);
    };
    const int pre = nk < S ? nk : S;
    for (int kt = 0; kt < pre; ++kt) {  // weights do not depend on the previous kernel
      mbar_arrive_expect_tx(&tma_full[kt], a_tx + b_bytes);
      load_a(sA + (size_t)kt * a_bytes, kt, &tma_full[kt]);
    }
    pdl_wait();  // activation codes come from the quantisation kernel
    for (int kt = 0; kt < pre; ++kt) tma_load_2d(sB + (size_t)kt * b_bytes, &tmB, kt * kBlockK, t0, &tma_full[kt]);
    int issued = pre;
    // slot and phase kept incrementally (no divisions by the runtime stage count in a loop one
    // thread runs per stage)
    int s = pre == S ? 0 : pre;
    uint32_t ph = 0;  // parity of the slot's previous use
    for (int kt = pre; kt < nk; ++kt) {
      if (!mbar_wait(&empty[s], ph, lim, abort)) {
        fail();
        break;
      }
      mbar_arrive_expect_tx(&tma_full[s], a_tx + b_bytes);
      load_a(sA + (size_t)s * a_bytes, kt, &tma_full[s]);
      tma_load_2d(sB + (size_t)s * b_bytes, &tmB, kt * kBlockK, t0, &tma_full[s]);
      issued = kt + 1;
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (*abort) {
      // no copy may land after the CTA exits: wait for the last load of every stage
      for (int kt = issued - S < 0 ? 0 : issued - S; kt < issued; ++kt)
        mbar_wait(&tma_full[kt % S], (uint32_t)(kt / S) & 1, kDrainLimit, nullptr);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues every MMA, so the loop body is kept to the MMAs themselves: instruction
    // descriptors are built once, and shared-memory descriptors (linear in the address: the
    // start-address field holds address / 16) advance by constants
    const uint32_t a_fmt = p.fp4 ? 5u : 0u;  // E2M1 or E4M3
    uint32_t idesc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) idesc[j] = idesc_mxf8f6f4(a_fmt, 0u, (uint32_t)p.sub_n, (uint32_t)j, (uint32_t)j);
    const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA)), b_desc0 = smem_desc_sw128(smem_u32(sB));
    const uint32_t a_step = a_bytes >> 4, b_step = b_bytes >> 4, b_sub = ((uint32_t)p.sub_n * kBlockK) >> 4;
    const uint32_t sf_stride = 4 + 4 * (uint32_t)p.nsub;
    const bool two = p.nsub > 1;
    // slot, parity and the stage's descriptor / scale-column offsets kept incrementally: this
    // thread's instructions per stage pace the tensor core
    int s = 0;
    uint32_t par = 0;
    uint64_t aoff = 0, boff = 0;
    uint32_t sfoff = 0;
    uint32_t ready = 0;  // bits 0 / 1: this stage's TMA / scale barriers already seen complete
    const uint32_t sf_base = p.resident ? kSfColResident : kSfCol0;
    for (int kt = 0; kt < nk; ++kt) {
      if (p.resident) {
        // resident scales: the first stages' vectors before stage 0, the rest before stage 8
        if ((kt == 0 || kt == kResidentFirst) && !mbar_wait(&sf_full[kt == 0 ? 0 : 1], 0, lim, abort)) {
          fail();
          break;
        }
        ready |= 2u;
      }
      if ((!(ready & 1) && !mbar_wait(&tma_full[s], par, lim, abort)) ||
          (!(ready & 2) && !mbar_wait(&sf_full[s], par, lim, abort))) {
        fail();
        break;
      }
      tc_fence_after();
      const uint64_t ad = a_desc0 + aoff, bd = b_desc0 + boff;
      const uint32_t sfa = tmem + sf_base + sfoff;
      // four 32-K steps (32 bytes = 2 descriptor units each), scale byte j of each vector; the
      // next stage's barriers are tested while the first token tile's MMAs issue
      const int sn = s + 1 == S ? 0 : s + 1;
      const uint32_t pn = s + 1 == S ? par ^ 1u : par;
      ready = mma4_mxf8f6f4_test2(tmem, ad, bd, idesc, sfa, sfa + 4, kt > 0 ? 1u : 0u, smem_u32(&tma_full[sn]),
                                  smem_u32(&sf_full[sn]), pn);
      if (two) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_mxf8f6f4(tmem + (uint32_t)p.sub_n, ad + 2 * j, bd + b_sub + 2 * j, idesc[j], sfa, sfa + 8,
                       (kt > 0 || j > 0) ? 1u : 0u);
      }
      tc_commit(&empty[s]);
      aoff += a_step;
      boff += b_step;
      sfoff += sf_stride;
      if (++s == S) {
        s = 0;
        par ^= 1u;
        aoff = boff = 0;
        if (!p.resident) sfoff = 0;  // resident scales: one column group per stage, no ring
      }
    }
    tc_commit(acc_full);  // completes once every MMA issued above has finished
    if (*abort) mbar_wait(acc_full, 0, kDrainLimit, nullptr);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ scale vectors, then epilogue
    pdl_wait();  // activation scales come from the quantisation kernel
    if (p.staged) {
      // warps 2..7 copy the CTA's scale bytes to shared memory once; out-of-range rows and
      // tokens get the neutral scale 2^0
      const int tid = threadIdx.x - 64, nthr = kThreads - 64;
      if (p.fp4) {
        uint32_t* w32 = reinterpret_cast<uint32_t*>(sc_w);
        for (int i = tid; i < 128 * nk; i += nthr) {
          const int r = i / nk, kt = i - r * nk;  // consecutive threads: consecutive stages of a row
          const int n = n0 + r;
          const uint32_t v =
              n < p.N ? __ldg(reinterpret_cast<const uint32_t*>(wsc + (int64_t)n * p.lds + 4 * kt)) : 0x7F7F7F7Fu;
          w32[kt * 128 + (r ^ (kt & 31))] = v;
        }
      } else {
        for (int kt = tid; kt < nk; kt += nthr) sc_w[kt] = n0 < p.N ? __ldg(wsc + (int64_t)(n0 / 128) * p.lds + kt) : 0x7F;
      }
      for (int i = tid; i < p.tt * nk; i += nthr) {
        const int kt = i / p.tt, t = i - kt * p.tt;  // consecutive threads: consecutive tokens
        sc_a[i] = t < ntok ? __ldg(p.as + (int64_t)(t0 + t) * p.las + kt) : 0x7F;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kThreads - 64) : "memory");
    }
  }
  if (warp >= 4) {
    const int q = warp - 4;  // tensor-memory lane quadrant of this warp
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    bool ok = true;
    // the scale words of a stage are read kPD stages ahead into registers (the loop is unrolled
    // by kPD so every array index is a constant).  Staged, they come from shared memory; else
    // from global memory, and then every stage also waits for an L2 round trip, because the
    // release of the mbarrier arrive waits for the loads issued before it
    constexpr int kPD = 4;
    uint32_t pw[kPD][4], pb[kPD][2][4];
    auto fetch = [&](int kt, uint32_t (&wa)[4], uint32_t (&wb)[2][4]) {
      if (kt >= nk) return;
      if (p.staged) {  // shared memory: no global load (and no wait for one) inside the loop
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = (p.sf_layout == 0) ? (lane + 32 * j) : (32 * q + lane);
          wa[j] = p.fp4 ? reinterpret_cast<const uint32_t*>(sc_w)[kt * 128 + (r ^ (kt & 31))] : rep4(sc_w[kt]);
        }
#pragma unroll
        for (int sub = 0; sub < 2; ++sub)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = (p.sf_layout == 0) ? (lane + 32 * j) : (32 * q + lane);
            wb[sub][j] = (sub < p.nsub && r < p.sub_n) ? rep4(sc_a[kt * p.tt + sub * p.sub_n + r]) : 0x7F7F7F7Fu;
          }
        return;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = (p.sf_layout == 0) ? (lane + 32 * j) : (32 * q + lane);
        const int n = n0 + r;
        uint32_t wv = 0x7F7F7F7Fu;
        if (n < p.N) {
          if (p.fp4) wv = __ldg(reinterpret_cast<const uint32_t*>(wsc + (int64_t)n * p.lds + 4 * kt));
          else wv = rep4(__ldg(wsc + (int64_t)(n0 / 128) * p.lds + kt));
        }
        wa[j] = wv;
      }
#pragma unroll
      for (int sub = 0; sub < 2; ++sub)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = (p.sf_layout == 0) ? (lane + 32 * j) : (32 * q + lane);
          const int tc = sub * p.sub_n + r;  // token column
          wb[sub][j] = (sub < p.nsub && r < p.sub_n && tc < ntok) ? rep4(__ldg(p.as + (int64_t)(t0 + tc) * p.las + kt))
                                                                  : 0x7F7F7F7Fu;
        }
    };
#pragma unroll
    for (int d = 0; d < kPD; ++d) fetch(d, pw[d], pb[d]);
    if (p.resident) {
      // every stage's vectors at its own columns, no ring and no wait: the MMAs start once the
      // first kResidentFirst stages are in (sf_full[0]) and take the rest after sf_full[1]
      const int first = nk < kResidentFirst ? nk : kResidentFirst;
      for (int kt = 0; kt < nk; ++kt) {
        uint32_t wa[4], wb[2][4];
        fetch(kt, wa, wb);
        const uint32_t sf_col = kSfColResident + (uint32_t)kt * (4 + 4 * p.nsub);
        tmem_st_x4(tmem + lane_base + sf_col, wa[0], wa[1], wa[2], wa[3]);
        tmem_st_x4(tmem + lane_base + sf_col + 4, wb[0][0], wb[0][1], wb[0][2], wb[0][3]);
        if (kt + 1 == first || kt + 1 == nk) {
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sf_full[kt + 1 == first ? 0 : 1]);
        }
      }
    }
    int s = 0;
    uint32_t ph = 1;  // parity of the slot's previous use (a fresh barrier passes parity 1)
    for (int k0 = 0; k0 < nk && ok && !p.resident; k0 += kPD) {
#pragma unroll
      for (int d = 0; d < kPD; ++d) {
        const int kt = k0 + d;
        if (kt >= nk) break;
        // lane 0 waits and the result is broadcast, so the warp stays converged for the
        // .sync.aligned tensor-memory stores below
        int got = 0;
        if (lane == 0) got = mbar_wait(&empty[s], ph, lim, abort);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sf_col = kSfCol0 + (uint32_t)s * (4 + 4 * p.nsub);
        // weight scale vectors: one byte per 32-K step (4 per stage) for each of the 128 rows;
        // then the activation scale vectors: the token's 1x128 scale repeated for the 4 steps
        tmem_st_x4(tmem + lane_base + sf_col, pw[d][0], pw[d][1], pw[d][2], pw[d][3]);
        tmem_st_x4(tmem + lane_base + sf_col + 4, pb[d][0][0], pb[d][0][1], pb[d][0][2], pb[d][0][3]);
        if (p.nsub > 1) tmem_st_x4(tmem + lane_base + sf_col + 8, pb[d][1][0], pb[d][1][1], pb[d][1][2], pb[d][1][3]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_full[s]);
        fetch(kt + kPD, pw[d], pb[d]);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // grouped: the tile's pair of every dispatch row into shared memory (every epilogue warp
    // gets here): read from global memory inside the output loop, each load waited behind the
    // previous outputs' stores
    __shared__ int32_t s_pairs[256];
    if (p.grouped) {
      for (int i = threadIdx.x - 128; i < p.tt; i += 128) s_pairs[i] = i < ntok ? p.pairs[t0 + i] : 0;
      asm volatile("bar.sync 2, 128;" ::: "memory");  // the four epilogue warps
    }
    int got = 0;
    if (ok && lane == 0) got = mbar_wait(acc_full, 0, lim, abort);
    got = __shfl_sync(0xffffffffu, got, 0);
    if (got) {
      tc_fence_after();
      const int n = n0 + 32 * q + lane;
      const float bias = (p.bias && n < p.N) ? bf16_bits_to_f32(p.bias[n]) : 0.f;
      for (int c0 = 0; c0 < p.tt; c0 += 32) {
        uint32_t r[32];
        tmem_ld_x32(tmem + lane_base + (uint32_t)c0, r);
        tmem_wait_ld();
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int tc = c0 + j;  // token column
            if (tc < p.tt && tc < ntok) {
              if (p.grouped) {  // fp32 row of the (token, slot) pair at this dispatch row
                p.out[(int64_t)s_pairs[tc] * p.ld_out + n] = __uint_as_float(r[j]);
              } else {
                uint16_t yb = f32_to_bf16_rn(__uint_as_float(r[j]));
                if (p.bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + bias);
                if (p.tma_y)  // [tt][128] tile in the idle stage ring, stored below
                  reinterpret_cast<uint16_t*>(smem)[tc * kBlockN + 32 * q + lane] = yb;
                else
                  p.y[(int64_t)(t0 + tc) * p.ldy + n] = yb;
              }
            }
          }
        }
      }
    } else if (ok && lane == 0) {
      fail();
    }
    if (p.tma_y) {
      // every epilogue warp reaches the barrier; the tile goes out in one store unless a wait
      // timed out
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> TMA reads
      asm volatile("bar.sync 2, 128;" ::: "memory");                // the four epilogue warps
      if (warp == 4 && lane == 0 && got && !*abort) {
        tma_store_2d(&tmY, smem_u32(smem), n0, t0);
        bulk_commit_and_wait_all();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

static bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) fprintf(stderr, "qlinear: cuTensorMapEncodeTiled failed (%d)\n", (int)r);
  return r == CUDA_SUCCESS;
}

// 3D view {inner, outer, experts} with a byte stride between experts, 128-byte swizzle
static bool make_map3(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t experts, uint64_t row_bytes, uint64_t expert_bytes, uint32_t box_inner,
                      uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, outer, experts};
  cuuint64_t strides[2] = {row_bytes, expert_bytes};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) fprintf(stderr, "qlinear: cuTensorMapEncodeTiled failed (%d)\n", (int)r);
  return r == CUDA_SUCCESS;
}

size_t act_q_bytes(int64_t M, int64_t K) { return (size_t)M * K; }
size_t act_s_bytes(int64_t M, int64_t K) { return (size_t)M * (K / 128); }

cudaError_t quantize_activations(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const GemmArgs& g,
                                 uint8_t* aq_dbg, uint8_t* as_dbg, cudaStream_t st) {
  return launch_quant_e4m3(x, (int)M, (int)K, ldx, g.aq, K, g.as, K / 128, 0, aq_dbg, as_dbg, st);
}

#ifndef QL_SF_LAYOUT
#define QL_SF_LAYOUT 0
#endif

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t st) {
  TcParams p = {};
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.fp4 = g.fp4;
  int mpad = ((g.M + 15) / 16) * 16;
  if (mpad > 256) mpad = 256;
  if (g.grouped) mpad = g.tt;  // tiles of the caller's width, one MMA sub-tile
  p.nsub = (mpad + 127) / 128;
  p.sub_n = (((mpad + p.nsub - 1) / p.nsub) + 15) / 16 * 16;
  p.tt = p.nsub * p.sub_n;
  const size_t stage = (size_t)kBlockN * kBlockK + (size_t)p.tt * kBlockK;
  const size_t budget = 227 * 1024 - 1024 - 2048;  // alignment slack, static shared memory
  const int nk = g.K / kBlockK;
  // stage the scales in shared memory when they take at most 48 KB and leave two stages
  const size_t sc_bytes = sc_w_bytes(g.fp4, nk) + (((size_t)p.tt * nk + 15) & ~(size_t)15);
  p.staged = (sc_bytes <= 48 * 1024 && budget >= sc_bytes + 2 * stage) ? 1 : 0;
  p.sc_w_bytes = p.staged ? sc_w_bytes(g.fp4, nk) : 0;
  const size_t extra = p.staged ? sc_bytes : 0;
  int S = (int)((budget - extra) / stage);
  if (S > 8) S = 8;
  p.stages = S;
  p.resident = (QL_RESIDENT_SCALES && p.staged && p.nsub == 1 && p.tt <= (int)kSfColResident &&
                kSfColResident + (uint32_t)nk * (4 + 4 * (uint32_t)p.nsub) <= kTmemCols)
                   ? 1
                   : 0;
  p.ws = g.ws;
  p.lds = g.lds;
  p.as = g.as;
  p.las = g.K / 128;
  p.y = g.y;
  p.ldy = g.ldy;
  p.bias = g.bias;
  p.status = g.status;
  p.wait_limit = g.wait_limit;
  p.sf_layout = QL_SF_LAYOUT;
  p.grouped = g.grouped;
  p.tiles = g.tiles;
  p.ntiles = g.ntiles;
  p.pairs = g.pairs;
  p.out = g.out;
  p.ld_out = g.ld_out;
  p.s_estride = g.grouped ? g.s_estride : 0;

  CUtensorMap ta, tb;
  const CUtensorMapDataType wt = g.fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const bool ok_a = g.grouped ? make_map3(&ta, wt, g.w, (uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.experts,
                                          (uint64_t)g.ldw, (uint64_t)g.w_estride, kBlockK, kBlockN)
                              : make_map(&ta, wt, g.w, (uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.ldw, kBlockK, kBlockN);
  const bool ok_b = make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.aq, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)g.K,
                             kBlockK, (uint32_t)p.tt);
  if (!ok_a || !ok_b) return cudaErrorInvalidValue;
  // the dense output: bf16 [M][ldy], stored a [tt][128] box per CTA when its rows can be TMA rows
  // (16-byte aligned base and row pitch) and N is a multiple of 8: a TMA store clips the inner
  // dimension at whole 16-byte chunks, so a row ending inside one would get the chunk's columns
  // past N written too; else the epilogue warps store it element by element
  CUtensorMap ty = ta;
  p.tma_y = 0;
  if (!g.grouped && g.y && g.N % 8 == 0 && (reinterpret_cast<uintptr_t>(g.y) & 15) == 0 && (g.ldy * 2) % 16 == 0) {
    auto fn = encode_fn();
    cuuint64_t dims[2] = {(cuuint64_t)g.N, (cuuint64_t)g.M};
    cuuint64_t strides[1] = {(cuuint64_t)g.ldy * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBlockN, (cuuint32_t)p.tt};
    cuuint32_t estr[2] = {1, 1};
    if (fn && fn(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.y, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      p.tma_y = 1;
  }

  const size_t smem = 1024 + (size_t)S * stage + (size_t)(3 * S + 2) * 8 + extra;
  static std::atomic<int> attr_set{0};
  if (!attr_set.load()) {
    cudaError_t e = raise_smem_limit(tc_gemm_kernel);
    if (e != cudaSuccess) return e;
    attr_set.store(1);
  }
  cudaLaunchConfig_t cfg = {};
  const unsigned gy = g.grouped ? (unsigned)g.tiles_max : (unsigned)((g.M + p.tt - 1) / p.tt);
  cfg.gridDim = dim3((unsigned)((g.N + kBlockN - 1) / kBlockN), gy, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel, ta, tb, ty, p);
}

}  // namespace tc
}  // namespace ql
