// Persistent, TMA-fed skinny GEMM (M <= 16 tokens) for INT8, FP8-block and MXFP4 weights.
//
// Work: the weight matrix is cut into units of (128-row block, 128 weight bytes of K).  The
// units, ordered row block by row block, are split into one contiguous range per CTA, one CTA
// per SM, so every SM streams the same number of weight bytes (no wave tail).  A row block split
// between CTAs cf..cl is settled by cf, the CTA holding its first unit: those units are the last
// ones cf streams, while cf+1..cl reach theirs earlier, store their partial sums and count
// themselves in (release); cf waits for the count (bounded), adds the partials in CTA order to
// its own and writes the outputs, so results do not depend on timing.
//
// Inside a CTA, warp 16 is the producer: it keeps a ring of up to a dozen stages in flight, each
// a 128x128-byte weight tile and the matching activation tile (f16, prepared once per call by
// the prologue kernel), both loaded by TMA with 128-byte swizzling, plus (MXFP4) the tile's
// per-32 scale bytes by cp.async.  Warps 0..7 consume, as 2 row groups (64 rows, four 16-row
// MMA tiles) x 4 K quarters (two 16-byte chunks of every unit): a warp loads its activation
// fragments once per unit and uses them for all four of its row tiles, which keeps the
// shared-memory traffic per weight byte low.  ldmatrix gives each thread 4 weight bytes of a
// chunk for rows g and g+8, converted to f16 in registers and fed to the warp MMA m16n8k16
// (f32 accumulate) against the activations.  Each MMA draws all its K values from one 16-byte
// chunk, i.e. from one 32-element MXFP4 scale group, so scales fold exactly per chunk (per
// 32 K within a 128x128 FP8 block, exact integers for INT8).  The four K quarters of a row
// group add their sums through shared memory when a row block ends.
#pragma once
#include "common.cuh"
#include "tc_ptx.cuh"

namespace ql {

constexpr int S2_TILES = 8;                      // 16-row tiles per unit
constexpr int S2_RG = 2;                         // row groups of 4 tiles (64 rows)
constexpr int S2_KQ = 4;                         // K quarters of a unit (2 chunks each)
constexpr int S2_TPW = S2_TILES / S2_RG;         // tiles per consumer warp
constexpr int S2_CONSUMERS = S2_RG * S2_KQ;      // 8 consumer warps
constexpr int S2_THREADS = 32 * (S2_CONSUMERS + 1);
constexpr int S2_ROWS = 16 * S2_TILES;           // 128 weight rows per unit
constexpr int S2_WB = 128;                       // weight bytes per row per unit

struct Skinny2Args {
  int M, N, K;
  int nk;          // units per row block
  int64_t total;   // row blocks x nk
  int maxseg;      // partial slots per row block
  const uint8_t* wsb;  // FP8: UE8M0 grid [ceil(N/bn), lds]; MXFP4: UE8M0 [N, lds]
  int64_t lds;
  int block_n, block_k;
  const float* w_scale;  // INT8 per-channel / per-tensor scales
  int w_scale_len;
  const float* x_s;       // INT8 per-token scales
  const float* tokscale;  // bf16 activations: per-token 2^p undone in the epilogue
  uint16_t* y;
  int64_t ldy;
  const uint16_t* bias;
  int32_t* acc_out;
  float* part;        // [row blocks][maxseg][16][128] partial sums (fp32 or int32 bits)
  unsigned* tickets;  // [row blocks] arrival counts of the partial sums
  uint32_t* status;
  uint32_t wait_limit;
  int stages;
  int xcopies;  // copies of the activation image; CTA c reads copy c % xcopies (spreads L2 load)
};

template <int FMT>
struct S2Traits {
  static constexpr int KPU = (FMT == FMT_MXFP4) ? 256 : 128;  // K elements per unit
  static constexpr int NXB = KPU / 64;                         // 64-element activation boxes per unit
  static constexpr int SCB = (FMT == FMT_MXFP4) ? S2_ROWS * 8 : 0;  // scale bytes per unit
};

template <int FMT, int MT>
__host__ __device__ constexpr uint32_t s2_stage_bytes() {
  return S2_ROWS * S2_WB + S2Traits<FMT>::NXB * (8 * MT) * 128 + S2Traits<FMT>::SCB;
}

// shared memory for the K-quarter exchange at row-block ends:
// [row group][3 non-lead quarters][4 tiles][32 lanes][4*MT] floats
template <int MT>
__host__ __device__ constexpr uint32_t s2_xchg_bytes() {
  return S2_RG * (S2_KQ - 1) * S2_TPW * 32 * 4 * MT * 4;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}
// named barrier of the consumer warps (the producer warp never joins it)
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// CTA owning unit s when `total` units are split into G contiguous ranges [c*T/G, (c+1)*T/G)
__device__ __forceinline__ int s2_cta_of(int64_t s, int64_t T, int G) {
  return (int)(((s + 1) * G + T - 1) / T) - 1;
}

// swizzled byte offset of (row, byte) inside a TMA tile of 128-byte rows (128B swizzle)
__device__ __forceinline__ uint32_t sw128(int row, int byte) {
  return (uint32_t)(row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15)));
}

template <int FMT, int MT>
__global__ void __launch_bounds__(S2_THREADS, 1)
    skinny2_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ Skinny2Args a) {
  using Tr = S2Traits<FMT>;
  constexpr int Mp = 8 * MT;
  constexpr uint32_t W_BYTES = S2_ROWS * S2_WB;
  constexpr uint32_t X_BOX = Mp * 128;
  constexpr uint32_t STAGE = s2_stage_bytes<FMT, MT>();
  constexpr bool kInt = (FMT == FMT_INT8);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * STAGE);
  uint64_t* empty = full + S;
  float* xchg = reinterpret_cast<float*>(empty + S);                        // pair exchange
  uint8_t* fp8sc = reinterpret_cast<uint8_t*>(xchg) + s2_xchg_bytes<MT>();  // FP8 scale rows
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int64_t T = a.total;
  const int64_t s0 = (int64_t)c * T / G, s1 = (int64_t)(c + 1) * T / G;
  const int nk = a.nk;
  const uint32_t lim = a.wait_limit;
  volatile int* abort = &s_abort;
  auto fail = [&]() {
    atomicOr(a.status, (uint32_t)QL_DEV_TIMEOUT);
    *abort = 1;
  };

  // FP8 block scales: the rows of every n-block this CTA's units touch, copied up front
  const int rb_first = (int)(s0 / nk);
  const int nbr = (a.block_n > 0) ? (S2_ROWS / a.block_n + 2) : 0;  // n-blocks a 128-row block spans
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], FMT == FMT_MXFP4 ? 1 + 32 : 1);
      tc::mbar_init(&empty[i], S2_CONSUMERS);
    }
    tc::fence_mbar_init();
    s_abort = 0;
    tc::tma_prefetch_desc(&tmW);
    tc::tma_prefetch_desc(&tmX);
  }
  if constexpr (FMT == FMT_FP8) {
    const int rb_last = (s1 > s0) ? (int)((s1 - 1) / nk) : rb_first;
    const int nrow_blocks = rb_last - rb_first + 1;
    const int nb0 = (rb_first * S2_ROWS) / a.block_n;
    const int nb_count = min(nrow_blocks * nbr, (int)((a.N + a.block_n - 1) / a.block_n) - nb0);
    for (int i = threadIdx.x; i < nb_count * a.lds; i += blockDim.x)
      fp8sc[i] = a.wsb[(int64_t)nb0 * a.lds + i];
  }
  __syncthreads();

  if (warp == S2_CONSUMERS) {
    // ------------------------------------------------------------ producer warp
    const int pre = (int)((int64_t)S < s1 - s0 ? (int64_t)S : s1 - s0);
    const int xrow = (c % a.xcopies) * Mp;  // first row of this CTA's copy of the activations
    bool ok = true;
    int64_t issued = s0;
    for (int64_t s = s0; s < s1; ++s) {
      const int i = (int)(s - s0);
      const int slot = i % S;
      int got = 1;
      if (lane == 0 && i >= S) got = tc::mbar_wait(&empty[slot], ((uint32_t)(i / S) - 1) & 1, lim, abort);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) fail();
        ok = false;
        break;
      }
      const int rb = (int)(s / nk), kt = (int)(s % nk);
      uint8_t* st = smem + (size_t)slot * STAGE;
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(&full[slot], W_BYTES + Tr::NXB * X_BOX);
        tc::tma_load_2d(st, &tmW, kt * S2_WB, rb * S2_ROWS, &full[slot]);
        if (i >= pre) {
#pragma unroll
          for (int b = 0; b < Tr::NXB; ++b)
            tc::tma_load_2d(st + W_BYTES + b * X_BOX, &tmX, kt * Tr::KPU + b * 64, xrow, &full[slot]);
        } else if (i == pre - 1) {
          // activations come from the prologue kernel: wait for it once, then load the
          // activation tiles of the stages already in flight
          pdl_wait();
          for (int j = 0; j < pre; ++j) {
            const int64_t sj = s0 + j;
            uint8_t* stj = smem + (size_t)(j % S) * STAGE;
#pragma unroll
            for (int b = 0; b < Tr::NXB; ++b)
              tc::tma_load_2d(stj + W_BYTES + b * X_BOX, &tmX, (int)(sj % nk) * Tr::KPU + b * 64, xrow, &full[j % S]);
          }
        }
      }
      if constexpr (FMT == FMT_MXFP4) {
        // per-32 scale bytes of the unit: 128 rows x 8 bytes, 4 rows per lane
        const uint32_t sc = tc::smem_u32(st + W_BYTES + Tr::NXB * X_BOX);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = lane * 4 + j;
          const int n = min(rb * S2_ROWS + r, a.N - 1);
          cp_async8(sc + r * 8, a.wsb + (int64_t)n * a.lds + kt * 8);
        }
        cp_async_mbar_arrive(&full[slot]);
      }
      issued = s + 1;
    }
    if (!ok && lane == 0) {
      // no copy may land after the CTA exits: wait for every stage still in flight
      for (int64_t s = max(s0, issued - S); s < issued; ++s) {
        const int i = (int)(s - s0);
        tc::mbar_wait(&full[i % S], (uint32_t)(i / S) & 1, 1u << 22, nullptr);
      }
    }
    if constexpr (FMT == FMT_MXFP4) asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }

  // -------------------------------------------------------------- consumer warps
  pdl_wait();
  const int g = lane >> 2, t = lane & 3;
  const int rg = warp / S2_KQ;   // row group: tiles 4*rg .. 4*rg+3 (rows 64*rg ..)
  const int kq = warp % S2_KQ;   // K quarter of every unit: chunks 2*kq, 2*kq+1
  const bool lead = kq == 0;     // the warp of the row group that writes results
  // per-token epilogue factors of this thread's columns (x_s or 2^p), loaded once
  float colf[MT][2];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = 2 * t + e + 8 * m;
      colf[m][e] = col < a.M ? (kInt ? a.x_s[col] : a.tokscale[col]) : 0.f;
    }
  // ldmatrix addressing: lane L feeds row (L & 7) + 8*((L >> 3) & 1) of its matrix, chunk L >> 4
  const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int lchk = lane >> 4;
  // accumulator element r of tile i, token tile m: row 16*(4*rg+i) + g + 8*(r>=2), col 2t+(r&1)+8m
  float acc[S2_TPW][MT][4];
  int32_t acci[S2_TPW][MT][4];
  float own[S2_TPW][MT][4];  // partial sums of the block this CTA settles (lead warps)
  int settle_rb = -1;
  bool ok = true;
  int64_t s = s0;
  while (s < s1) {
    const int rb = (int)(s / nk);
    const int kt0 = (int)(s % nk);
    const int64_t seg_end = min(s1, (int64_t)(rb + 1) * nk);
#pragma unroll
    for (int i = 0; i < S2_TPW; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) { acc[i][m][r] = 0.f; acci[i][m][r] = 0; }
    const int row_g = rb * S2_ROWS + 64 * rg;  // first row of this warp's row group
    // FP8 scale row of each tile's n-block (block_n >= 16 may split a row group)
    const uint8_t* sc_row[S2_TPW];
#pragma unroll
    for (int ti = 0; ti < S2_TPW; ++ti) sc_row[ti] = nullptr;
    if constexpr (FMT == FMT_FP8) {
#pragma unroll
      for (int ti = 0; ti < S2_TPW; ++ti) {
        const int nb = min(row_g + 16 * ti, a.N - 1) / a.block_n;
        sc_row[ti] = fp8sc + (int64_t)(nb - (rb_first * S2_ROWS) / a.block_n) * a.lds;
      }
    }
    for (; s < seg_end; ++s) {
      const int i = (int)(s - s0);
      const int slot = i % S;
      int got = 0;
      if (lane == 0 && ok) got = tc::mbar_wait(&full[slot], (uint32_t)(i / S) & 1, lim, abort);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        // timed out (or another role did): stop computing but keep walking the units, so
        // every consumer warp still reaches the same named barriers below
        if (lane == 0 && ok) fail();
        ok = false;
        continue;
      }
      const int kt = (int)(s % nk);
      const uint32_t st = tc::smem_u32(smem + (size_t)slot * STAGE);
      const uint32_t xt = st + W_BYTES;
      // weight fragments of the warp's 4 tiles x 2 chunks: q[i][0..3] = (rows g, chunk c),
      // (g+8, c), (g, c+1), (g+8, c+1) of tile i, c = 2*kq
      uint32_t q[S2_TPW][4];
#pragma unroll
      for (int ti = 0; ti < S2_TPW; ++ti)
        ldmatrix_x4(st + sw128(16 * (S2_TPW * rg + ti) + lrow, (2 * kq + lchk) * 16), q[ti][0], q[ti][1], q[ti][2],
                    q[ti][3]);
      if constexpr (FMT == FMT_MXFP4) {
        // activation fragments of the two chunks (each 32 K = one scale group), both halves
        uint2 xv[2][2][MT];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const int kl = 32 * (2 * kq + j) + 8 * t + 4 * h;
              xv[j][h][m] = lds64(xt + (kl >> 6) * X_BOX + sw128(g + 8 * m, (kl & 63) * 2));
            }
        // scale bytes 2*kq, 2*kq+1 of rows g and g+8 of each tile
        const uint32_t sbase = st + W_BYTES + Tr::NXB * X_BOX;
        uint32_t sa[S2_TPW], sb[S2_TPW];
#pragma unroll
        for (int ti = 0; ti < S2_TPW; ++ti) {
          const int r0 = 16 * (S2_TPW * rg + ti) + g;
          const uint2 va = lds64(sbase + r0 * 8), vb = lds64(sbase + (r0 + 8) * 8);
          sa[ti] = (kq < 2 ? va.x : va.y) >> (16 * (kq & 1));
          sb[ti] = (kq < 2 ? vb.x : vb.y) >> (16 * (kq & 1));
        }
        // chunk by chunk: MMAs of the 4 tiles, then the per-row scale fold of that chunk
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float blk[S2_TPW][MT][4];
#pragma unroll
          for (int ti = 0; ti < S2_TPW; ++ti) {
#pragma unroll
            for (int m = 0; m < MT; ++m) blk[ti][m][0] = blk[ti][m][1] = blk[ti][m][2] = blk[ti][m][3] = 0.f;
            const uint32_t qa = q[ti][2 * j], qb = q[ti][2 * j + 1];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t a0 = e2m1x2_to_f16x2(qa >> (16 * h));
              const uint32_t a2 = e2m1x2_to_f16x2(qa >> (16 * h + 8));
              const uint32_t a1 = e2m1x2_to_f16x2(qb >> (16 * h));
              const uint32_t a3 = e2m1x2_to_f16x2(qb >> (16 * h + 8));
#pragma unroll
              for (int m = 0; m < MT; ++m) mma_f16_16816(blk[ti][m], a0, a1, a2, a3, xv[j][h][m].x, xv[j][h][m].y);
            }
          }
          if (j == 1) {  // every shared-memory fragment has been consumed: hand the stage back
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&empty[slot]);
          }
#pragma unroll
          for (int ti = 0; ti < S2_TPW; ++ti) {
            const float fa = ue8m0_to_f32(sa[ti] >> (8 * j)), fb = ue8m0_to_f32(sb[ti] >> (8 * j));
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              acc[ti][m][0] = fmaf(blk[ti][m][0], fa, acc[ti][m][0]);
              acc[ti][m][1] = fmaf(blk[ti][m][1], fa, acc[ti][m][1]);
              acc[ti][m][2] = fmaf(blk[ti][m][2], fb, acc[ti][m][2]);
              acc[ti][m][3] = fmaf(blk[ti][m][3], fb, acc[ti][m][3]);
            }
          }
        }
      } else {
        uint2 xv[2][MT];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const int kl = 16 * (2 * kq + j) + 4 * t;
            xv[j][m] = lds64(xt + (kl >> 6) * X_BOX + sw128(g + 8 * m, (kl & 63) * 2));
          }
        float blk[S2_TPW][MT][4];
#pragma unroll
        for (int ti = 0; ti < S2_TPW; ++ti) {
#pragma unroll
          for (int m = 0; m < MT; ++m) blk[ti][m][0] = blk[ti][m][1] = blk[ti][m][2] = blk[ti][m][3] = 0.f;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t qa = q[ti][2 * j], qb = q[ti][2 * j + 1];
            uint32_t a0, a1, a2, a3;
            if constexpr (FMT == FMT_INT8) {
              s8x4_to_f16x2x2(qa, a0, a2);
              s8x4_to_f16x2x2(qb, a1, a3);
            } else {
              a0 = e4m3x2_to_f16x2((uint16_t)(qa & 0xFFFFu));
              a2 = e4m3x2_to_f16x2((uint16_t)(qa >> 16));
              a1 = e4m3x2_to_f16x2((uint16_t)(qb & 0xFFFFu));
              a3 = e4m3x2_to_f16x2((uint16_t)(qb >> 16));
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) mma_f16_16816(blk[ti][m], a0, a1, a2, a3, xv[j][m].x, xv[j][m].y);
          }
        }
        // every shared-memory fragment has been consumed: hand the stage back before folding
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[slot]);
        if constexpr (FMT == FMT_INT8) {
          // each tile's chain sums 2 x 16 products of at most 127 x 127: exact in fp32
#pragma unroll
          for (int ti = 0; ti < S2_TPW; ++ti)
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
              for (int r = 0; r < 4; ++r) acci[ti][m][r] += __float2int_rn(blk[ti][m][r]);
        } else if (kt * 128 + 32 * kq < a.K) {  // a K tail past the last block has no scale
          const int kb = (kt * 128 + 32 * kq) / a.block_k;
#pragma unroll
          for (int ti = 0; ti < S2_TPW; ++ti) {
            const float f = ue8m0_to_f32(sc_row[ti][kb]);
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
              for (int r = 0; r < 4; ++r) acc[ti][m][r] = fmaf(blk[ti][m][r], f, acc[ti][m][r]);
          }
        }
      }
    }

    // ------------------------------------------------------------ row-block (segment) end
    // the four K quarters of each row group add up: quarters 1..3 hand their sums to quarter 0
    if (!lead) {
      float* xs = xchg + (((rg * (S2_KQ - 1) + (kq - 1)) * S2_TPW) * 32 + lane) * 4 * MT;
#pragma unroll
      for (int ti = 0; ti < S2_TPW; ++ti)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int r = 0; r < 4; ++r)
            xs[ti * 32 * 4 * MT + m * 4 + r] = kInt ? __int_as_float(acci[ti][m][r]) : acc[ti][m][r];
    }
    consumer_sync();
    float res[S2_TPW][MT][4];
#pragma unroll
    for (int ti = 0; ti < S2_TPW; ++ti)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) res[ti][m][r] = kInt ? __int_as_float(acci[ti][m][r]) : acc[ti][m][r];
    if (lead) {
#pragma unroll
      for (int q3 = 0; q3 < S2_KQ - 1; ++q3) {
        const float* xs = xchg + (((rg * (S2_KQ - 1) + q3) * S2_TPW) * 32 + lane) * 4 * MT;
#pragma unroll
        for (int ti = 0; ti < S2_TPW; ++ti)
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const float o = xs[ti * 32 * 4 * MT + m * 4 + r];
              res[ti][m][r] = kInt ? __int_as_float(__float_as_int(res[ti][m][r]) + __float_as_int(o)) : res[ti][m][r] + o;
            }
      }
    }
    consumer_sync();  // the exchange slots are free again
    const int kt_end = (int)(seg_end - (int64_t)rb * nk);
    if (!(kt0 == 0 && kt_end == nk)) {
      const int cf = s2_cta_of((int64_t)rb * nk, T, G);
      if (c == cf) {
        // this CTA settles the block after its last unit (this is its last segment)
#pragma unroll
        for (int ti = 0; ti < S2_TPW; ++ti)
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < 4; ++r) own[ti][m][r] = res[ti][m][r];
        settle_rb = rb;
        continue;
      }
      // another CTA settles it: store the partial sums, then count in with release order
      if (lead) {
        float* pb = a.part + ((int64_t)rb * a.maxseg + (c - cf)) * 16 * S2_ROWS;
#pragma unroll
        for (int ti = 0; ti < S2_TPW; ++ti)
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int col = 2 * t + (r & 1) + 8 * m;
              const int rl = 16 * (S2_TPW * rg + ti) + g + (r >= 2 ? 8 : 0);
              pb[col * S2_ROWS + rl] = res[ti][m][r];
            }
      }
      __threadfence();
      consumer_sync();
      if (threadIdx.x == 0) atomicAdd(&a.tickets[rb], 1u);
      continue;
    }
    // ------------------------------------------------------------ epilogue (whole row block)
    if (lead) {
#pragma unroll
      for (int ti = 0; ti < S2_TPW; ++ti) {
        const int row0 = row_g + 16 * ti + g;
        float rf[2] = {1.f, 1.f}, rbv[2] = {0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = min(row0 + 8 * e, a.N - 1);
          if (kInt) rf[e] = a.w_scale[a.w_scale_len > 1 ? row : 0];
          if (a.bias) rbv[e] = bf16_bits_to_f32(a.bias[row]);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int col = 2 * t + (r & 1) + 8 * m;
            const int row = row0 + (r >= 2 ? 8 : 0);
            if (row >= a.N || col >= a.M) continue;
            uint16_t yb;
            if constexpr (kInt) {
              const int32_t v = __float_as_int(res[ti][m][r]);
              if (a.acc_out) a.acc_out[(int64_t)col * a.N + row] = v;
              yb = f32_to_bf16_rn(__fmul_rn(__fmul_rn((float)v, colf[m][r & 1]), rf[r >> 1]));
            } else {
              yb = f32_to_bf16_rn(res[ti][m][r] * colf[m][r & 1]);
            }
            if (a.bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + rbv[r >> 1]);
            a.y[(int64_t)col * a.ldy + row] = yb;
          }
      }
    }
  }

  // -------------------------------------------------------------- settle the shared block
  if (settle_rb >= 0) {
    const int rb = settle_rb;
    const int cl = s2_cta_of((int64_t)rb * nk + nk - 1, T, G);
    const int count = cl - c + 1;
    // the other CTAs' partial sums: wait (bounded) until all count-1 of them are in
    if (threadIdx.x == 0) {
      uint32_t n = 0;
      while (true) {
        unsigned v;
        asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(a.tickets + rb) : "memory");
        if (v >= (unsigned)(count - 1)) break;
        if (++n > lim) {
          fail();
          break;
        }
        __nanosleep(64);
      }
    }
    consumer_sync();
    if (lead) {
      const float* pb = a.part + (int64_t)rb * a.maxseg * 16 * S2_ROWS;
      const int row_g = rb * S2_ROWS + 64 * rg;
#pragma unroll
      for (int ti = 0; ti < S2_TPW; ++ti) {
        const int row0 = row_g + 16 * ti + g;
        float rf[2] = {1.f, 1.f}, rbv[2] = {0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = min(row0 + 8 * e, a.N - 1);
          if (kInt) rf[e] = a.w_scale[a.w_scale_len > 1 ? row : 0];
          if (a.bias) rbv[e] = bf16_bits_to_f32(a.bias[row]);
        }
        // slot 0 is this CTA (registers); slots 1..count-1 the later CTAs, loaded together
        float v[MT][4][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int col = 2 * t + (r & 1) + 8 * m;
            const int rl = 16 * (S2_TPW * rg + ti) + g + (r >= 2 ? 8 : 0);
            v[m][r][0] = own[ti][m][r];
#pragma unroll
            for (int u = 1; u < 4; ++u)
              v[m][r][u] = (u < count) ? __ldcg(pb + ((int64_t)u * 16 + col) * S2_ROWS + rl) : 0.f;
          }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int col = 2 * t + (r & 1) + 8 * m;
            const int rl = 16 * (S2_TPW * rg + ti) + g + (r >= 2 ? 8 : 0);
            float sum = 0.f;
            int sumi = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (kInt) sumi += __float_as_int(v[m][r][u]); else sum += v[m][r][u];
            }
            for (int sg = 4; sg < count; ++sg) {  // a row block spread over more than 4 CTAs
              const float x = __ldcg(pb + ((int64_t)sg * 16 + col) * S2_ROWS + rl);
              if (kInt) sumi += __float_as_int(x); else sum += x;
            }
            const int row = row0 + (r >= 2 ? 8 : 0);
            if (row >= a.N || col >= a.M) continue;
            uint16_t yb;
            if constexpr (kInt) {
              if (a.acc_out) a.acc_out[(int64_t)col * a.N + row] = sumi;
              yb = f32_to_bf16_rn(__fmul_rn(__fmul_rn((float)sumi, colf[m][r & 1]), rf[r >> 1]));
            } else {
              yb = f32_to_bf16_rn(sum * colf[m][r & 1]);
            }
            if (a.bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + rbv[r >> 1]);
            a.y[(int64_t)col * a.ldy + row] = yb;
          }
      }
    }
    if (threadIdx.x == 0) a.tickets[rb] = 0;  // ready for the next call
  }
}

}  // namespace ql
