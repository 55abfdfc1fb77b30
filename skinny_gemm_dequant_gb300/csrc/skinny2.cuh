// Persistent, TMA-fed skinny GEMM (M <= 16 tokens) for INT8, FP8-block and MXFP4 weights.
//
// Work: the weight matrix is cut into units of (128-row block, 256 weight bytes of K).  The
// units, ordered row block by row block, are split into one contiguous range per CTA, one CTA
// per SM, so every SM streams the same number of weight bytes (no wave tail).  A row block split
// between CTAs cf..cl is settled by cf, the CTA holding its first unit: those units are the last
// ones cf streams, while cf+1..cl reach theirs earlier, store their partial sums and count
// themselves in (release); cf waits for the count (bounded), adds the partials in CTA order to
// its own and writes the outputs, so results do not depend on timing.
//
// Activations: the per-token preparation (INT8 quantisation, or the f16 image of bf16 values)
// is part of this kernel, so a call is one launch.  After the grid-dependency wait, the
// consumer warps of CTAs 0..M*copies-1 each write one (token, copy) row of an f16 image in
// global memory, zero-padded to whole units, and count it in on a release counter; every
// producer acquires the full count (bounded wait) before its first activation load.  The
// weight stream does not wait: producers start loading weights as soon as the CTA starts,
// which, with programmatic dependent launch, overlaps the previous kernel's last CTAs.  The
// image is kept in several copies (CTA c reads copy c % copies) to spread the L2 traffic.
//
// Inside a CTA, warp 8 is the producer.  It keeps a ring of stages in flight; a stage holds one
// unit and is filled by two TMA operations: the weights as one 3D box (128 rows x two 128-byte
// K chunks, 32 KB) and the matching activations as one 4D box, plus (MXFP4) the unit's per-32
// scale bytes by cp.async.  The TMA unit streams HBM at close to its peak only with large
// operations: a 16 KB box per operation, or extra small boxes beside it, leave it well short.
// A unit holding the ragged end of a row (K bytes not a multiple of 128) is loaded a chunk at
// a time as 2D boxes, whose out-of-range bytes the TMA unit fills with zeros.
//
// Warps 0..7 consume, each a 16-row tile of the unit over its two chunks: ldmatrix gives each
// thread 4 weight bytes of every 16-byte piece for rows g and g+8, converted to f16 in
// registers and fed to the warp MMA m16n8k16 (f32 accumulate) against the activations.  Each
// MMA draws all its K values from one 16-byte piece, i.e. from one 32-element MXFP4 scale
// group, so scales fold exactly per piece (per 64 K inside one FP8 block; exact integers for
// INT8).
#pragma once
#include "common.cuh"
#include "tc_ptx.cuh"

namespace ql {

constexpr int S2_CONSUMERS = 8;             // consumer warps, one 16-row tile each
constexpr int S2_THREADS = 32 * (S2_CONSUMERS + 1);
constexpr int S2_ROWS = 16 * S2_CONSUMERS;  // 128 weight rows per unit
constexpr int S2_CHUNKS = 2;                // 128-byte K chunks per unit
constexpr int S2_WB = 128 * S2_CHUNKS;      // weight bytes per row per unit

struct Skinny2Args {
  int M, N, K;
  int wbytes;      // weight bytes of one row that hold K (K, or K/2 for MXFP4)
  int nk;          // units per row block
  int64_t total;   // row blocks x nk
  int maxseg;      // partial slots per row block
  const uint8_t* wsb;  // FP8: UE8M0 grid [ceil(N/bn), lds]; MXFP4: UE8M0 [N, lds]
  int64_t lds;
  int block_n, block_k;
  int bk_shift;          // log2(block_k) (FP8: block_k is a power of two)
  const float* w_scale;  // INT8 per-channel / per-tensor scales
  int w_scale_len;
  // activations and their preparation (done inside this kernel, see s2_prepare)
  const uint16_t* x;      // bf16 [M, ldx]
  int64_t ldx;
  uint16_t* x16;          // f16 image [xcopies][M][kpad] (codes for INT8, x * 2^-p otherwise)
  int64_t kpad;           // K rounded up to whole units
  float* tokf;            // per token: INT8 x_s, bf16 paths 2^p (undone in the epilogue)
  int8_t* xq_dbg;         // optional INT8 codes [M, K]
  float* xs_dbg;          // optional INT8 x_s [M]
  unsigned* ready;        // image rows written so far (release); back to 0 at kernel end
  unsigned* done;         // producers past the hand-off; the last one resets both counters
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
  static constexpr int KPC = (FMT == FMT_MXFP4) ? 256 : 128;  // K elements per 128-byte chunk
  static constexpr int KPU = KPC * S2_CHUNKS;                  // K elements per unit
  static constexpr int NXB = KPU / 64;                         // 64-element activation slabs per unit
  static constexpr int SCB = (FMT == FMT_MXFP4) ? S2_ROWS * 8 * S2_CHUNKS : 0;  // scale bytes per unit
};

// resident CTAs per SM: more warps per scheduler hide the consumers' dependency chains
__host__ __device__ constexpr int s2_ctas_per_sm(int mt) { return mt == 1 ? 2 : 1; }

template <int FMT, int MT>
__host__ __device__ constexpr uint32_t s2_stage_bytes() {
  return S2_ROWS * S2_WB + S2Traits<FMT>::NXB * (8 * MT) * 128 + S2Traits<FMT>::SCB;
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
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
// 8-byte copy global -> shared; src_bytes 0 writes zeros and reads nothing
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(tc::smem_u32(bar))
      : "memory");
}
// named barrier of the consumer warps (the producer warp never joins it)
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// K slices per token of the activation image.  Every job reads its token's whole row (for the
// amax): eight readers per row keep the L2 traffic on those lines low while splitting the
// conversion eight ways; fewer when the grid is small.
__host__ __device__ __forceinline__ int s2_slices(int M, int G) {
  const int n = G / M;
  return n < 1 ? 1 : (n > 8 ? 8 : n);
}

// CTA owning unit s when `total` units are split into G contiguous ranges [c*T/G, (c+1)*T/G)
__device__ __forceinline__ int s2_cta_of(int64_t s, int64_t T, int G) {
  return (int)(((s + 1) * G + T - 1) / T) - 1;
}

// swizzled byte offset of (row, byte) inside a TMA tile of 128-byte rows (128B swizzle)
__device__ __forceinline__ uint32_t sw128(int row, int byte) {
  return (uint32_t)(row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15)));
}

__device__ __forceinline__ float bf16x2_absmax(uint32_t w) {
  return fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xFFFF0000u)));
}

// INT8 code of x for the per-token scale s (> 0, normal) with r = RN(1/s): rint(RN(x/s))
// clamped to +-127, bit for bit.  The product y = RN(x*r) is within 127*1.2e-7 < 1.6e-5 of x/s
// and RN(x/s) within 7.7e-6 of it, so rint(y) and rint(RN(x/s)) can only differ when y lies
// within 2.4e-5 of a half-integer; there (rarely) the IEEE quotient is taken instead.
__device__ __forceinline__ float s2_code(float xv, float s, float r) {
  float y = xv * r;
  if (fabsf((y - floorf(y)) - 0.5f) < 6.1e-5f) y = __fdiv_rn(xv, s);
  return fminf(fmaxf(rintf(y), -127.f), 127.f);
}

// Activation image, one job = (token m, slice sl of nsl): the 256 consumer threads of a CTA
// (thread tid) find the token's amax over all of K, then write their slice of the row into
// every copy of the image.  INT8: dynamic per-token quantisation, x_s = amax/127 and codes
// clamp(rint(x/x_s), -127, 127) with IEEE rounding, as exact f16 integers.  bf16 activations:
// f16 image x * 2^-p with p from the token's amax (scaled amax in [2^14, 2^15)), so every bf16
// value keeps its full significand unless it is below 2^-24 of the amax.  Slice 0 also writes
// the per-token factor the epilogue applies (x_s or 2^p) and the INT8 x_s debug output.
template <int FMT>
__device__ void s2_prepare(const Skinny2Args& a, int m, int sl, int nsl, int tid, float* red) {
  constexpr int V = 8;  // 16-byte vectors a thread holds: one pass over x for K <= 256*8*8
  const uint16_t* xr = a.x + (int64_t)m * a.ldx;
  const int nvec = a.K / 8;
  const int v0 = (int)((int64_t)sl * nvec / nsl), v1 = (int)((int64_t)(sl + 1) * nvec / nsl);
  const bool one_pass = nvec <= V * 256;
  uint4 v[V];
  float amax = 0.f;
  if (one_pass) {
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int i = tid + 256 * j;
      v[j] = i < nvec ? *reinterpret_cast<const uint4*>(xr + 8 * i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < V; ++j)
      amax = fmaxf(amax, fmaxf(fmaxf(bf16x2_absmax(v[j].x), bf16x2_absmax(v[j].y)),
                               fmaxf(bf16x2_absmax(v[j].z), bf16x2_absmax(v[j].w))));
  } else {
    for (int i = tid; i < nvec; i += 256) {
      const uint4 u = *reinterpret_cast<const uint4*>(xr + 8 * i);
      amax = fmaxf(amax, fmaxf(fmaxf(bf16x2_absmax(u.x), bf16x2_absmax(u.y)), fmaxf(bf16x2_absmax(u.z), bf16x2_absmax(u.w))));
    }
  }
  amax = warp_max(amax);
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  consumer_sync();
  amax = fmaxf(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])), fmaxf(fmaxf(red[4], red[5]), fmaxf(red[6], red[7])));
  float f, inv = 1.f;  // INT8: f = x_s and inv = RN(1/x_s); else f = 2^p and inv = 2^-p
  bool fast = true;    // INT8: x_s normal, so the reciprocal path is exact (see s2_code)
  if constexpr (FMT == FMT_INT8) {
    f = __fdiv_rn(amax, 127.0f);
    fast = f >= 1.17549435e-38f;
    if (fast) inv = __frcp_rn(f);
  } else {
    int p = 0;
    if (amax > 0.f) p = max((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127, -126) - 14;
    p = max(-100, min(100, p));
    f = __uint_as_float((uint32_t)(127 + p) << 23);
    inv = __uint_as_float((uint32_t)(127 - p) << 23);
  }
  const int64_t cstride = (int64_t)a.M * a.kpad;  // elements between copies
  uint16_t* out = a.x16 + (int64_t)m * a.kpad;
  auto conv = [&](const uint4 u, int i) {
    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
    uint32_t h[4];
    if constexpr (FMT == FMT_INT8) {
      float qv[8];
      uint32_t qb[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xv = (e & 1) ? __uint_as_float(wv[e >> 1] & 0xFFFF0000u) : __uint_as_float(wv[e >> 1] << 16);
        float q = 0.f;
        if (fast)
          q = s2_code(xv, f, inv);
        else if (f > 0.f)
          q = fminf(fmaxf(rintf(__fdiv_rn(xv, f)), -127.f), 127.f);
        qv[e] = q;
        qb[e >> 2] |= ((uint32_t)((int)q & 0xFF)) << (8 * (e & 3));
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = pack_f16x2(qv[2 * j], qv[2 * j + 1]);  // exact: |q| <= 127
      if (a.xq_dbg) *reinterpret_cast<uint2*>(a.xq_dbg + (int64_t)m * a.K + 8 * i) = make_uint2(qb[0], qb[1]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        h[j] = pack_f16x2(__uint_as_float(wv[j] << 16) * inv, __uint_as_float(wv[j] & 0xFFFF0000u) * inv);
    }
    const uint4 hv = make_uint4(h[0], h[1], h[2], h[3]);
    for (int cp = 0; cp < a.xcopies; ++cp) *reinterpret_cast<uint4*>(out + cp * cstride + 8 * i) = hv;
  };
  if (one_pass) {
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int i = tid + 256 * j;
      if (i >= v0 && i < v1) conv(v[j], i);
    }
  } else {
    for (int i = v0 + tid; i < v1; i += 256) conv(*reinterpret_cast<const uint4*>(xr + 8 * i), i);
  }
  if (sl == nsl - 1)  // the tail past K (to whole units) is zero
    for (int i = nvec + tid; i < (int)(a.kpad / 8); i += 256)
      for (int cp = 0; cp < a.xcopies; ++cp) *reinterpret_cast<uint4*>(out + cp * cstride + 8 * i) = make_uint4(0, 0, 0, 0);
  if (sl == 0 && tid == 0) {
    a.tokf[m] = f;
    if (FMT == FMT_INT8 && a.xs_dbg) a.xs_dbg[m] = f;
  }
  consumer_sync();  // red[] is reused by the next job
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* m, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(tc::smem_u32(bar))
      : "memory");
}

// tmW: 3D view {128 bytes, N rows, full 128-byte chunks} (strides ldw, 128), box {128, 128, 2}
// tmW2: 2D view {wbytes, N}, box {128, 128}: units holding a partial chunk
// tmX: 4D view of the activation image {64 f16, M rows, copies, kpad/64}, box {64, Mp, 1, NXB}
//      (rows M..Mp-1 of the box are out of range and read as zeros)
template <int FMT, int MT>
__global__ void __launch_bounds__(S2_THREADS, s2_ctas_per_sm(MT))
    skinny2_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW2,
                   const __grid_constant__ CUtensorMap tmX, const __grid_constant__ Skinny2Args a) {
  using Tr = S2Traits<FMT>;
  constexpr int Mp = 8 * MT;
  constexpr uint32_t W_CHUNK = S2_ROWS * 128;  // one 128-byte chunk of all 128 rows (16 KB)
  constexpr uint32_t W_BYTES = W_CHUNK * S2_CHUNKS;
  constexpr uint32_t X_BOX = Mp * 128;         // one 64-element slab of all token rows
  constexpr uint32_t X_BYTES = Tr::NXB * X_BOX;
  constexpr uint32_t STAGE = s2_stage_bytes<FMT, MT>();
  constexpr bool kInt = (FMT == FMT_INT8);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * STAGE);
  uint64_t* empty = full + S;
  uint8_t* fp8sc = reinterpret_cast<uint8_t*>(empty + S);  // FP8 scale rows of this CTA's row blocks
  __shared__ int s_abort;

  // the next kernel in the stream (the next call's prologue) may launch now: it waits for this
  // grid to finish before it touches memory, and meanwhile the GEMM after it can take each SM
  // this grid leaves and start streaming its own weights
  pdl_launch_dependents();
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
    const int nbr = S2_ROWS / a.block_n + 2;  // n-blocks a 128-row block can touch
    const int rb_last = (int)((s1 - 1) / nk);
    const int nrow_blocks = rb_last - rb_first + 1;
    const int nb0 = (rb_first * S2_ROWS) / a.block_n;
    const int nb_count = min(nrow_blocks * nbr, (int)((a.N + a.block_n - 1) / a.block_n) - nb0);
    for (int i = threadIdx.x; i < nb_count * a.lds; i += blockDim.x) fp8sc[i] = a.wsb[(int64_t)nb0 * a.lds + i];
  }
  __syncthreads();

  if (warp == S2_CONSUMERS) {
    // ------------------------------------------------------------ producer warp
    const int pre = (int)((int64_t)S < s1 - s0 ? (int64_t)S : s1 - s0);
    const int xcp = c % a.xcopies;  // this CTA's copy of the activation image
    const bool whole_chunks = (a.wbytes & 127) == 0;
    const int ksc = a.K / 32;  // MXFP4 scale bytes of a row that belong to K
    bool ok = true;
    const int n_units = (int)(s1 - s0);
    int issued = 0;
    // unit counters kept incrementally: no divisions in the loop
    int rb = rb_first, kt = (int)(s0 - (int64_t)rb_first * nk);
    int slot = 0;
    uint32_t phase = 0;  // (i / S) & 1
    for (int i = 0; i < n_units; ++i) {
      int got = 1;
      if (lane == 0 && i >= S) got = tc::mbar_wait(&empty[slot], phase ^ 1u, lim, abort);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) fail();
        ok = false;
        break;
      }
      const uint32_t st = tc::smem_u32(smem + (size_t)slot * STAGE);
      if (lane == 0) {
        // weights: chunks 2kt, 2kt+1 of rows rb*128.. -> smem [chunk][row][128 B]
        if (whole_chunks || (kt + 1) * S2_WB <= a.wbytes) {
          tc::mbar_arrive_expect_tx(&full[slot], W_BYTES + X_BYTES);
          tma_load_3d(st, &tmW, 0, rb * S2_ROWS, kt * S2_CHUNKS, &full[slot]);
        } else {
          // the row ends inside this unit, off a chunk boundary: a chunk at a time from the 2D
          // view, whose bytes past the end (a whole chunk, possibly) are filled with zeros
          tc::mbar_arrive_expect_tx(&full[slot], W_BYTES + X_BYTES);
          tc::tma_load_2d(smem + (size_t)slot * STAGE, &tmW2, kt * S2_WB, rb * S2_ROWS, &full[slot]);
          tc::tma_load_2d(smem + (size_t)slot * STAGE + W_CHUNK, &tmW2, kt * S2_WB + 128, rb * S2_ROWS, &full[slot]);
        }
        if (i >= pre) {
          tma_load_4d(st + W_BYTES, &tmX, 0, 0, xcp, kt * Tr::NXB, &full[slot]);
        } else if (i == pre - 1) {
          // the activation image is written by this grid's consumer warps: wait (bounded) until
          // all its rows are in, then load the activation tiles of the stages already in flight.
          // On a timeout the status is flagged and the loads still go out, so no stage waits
          // forever.
          // the counters belong to the previous call until its grid is done: wait for it first
          pdl_wait();
          const unsigned need = (unsigned)(a.M * s2_slices(a.M, G));
          for (uint32_t n = 0;; ++n) {
            unsigned v;
            asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(a.ready) : "memory");
            if (v >= need) break;
            if (n >= lim) {
              fail();
              break;
            }
            __nanosleep(32);
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");  // generic writes -> TMA reads
          // the last producer past this point returns both counters to zero for the next call
          if (atomicAdd(a.done, 1u) == (unsigned)G - 1) {
            *a.ready = 0;
            *a.done = 0;
          }
          int ktj = (int)(s0 - (int64_t)rb_first * nk);
          for (int j = 0; j < pre; ++j) {  // pre <= S: stage j is slot j
            const uint32_t stj = tc::smem_u32(smem + (size_t)j * STAGE);
            tma_load_4d(stj + W_BYTES, &tmX, 0, 0, xcp, ktj * Tr::NXB, &full[j]);
            if (++ktj == nk) ktj = 0;
          }
        }
      }
      if constexpr (FMT == FMT_MXFP4) {
        // per-32 scale bytes of the unit: 128 rows x (8 bytes per chunk); bytes past K read as 0
        const uint32_t sc = st + W_BYTES + X_BYTES;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = lane * 4 + (j >> 1), h = j & 1;
          const int n = min(rb * S2_ROWS + r, a.N - 1);
          const int b0 = kt * 16 + h * 8;
          cp_async8(sc + r * 16 + h * 8, a.wsb + (int64_t)n * a.lds + (b0 < ksc ? b0 : 0), b0 < ksc ? 8u : 0u);
        }
        cp_async_mbar_arrive(&full[slot]);
      }
      issued = i + 1;
      if (++kt == nk) {
        kt = 0;
        ++rb;
      }
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (!ok && lane == 0) {
      // no copy may land after the CTA exits: wait for every stage still in flight
      for (int i = max(0, issued - S); i < issued; ++i)
        tc::mbar_wait(&full[i % S], (uint32_t)(i / S) & 1, 1u << 22, nullptr);
    }
    if constexpr (FMT == FMT_MXFP4) asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }

  // -------------------------------------------------------------- consumer warps
  // activations may come from the previous kernel in the stream: wait for it, then write this
  // CTA's rows of the activation image (rows j = c, c + G, ... of M x copies) and count them in
  pdl_wait();
  {
    __shared__ float s_red[S2_CONSUMERS];
    const int nsl = s2_slices(a.M, G);
    const int njobs = a.M * nsl;
    unsigned mine = 0;
    for (int j = c; j < njobs; j += G, ++mine) s2_prepare<FMT>(a, j % a.M, j / a.M, nsl, threadIdx.x, s_red);
    if (mine) {
      // the rows are read by TMA (async proxy) in other CTAs: proxy fence, then one release
      // (cumulative over the CTA's writes, ordered before it by the barrier)
      asm volatile("fence.proxy.async.global;" ::: "memory");
      consumer_sync();
      if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a.ready), "r"(mine) : "memory");
    }
  }
  const int g = lane >> 2, t = lane & 3;
  const int w = warp;  // 16-row tile of the unit
  // per-token epilogue factors of this thread's columns (x_s or 2^p), loaded at the first
  // segment end: a stage has arrived by then, and its activations were loaded only after the
  // image, factors included, was complete
  float colf[MT][2] = {};
  bool have_colf = false;
  // ldmatrix addressing: lane L feeds row 16w + (L & 7) + 8*((L >> 3) & 1) of piece 2p + (L >> 4)
  const int lrow = 16 * w + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int lpc = lane >> 4;
  float acc[MT][4];
  int32_t acci[MT][4];
  float own[MT][4];  // partial sums of the block this CTA settles
  int settle_rb = -1;
  bool ok = true;
  int rb = rb_first;
  int kt = (int)(s0 - (int64_t)rb_first * nk);
  int slot = 0;
  uint32_t phase = 0;
  int left = (int)(s1 - s0);  // units still to consume
  while (left > 0) {
    const int kt0 = kt;
    const int seg_units = min(nk - kt, left);  // this row block's units in the range
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        acc[m][r] = 0.f;
        acci[m][r] = 0;
      }
    const int row_w = rb * S2_ROWS + 16 * w;  // first row of this warp's tile
    const uint8_t* sc_row = nullptr;          // FP8 scale row of this warp's n-block
    if constexpr (FMT == FMT_FP8) {
      const int nb = min(row_w, a.N - 1) / a.block_n;
      sc_row = fp8sc + (int64_t)(nb - (rb_first * S2_ROWS) / a.block_n) * a.lds;
    }
    for (int u = 0; u < seg_units; ++u, ++kt) {
      int got = 0;
      if (lane == 0 && ok) got = tc::mbar_wait(&full[slot], phase, lim, abort);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        // timed out (or another role did): stop computing but keep walking the units, so
        // every consumer warp still reaches the same named barriers below
        if (lane == 0 && ok) fail();
        ok = false;
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
        continue;
      }
      const uint32_t st = tc::smem_u32(smem + (size_t)slot * STAGE);
      const uint32_t xt = st + W_BYTES;
      // INT8: the unit's sums in two fp32 chains; every partial sum is an integer of at most
      // 256 x 127 x 127 < 2^24 in magnitude, so they are exact and convert once per unit
      float ui[2][MT][4];
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int m = 0; m < MT; ++m) ui[e][m][0] = ui[e][m][1] = ui[e][m][2] = ui[e][m][3] = 0.f;
#pragma unroll
      for (int ck = 0; ck < S2_CHUNKS; ++ck) {
        const uint32_t wt = st + ck * W_CHUNK;
        // the chunk's 8 sixteen-byte pieces for this warp's 16 rows (4 ldmatrix.x4):
        // q[p] = (row g, piece 2p), (g+8, 2p), (g, 2p+1), (g+8, 2p+1)
        uint32_t q[4][4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
          ldmatrix_x4(wt + sw128(lrow, (2 * p + lpc) * 16), q[p][0], q[p][1], q[p][2], q[p][3]);
        if constexpr (FMT == FMT_MXFP4) {
          // scale bytes of rows g and g+8 for the chunk's 8 groups
          const uint32_t sbase = st + W_BYTES + X_BYTES;
          const uint2 sa8 = lds64(sbase + (16 * w + g) * 16 + ck * 8);
          const uint2 sb8 = lds64(sbase + (16 * w + g + 8) * 16 + ck * 8);
#pragma unroll
          for (int pc = 0; pc < 8; ++pc) {  // piece = one 32-element scale group
            const uint32_t qa = q[pc >> 1][2 * (pc & 1)], qb = q[pc >> 1][2 * (pc & 1) + 1];
            // this thread's 8 weights of the piece are K 8t..8t+7: the activations of those
            // K are 16 contiguous bytes of the token's row
            const int kx = 32 * pc + 8 * t;  // K within the chunk
            uint4 xv[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m)
              xv[m] = lds128(xt + (4 * ck + (kx >> 6)) * X_BOX + sw128(g + 8 * m, (kx & 63) * 2));
            float blk[MT][4];
#pragma unroll
            for (int m = 0; m < MT; ++m) blk[m][0] = blk[m][1] = blk[m][2] = blk[m][3] = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t a0 = e2m1x2_to_f16x2(qa >> (16 * h));
              const uint32_t a2 = e2m1x2_to_f16x2(qa >> (16 * h + 8));
              const uint32_t a1 = e2m1x2_to_f16x2(qb >> (16 * h));
              const uint32_t a3 = e2m1x2_to_f16x2(qb >> (16 * h + 8));
#pragma unroll
              for (int m = 0; m < MT; ++m)
                mma_f16_16816(blk[m], a0, a1, a2, a3, h ? xv[m].z : xv[m].x, h ? xv[m].w : xv[m].y);
            }
            const float fa = ue8m0_to_f32((pc < 4 ? sa8.x : sa8.y) >> (8 * (pc & 3)));
            const float fb = ue8m0_to_f32((pc < 4 ? sb8.x : sb8.y) >> (8 * (pc & 3)));
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              acc[m][0] = fmaf(blk[m][0], fa, acc[m][0]);
              acc[m][1] = fmaf(blk[m][1], fa, acc[m][1]);
              acc[m][2] = fmaf(blk[m][2], fb, acc[m][2]);
              acc[m][3] = fmaf(blk[m][3], fb, acc[m][3]);
            }
          }
        } else if constexpr (FMT == FMT_INT8) {
#pragma unroll
          for (int pc = 0; pc < 8; ++pc) {
            const uint32_t qa = q[pc >> 1][2 * (pc & 1)], qb = q[pc >> 1][2 * (pc & 1) + 1];
            uint32_t a0, a1, a2, a3;
            s8x4_to_f16x2x2(qa, a0, a2);
            s8x4_to_f16x2x2(qb, a1, a3);
            const int kx = 16 * pc + 4 * t;  // K within the chunk of this thread's 4 weights
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const uint2 xv = lds64(xt + (2 * ck + (kx >> 6)) * X_BOX + sw128(g + 8 * m, (kx & 63) * 2));
              mma_f16_16816(ui[pc & 1][m], a0, a1, a2, a3, xv.x, xv.y);
            }
          }
        } else {
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {  // 64-K halves of the chunk: the FP8 fold granularity
            float blk[2][MT][4];            // two chains so consecutive MMAs are independent
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
              for (int m = 0; m < MT; ++m) blk[e][m][0] = blk[e][m][1] = blk[e][m][2] = blk[e][m][3] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int pc = 4 * hb + j;
              const uint32_t qa = q[pc >> 1][2 * (pc & 1)], qb = q[pc >> 1][2 * (pc & 1) + 1];
              const uint32_t a0 = e4m3x2_to_f16x2((uint16_t)(qa & 0xFFFFu));
              const uint32_t a2 = e4m3x2_to_f16x2((uint16_t)(qa >> 16));
              const uint32_t a1 = e4m3x2_to_f16x2((uint16_t)(qb & 0xFFFFu));
              const uint32_t a3 = e4m3x2_to_f16x2((uint16_t)(qb >> 16));
              const int kx = 16 * pc + 4 * t;  // K within the chunk of this thread's 4 weights
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                const uint2 xv = lds64(xt + (2 * ck + (kx >> 6)) * X_BOX + sw128(g + 8 * m, (kx & 63) * 2));
                mma_f16_16816(blk[j & 1][m], a0, a1, a2, a3, xv.x, xv.y);
              }
            }
            const int k0 = (kt * S2_CHUNKS + ck) * 128 + 64 * hb;  // first K of this half
            // block_k is a power of two; K past the last block (zero weights) has no scale byte
            const float f = k0 < a.K ? ue8m0_to_f32(sc_row[min(k0, a.K - 1) >> a.bk_shift]) : 0.f;
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
              for (int r = 0; r < 4; ++r) acc[m][r] = fmaf(blk[0][m][r] + blk[1][m][r], f, acc[m][r]);
          }
        }
      }
      if constexpr (FMT == FMT_INT8) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int r = 0; r < 4; ++r) acci[m][r] += __float2int_rn(ui[0][m][r] + ui[1][m][r]);
      }
      // every shared-memory fragment of the unit has been read: hand the stage back
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[slot]);
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }
    left -= seg_units;

    // ------------------------------------------------------------ row-block (segment) end
    if (!have_colf) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = 2 * t + e + 8 * m;
          colf[m][e] = col < a.M ? a.tokf[col] : 0.f;
        }
      have_colf = true;
    }
    float res[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) res[m][r] = kInt ? __int_as_float(acci[m][r]) : acc[m][r];
    const int kt_end = kt;
    const int seg_rb = rb;
    rb += 1;  // the next segment (if any) starts a new row block
    kt = 0;
    if (!(kt0 == 0 && kt_end == nk)) {
      const int cf = s2_cta_of((int64_t)seg_rb * nk, T, G);
      if (c == cf) {
        // this CTA settles the block after its last unit (this is its last segment)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int r = 0; r < 4; ++r) own[m][r] = res[m][r];
        settle_rb = seg_rb;
        continue;
      }
      // another CTA settles it: store the partial sums, then count in with release order
      float* pb = a.part + ((int64_t)seg_rb * a.maxseg + (c - cf)) * 16 * S2_ROWS;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int col = 2 * t + (r & 1) + 8 * m;
          const int rl = 16 * w + g + (r >= 2 ? 8 : 0);
          pb[col * S2_ROWS + rl] = res[m][r];
        }
      __threadfence();
      consumer_sync();
      if (threadIdx.x == 0) atomicAdd(&a.tickets[seg_rb], 1u);
      continue;
    }
    // ------------------------------------------------------------ epilogue (whole row block)
    float rowf[2] = {1.f, 1.f}, rowb[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int row = min(row_w + g + 8 * e, a.N - 1);
      if (kInt) rowf[e] = a.w_scale[a.w_scale_len > 1 ? row : 0];
      if (a.bias) rowb[e] = bf16_bits_to_f32(a.bias[row]);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int col = 2 * t + (r & 1) + 8 * m;
        const int row = row_w + g + (r >= 2 ? 8 : 0);
        if (row >= a.N || col >= a.M) continue;
        uint16_t yb;
        if constexpr (kInt) {
          const int32_t v = __float_as_int(res[m][r]);
          if (a.acc_out) a.acc_out[(int64_t)col * a.N + row] = v;
          yb = f32_to_bf16_rn(__fmul_rn(__fmul_rn((float)v, colf[m][r & 1]), rowf[r >> 1]));
        } else {
          yb = f32_to_bf16_rn(res[m][r] * colf[m][r & 1]);
        }
        if (a.bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + rowb[r >> 1]);
        a.y[(int64_t)col * a.ldy + row] = yb;
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
        if (++n > lim || *abort) {
          fail();
          break;
        }
        __nanosleep(64);
      }
    }
    consumer_sync();
    const float* pb = a.part + (int64_t)rb * a.maxseg * 16 * S2_ROWS;
    const int row_w = rb * S2_ROWS + 16 * w;
    float rf[2] = {1.f, 1.f}, rbv[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int row = min(row_w + g + 8 * e, a.N - 1);
      if (kInt) rf[e] = a.w_scale[a.w_scale_len > 1 ? row : 0];
      if (a.bias) rbv[e] = bf16_bits_to_f32(a.bias[row]);
    }
    // slot 0 is this CTA (registers); slots 1..count-1 the later CTAs, added in CTA order,
    // read four slots at a time so the loads of a batch overlap
    float sum[MT][4];
    int32_t sumi[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        sum[m][r] = own[m][r];
        sumi[m][r] = __float_as_int(own[m][r]);
      }
    for (int u0 = 1; u0 < count; u0 += 4) {
      float v[MT][4][4];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int col = 2 * t + (r & 1) + 8 * m;
          const int rl = 16 * w + g + (r >= 2 ? 8 : 0);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            v[m][r][u] = (u0 + u < count) ? __ldcg(pb + ((int64_t)(u0 + u) * 16 + col) * S2_ROWS + rl) : 0.f;
        }
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (u0 + u >= count) break;
            if (kInt)
              sumi[m][r] += __float_as_int(v[m][r][u]);
            else
              sum[m][r] += v[m][r][u];
          }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int col = 2 * t + (r & 1) + 8 * m;
        const int row = row_w + g + (r >= 2 ? 8 : 0);
        if (row >= a.N || col >= a.M) continue;
        uint16_t yb;
        if constexpr (kInt) {
          if (a.acc_out) a.acc_out[(int64_t)col * a.N + row] = sumi[m][r];
          yb = f32_to_bf16_rn(__fmul_rn(__fmul_rn((float)sumi[m][r], colf[m][r & 1]), rf[r >> 1]));
        } else {
          yb = f32_to_bf16_rn(sum[m][r] * colf[m][r & 1]);
        }
        if (a.bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + rbv[r >> 1]);
        a.y[(int64_t)col * a.ldy + row] = yb;
      }
    if (threadIdx.x == 0) a.tickets[rb] = 0;  // ready for the next call
  }
}

}  // namespace ql
