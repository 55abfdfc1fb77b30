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
// consumer warps of CTAs 0..M*slices-1 each take one (token, K slice) job: read the token's row
// (for its amax), write the slice of its f16 image row in global memory into every copy of the
// image (zero-padded to whole units), and count the job in on a release counter; every producer
// acquires the full count (bounded wait) before its first activation load.  The weight stream
// does not wait: producers start loading weights as soon as the CTA starts (MoE gate_up: once
// it has routed), which, with programmatic dependent launch, overlaps the previous kernel's last
// CTAs.  The image is kept in two copies (CTA c reads copy c % copies) to spread the L2 traffic.
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
#include "route.cuh"
#include "tc_ptx.cuh"

namespace ql {

constexpr int S2_CONSUMERS = 8;             // consumer warps, one 16-row tile each
constexpr int S2_THREADS = 32 * (S2_CONSUMERS + 1);
constexpr int S2_ROWS = 16 * S2_CONSUMERS;  // 128 weight rows per unit
constexpr int S2_CHUNKS = 2;                // 128-byte K chunks per unit
constexpr int S2_WB = 128 * S2_CHUNKS;      // weight bytes per row per unit

// what one launch computes: a dense linear layer, or one of the two expert GEMVs of the MoE
// (S2_DENSE_LOCAL: a dense layer whose CTAs build their own activation image, s2_local_image)
enum { S2_DENSE = 0, S2_MOE_GU = 1, S2_MOE_DN = 2, S2_DENSE_LOCAL = 3 };

struct Skinny2Args {
  int M, N, K;     // N: weight rows (per expert for the MoE kinds); M: tokens
  int wbytes;      // weight bytes of one row that hold K (K, or K/2 for MXFP4)
  int nk;          // units per row block
  int nb;          // 128-row blocks (per expert)
  int64_t total;   // dense: row blocks x nk (MoE: the distinct-expert count decides, on the device)
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
  int img_rows;           // rows of one image copy: M (dense, MoE gate_up) or slots x slot_rows (down)
  float* tokf;            // per token: INT8 x_s, bf16 paths 2^p (undone in the epilogue)
  int8_t* xq_dbg;         // optional INT8 codes [M, K]
  float* xs_dbg;          // optional INT8 x_s [M]
  unsigned* ready;        // image rows written so far (release); back to 0 at kernel end
  unsigned* done;         // producers past the hand-off; the last one resets both counters
  uint16_t* y;
  int64_t ldy;
  const uint16_t* bias;
  int32_t* acc_out;
  float* part;        // [CTAs][16][128] partial sums (fp32 or int32 bits): each CTA posts at most one
  unsigned* tickets;  // [row blocks] arrival counts of the partial sums
  // MoE routing: the gate_up launch routes (every CTA, identically) and its CTA 0 writes the
  // results below, which the down launch and the combine read; experts sit in distinct-expert
  // slots in increasing id
  const uint16_t* logits;  // bf16 [M, E] router logits, or null with ids_in / w_in given
  const int32_t* ids_in;   // [M*topk] given expert ids
  const float* w_in;       // [M*topk] given routing weights
  int renorm;              // renormalise the top-k probabilities to sum 1
  int32_t* ids_dbg;        // optional copies of ids / weights
  float* w_dbg;
  float* wts;              // [M*topk] routing weights
  int32_t* nuniq;          // distinct experts
  int32_t* uniq;           // [slots] expert of each slot
  int32_t* offsets;        // [E+1] dispatch positions of each expert's (token, slot) pairs
  int32_t* pairs;          // [pairs] pair index m*topk+j at each dispatch position
  int32_t* ids;            // [M*topk] expert of each pair (-1: none)
  int32_t* rows;           // [pairs] down-stage image row of each dispatch position (-1: none)
  int topk, E;
  int slot_rows;           // MoE down: image rows per expert slot (8*MT)
  int64_t s_estride;       // MXFP4 scale bytes per expert
  float* gu;               // gate_up out / down in: [M*topk][2I] fp32 raw sums (gate rows, then up)
  int I;                   // expert intermediate size
  uint16_t* h_dbg;         // optional h = bf16(silu(g) * u) [M*topk][I]
  float act_alpha, act_limit;  // expert activation silu(alpha * min(g, limit)) * clamp(u, +-limit)
  float* o;                // down out: [M*topk][H] fp32
  uint32_t* status;
  uint32_t wait_limit;
  int stages;
  int xcopies;  // copies of the activation image; CTA c reads copy c % xcopies (spreads L2 load)
  // INT8 dense layers of up to 4 tokens: every output is settled by the contribution that
  // completes it (cells, see s2_cell_*)
  unsigned long long* cells;  // [M][N]: (units added << 48) + exact int32 sum
  int cells_clean;            // 1: the cells start at zero and each is reset after it settles;
                              // 0: the activation jobs zero them before the hand-off
  // K shards of a row-parallel layer: INT8 quantises with the caller's per-token amax (taken
  // over the whole row) and may leave y null (acc_out only); FP8 / MXFP4 write fp32 partial
  // sums to y32 (no bias) instead of bf16 y
  const float* amax_in;
  float* y32;
  int64_t ldy32;
  // dense layers with few tokens: each CTA builds the image of its own units in shared memory
  // (s2_local_image, launch kind S2_DENSE_LOCAL) instead of the grid sharing one in global memory
  int local;        // the host asks for it
  int local_bytes;  // shared memory of the local image (behind the ring's barriers)
};

// A self-settling output cell of the INT8 kernel: a 64-bit word holding (units << 48) + s,
// where s is the exact int32 sum of the partial dot products added so far (two's complement
// across the word: |s| < 2^31 < 2^47).  Every contribution is one atomic add of
// (n << 48) + partial, n = the units it covers, so the contribution whose add brings the count
// to the row block's unit count holds the complete sum in the add's result, and settles the
// output itself: no CTA waits for another, and the order of arrival cannot change the sum.
__host__ __device__ __forceinline__ unsigned long long s2_cell_add(int units, int32_t partial) {
  return ((unsigned long long)units << 48) + (unsigned long long)(long long)partial;
}
__host__ __device__ __forceinline__ int s2_cell_units(unsigned long long v) { return (int)((v + (1ull << 47)) >> 48); }
__host__ __device__ __forceinline__ int32_t s2_cell_sum(unsigned long long v) {
  return (int32_t)(long long)(v - ((unsigned long long)s2_cell_units(v) << 48));
}

template <int FMT>
struct S2Traits {
  static constexpr int KPC = (FMT == FMT_MXFP4) ? 256 : (FMT == FMT_BF16 ? 64 : 128);  // K per 128-byte chunk
  static constexpr int KPU = KPC * S2_CHUNKS;                  // K elements per unit
  static constexpr int NXB = KPU / 64;                         // 64-element activation slabs per unit
  static constexpr int SCB = (FMT == FMT_MXFP4) ? S2_ROWS * 8 * S2_CHUNKS : 0;  // scale bytes per unit
};

// resident CTAs per SM: more warps per scheduler hide the consumers' dependency chains.  Two,
// except for 9..16 tokens (MT = 2) with INT8, FP8 or BF16 weights: the MXFP4 consumers are
// compute-bound, so their MT = 2 kernels gain from a second CTA's warps (-3.5 % on the MoE
// decode bench), while the others lose 1.6 % (INT8 decode bench) to the halved ring per CTA.
__host__ __device__ constexpr int s2_ctas_per_sm(int fmt, int mt) { return mt == 1 || fmt == FMT_MXFP4 ? 2 : 1; }

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
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
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

// K slices per token of the activation image, at most `cap` (fewer when the grid is small).
// Every job reads its token's whole row (for the amax) and converts one slice, so more slices
// shorten the longest job.  Measured: a dense layer's hand-off gains from 32 (INT8 decode bench
// -1.2 % against 8, FP8 unchanged); the MoE launches, whose jobs run beside routing or the down launch's
// gathers, lose 0.3 % and keep 8.
__host__ __device__ __forceinline__ int s2_slices(int M, int G, int cap) {
  const int n = G / M;
  return n < 1 ? 1 : (n > cap ? cap : n);
}

// CTA owning unit s when `total` units are split into G contiguous ranges [c*T/G, (c+1)*T/G)
__device__ __forceinline__ int s2_cta_of(int64_t s, int64_t T, int G) {
  return (int)(((s + 1) * G + T - 1) / T) - 1;
}

// MMA token column j (0..7 within each group of 8) reads activation row rho(j), the 3-bit bit
// reversal of j.  A quarter warp (128-bit loads) or half warp (64-bit loads) then reads rows
// whose 128B-swizzle patterns differ in the bits that separate its 16-byte chunks, so the
// activation loads are free of bank conflicts.  The epilogue maps column j back to token rho(j).
__host__ __device__ __forceinline__ int s2_rho(int j) { return ((j & 1) << 2) | (j & 2) | ((j >> 2) & 1); }

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

// The per-token factors of the activation image from the token's amax.  INT8: f = x_s =
// amax / 127 (IEEE division) and inv = RN(1/x_s), fast when x_s is normal (see s2_code).
// bf16 paths: f = 2^p and inv = 2^-p with p from the amax's exponent (scaled amax in
// [2^14, 2^15)).
template <int FMT>
__device__ __forceinline__ void s2_token_factors(float amax, float& f, float& inv, bool& fast) {
  inv = 1.f;
  fast = true;
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
}

// Eight bf16 values (one 16-byte vector) to their four f16x2 image words: INT8 codes
// clamp(rint(x / x_s), -127, 127) as exact f16 integers (qb: the codes as bytes), or x * 2^-p.
template <int FMT>
__device__ __forceinline__ void s2_conv8(const uint4 u, float f, float inv, bool fast, uint32_t (&h)[4],
                                         uint32_t (&qb)[2]) {
  const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
  qb[0] = qb[1] = 0u;
  if constexpr (FMT == FMT_INT8) {
    float qv[8];
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
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      h[j] = pack_f16x2(__uint_as_float(wv[j] << 16) * inv, __uint_as_float(wv[j] & 0xFFFF0000u) * inv);
  }
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
  constexpr bool kCompact = FMT != FMT_MXFP4;
  const uint16_t* xr = a.x + (int64_t)m * a.ldx;
  const int nvec = a.K / 8;
  const int v0 = (int)((int64_t)sl * nvec / nsl), v1 = (int)((int64_t)(sl + 1) * nvec / nsl);
  const bool one_pass = nvec <= V * 256;
  uint4 v[V];
  float amax = 0.f;
  if (one_pass) {
    // thread tid holds vectors v0 + tid + 256 j (wrapping at the row end): the whole row for the
    // amax, and first the one of the slice it converts, so the conversion below is one copy of
    // its code (this code runs once per call, from a cold instruction cache)
    // (MXFP4 keeps the plain order: its MoE kernels run at the register cap of two CTAs per SM)
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int t = tid + 256 * j;
      int i = kCompact ? v0 + t : t;
      if (kCompact && i >= nvec) i -= nvec;
      v[j] = t < nvec ? *reinterpret_cast<const uint4*>(xr + 8 * i) : make_uint4(0, 0, 0, 0);
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
  if (FMT == FMT_INT8 && a.amax_in) amax = a.amax_in[m];  // a K shard: the whole row's amax, from the caller
  float f, inv;  // INT8: f = x_s and inv = RN(1/x_s); else f = 2^p and inv = 2^-p
  bool fast;     // INT8: x_s normal, so the reciprocal path is exact (see s2_code)
  s2_token_factors<FMT>(amax, f, inv, fast);
  const int64_t cstride = (int64_t)a.img_rows * a.kpad;  // elements between copies
  uint16_t* out = a.x16 + (int64_t)m * a.kpad;
  auto conv = [&](const uint4 u, int i) {
    uint32_t h[4], qb[2];
    s2_conv8<FMT>(u, f, inv, fast, h, qb);
    if (FMT == FMT_INT8 && a.xq_dbg) *reinterpret_cast<uint2*>(a.xq_dbg + (int64_t)m * a.K + 8 * i) = make_uint2(qb[0], qb[1]);
    const uint4 hv = make_uint4(h[0], h[1], h[2], h[3]);
    for (int cp = 0; cp < a.xcopies; ++cp) *reinterpret_cast<uint4*>(out + cp * cstride + 8 * i) = hv;
  };
  if (one_pass && kCompact) {
    if (tid < v1 - v0) conv(v[0], v0 + tid);
    for (int t = tid + 256; t < v1 - v0; t += 256)  // slices above 256 vectors
      conv(*reinterpret_cast<const uint4*>(xr + 8 * (v0 + t)), v0 + t);
  } else if (one_pass) {
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
  if constexpr (FMT == FMT_INT8) {  // this slice of token m's output cells starts at zero
    if (a.cells && !a.cells_clean) {
      const int r0 = (int)((int64_t)sl * a.N / nsl), r1 = (int)((int64_t)(sl + 1) * a.N / nsl);
      for (int r = r0 + tid; r < r1; r += 256) a.cells[(int64_t)m * a.N + r] = 0ull;
    }
  }
  consumer_sync();  // red[] is reused by the next job
}

// The local activation image of a CTA (dense layers with few tokens, a.local): the CTA reads
// its tokens' whole rows for their amax, then writes the image values of the K units it
// streams into shared memory - no image in global memory, no hand-off between CTAs.  The
// CTA's units are n_slots consecutive K units starting at kt0 (wrapping at nk); slot s holds
// unit kt0 + s as NXB slabs of 64 K, each slab M rows of 128 bytes with the 128-byte swizzle
// of a TMA tile (the consumers address it the same way, with row indices clamped to M - 1).
// Also writes the tokens' factors to tokf (shared), the INT8 codes of those units to xq_dbg
// and, in CTA 0, the INT8 x_s to xs_dbg.  All 256 consumer threads call this.
template <int FMT>
__device__ void s2_local_image(const Skinny2Args& a, uint32_t L, int kt0, int n_slots, int tid, float* red,
                               float* tokf) {
  constexpr int KPU = S2Traits<FMT>::KPU, VPU = KPU / 8;  // 8-element vectors per unit
  constexpr int KEEP = 4;  // vectors of the CTA's own units a thread holds (the host keeps n_slots * VPU <= 1024)
  const int nvec = a.K / 8, M = a.M;
  const int nneed = n_slots * VPU;
  const uint32_t slot_bytes = (uint32_t)(S2Traits<FMT>::NXB * M * 128);
  for (int m = 0; m < M; ++m) {
    const uint16_t* xr = a.x + (int64_t)m * a.ldx;
    // the vectors of this CTA's units (thread tid: t = tid + 256 j) and, at the same time, the
    // whole row for the amax: every load goes out before any result is used (one round trip)
    uint4 keep[KEEP];
#pragma unroll
    for (int j = 0; j < KEEP; ++j) {
      const int t = tid + 256 * j;
      int kt = kt0 + t / VPU;
      if (kt >= a.nk) kt -= a.nk;
      const int vi = kt * VPU + t % VPU;
      keep[j] = (t < nneed && vi < nvec) ? *reinterpret_cast<const uint4*>(xr + 8 * vi) : make_uint4(0, 0, 0, 0);
    }
    float amax = 0.f;
#pragma unroll 4
    for (int i = tid; i < nvec; i += 256) {
      const uint4 u = *reinterpret_cast<const uint4*>(xr + 8 * i);
      amax = fmaxf(amax, fmaxf(fmaxf(bf16x2_absmax(u.x), bf16x2_absmax(u.y)), fmaxf(bf16x2_absmax(u.z), bf16x2_absmax(u.w))));
    }
    amax = warp_max(amax);
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    consumer_sync();
    amax = fmaxf(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])), fmaxf(fmaxf(red[4], red[5]), fmaxf(red[6], red[7])));
    if (FMT == FMT_INT8 && a.amax_in) amax = a.amax_in[m];  // a K shard: the whole row's amax
    float f, inv;
    bool fast;
    s2_token_factors<FMT>(amax, f, inv, fast);
    if (tid == 0) {
      tokf[m] = f;
      if (FMT == FMT_INT8 && a.xs_dbg && blockIdx.x == 0) a.xs_dbg[m] = f;
    }
    // one copy of the conversion code (it runs once per call, from a cold instruction cache):
    // the held vectors are picked by selects, not by unrolling the loop
#pragma unroll 1
    for (int j = 0; j < KEEP; ++j) {
      const int t = tid + 256 * j;
      if (t >= nneed) break;
      uint4 u = keep[0];
#pragma unroll
      for (int q = 1; q < KEEP; ++q)
        if (j == q) u = keep[q];
      const int sl = t / VPU, c8 = t - sl * VPU;
      int kt = kt0 + sl;
      if (kt >= a.nk) kt -= a.nk;
      const int k = kt * KPU + c8 * 8;
      uint32_t h[4], qb[2];
      s2_conv8<FMT>(u, f, inv, fast, h, qb);
      if (FMT == FMT_INT8 && a.xq_dbg && k < a.K)
        *reinterpret_cast<uint2*>(a.xq_dbg + (int64_t)m * a.K + k) = make_uint2(qb[0], qb[1]);
      const int jj = c8 >> 3, c16 = c8 & 7;  // slab, 16-byte chunk of the 128-byte row
      const uint32_t dst = L + (uint32_t)sl * slot_bytes + (uint32_t)(jj * M + m) * 128u + (uint32_t)((c16 ^ (m & 7)) << 4);
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                   : "memory");
    }
    consumer_sync();  // red[] is reused by the next token
  }
}

// The same image for 2..8 tokens in one pass over the rows: thread tid reads token tid % M
// (eight of its vectors in flight at a time) for the token's amax, and stores the vectors of
// this CTA's own units raw into their image slots on the way; the per-token maxima meet in
// shared memory, and the slots are then converted in place (a bf16 vector and its f16 image
// are both 16 bytes).  Token by token (s2_local_image) took an L2 round trip and two barriers
// per token.  red: >= 24 floats, red[0, 8) zero on entry (per-token amax bits, then factors).
template <int FMT>
__device__ void s2_local_image_multi(const Skinny2Args& a, uint32_t L, int kt0, int n_slots, int tid, float* red,
                                     float* tokf) {
  constexpr int KPU = S2Traits<FMT>::KPU, VPU = KPU / 8;
  const int nvec = a.K / 8, M = a.M, nk = a.nk;
  const uint32_t slot_bytes = (uint32_t)(S2Traits<FMT>::NXB * M * 128);
  auto slot_addr = [&](int sl, int c8, int m) {
    const int jj = c8 >> 3, c16 = c8 & 7;  // slab, 16-byte chunk of the 128-byte row
    return L + (uint32_t)sl * slot_bytes + (uint32_t)(jj * M + m) * 128u + (uint32_t)((c16 ^ (m & 7)) << 4);
  };
  const int m = tid % M, ti = tid / M, nth = (255 - m) / M + 1;  // this thread's token, rank, peers
  const uint16_t* xr = a.x + (int64_t)m * a.ldx;
  float am = 0.f;
#pragma unroll 1
  for (int i0 = ti; i0 < nvec; i0 += 8 * nth) {
    uint4 u[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = i0 + r * nth;
      if (i < nvec) u[r] = *reinterpret_cast<const uint4*>(xr + 8 * i);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = i0 + r * nth;
      if (i >= nvec) break;
      am = fmaxf(am, fmaxf(fmaxf(bf16x2_absmax(u[r].x), bf16x2_absmax(u[r].y)),
                           fmaxf(bf16x2_absmax(u[r].z), bf16x2_absmax(u[r].w))));
      const int kt = i / VPU, c8 = i - kt * VPU;
      int sl = kt - kt0;
      if (sl < 0) sl += nk;
      if (sl < n_slots)
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(slot_addr(sl, c8, m)), "r"(u[r].x), "r"(u[r].y),
                     "r"(u[r].z), "r"(u[r].w)
                     : "memory");
    }
  }
  // own vectors past the row's end (K not a multiple of the unit): zeros
  for (int t = tid; t < n_slots * VPU; t += 256) {
    const int sl = t / VPU, c8 = t - sl * VPU;
    int kt = kt0 + sl;
    if (kt >= nk) kt -= nk;
    if (kt * VPU + c8 < nvec) continue;
    for (int mm = 0; mm < M; ++mm)
      asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(slot_addr(sl, c8, mm)), "r"(0u) : "memory");
  }
  // non-negative floats order as their bit patterns
  atomicMax(reinterpret_cast<int*>(red) + m, __float_as_int(am));
  consumer_sync();
  if (tid < M) {
    float amax = red[tid];
    if (FMT == FMT_INT8 && a.amax_in) amax = a.amax_in[tid];  // a K shard: the whole row's amax
    float f, inv;
    bool fast;
    s2_token_factors<FMT>(amax, f, inv, fast);
    tokf[tid] = f;
    red[8 + tid] = inv;
    red[16 + tid] = fast ? 1.f : 0.f;
    if (FMT == FMT_INT8 && a.xs_dbg && blockIdx.x == 0) a.xs_dbg[tid] = f;
  }
  consumer_sync();
  // in place: one copy of the conversion code (it runs once per call, from a cold instruction cache)
#pragma unroll 1
  for (int e = tid; e < n_slots * VPU * M; e += 256) {
    const int mm = e % M, t = e / M;
    const int sl = t / VPU, c8 = t - sl * VPU;
    const uint32_t ad = slot_addr(sl, c8, mm);
    uint4 u;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w) : "r"(ad));
    uint32_t h[4], qb[2];
    s2_conv8<FMT>(u, tokf[mm], red[8 + mm], red[16 + mm] != 0.f, h, qb);
    int kt = kt0 + sl;
    if (kt >= nk) kt -= nk;
    const int k = kt * KPU + c8 * 8;
    if (FMT == FMT_INT8 && a.xq_dbg && k < a.K)
      *reinterpret_cast<uint2*>(a.xq_dbg + (int64_t)mm * a.K + k) = make_uint2(qb[0], qb[1]);
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(ad), "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                 : "memory");
  }
  consumer_sync();
}

// MoE down activations, one job = (dispatch position q, slice sl of nsl).  The pair p = m*topk+j
// at position q went to expert e; its gate and up sums g, u (length I) are gu[p].  Its activation
// row is h = bf16(silu(g) * u), or with a clamp bf16(silu(alpha min(g, limit)) clamp(u, +-limit))
// (the expert's intermediate, rounded to bf16 as the pages' BF16
// experts do), written as an f16 image row h * 2^-p (p from the row's amax, as for bf16 inputs)
// at row rows[q] = slot(e) * slot_rows + (q - offsets[e]) of every copy (the routing wrote it);
// slice 0 writes 2^p for the epilogue.  A pair beyond slot_rows of its expert (only possible when a token lists an expert
// twice) gets no row.
__device__ inline void s2_prepare_h(const Skinny2Args& a, int q, int sl, int nsl, int tid, float* red) {
  const int p = a.pairs[q];
  const int r = a.rows[q];  // slot(e) * slot_rows + rank within the expert's pairs, or -1
  const bool has_row = r >= 0;
  const int I = a.I, nvec = I / 8;
  const float* gp = a.gu + (int64_t)p * 2 * I;
  auto hvals = [&](int i, float (&h)[8], uint16_t (&hb)[8]) {
    const float4 g0 = __ldcg(reinterpret_cast<const float4*>(gp + 8 * i));
    const float4 g1 = __ldcg(reinterpret_cast<const float4*>(gp + 8 * i + 4));
    const float4 u0 = __ldcg(reinterpret_cast<const float4*>(gp + I + 8 * i));
    const float4 u1 = __ldcg(reinterpret_cast<const float4*>(gp + I + 8 * i + 4));
    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      hb[k] = f32_to_bf16_rn(swiglu_f32(gv[k], uv[k], a.act_alpha, a.act_limit));
      h[k] = bf16_bits_to_f32(hb[k]);
    }
  };
  float amax = 0.f;
  for (int i = tid; i < nvec; i += 256) {
    float h[8];
    uint16_t hb[8];
    hvals(i, h, hb);
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(h[k]));
  }
  amax = warp_max(amax);
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  consumer_sync();
  amax = fmaxf(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])), fmaxf(fmaxf(red[4], red[5]), fmaxf(red[6], red[7])));
  int pe = 0;
  if (amax > 0.f) pe = max((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127, -126) - 14;
  pe = max(-100, min(100, pe));
  const float inv = __uint_as_float((uint32_t)(127 - pe) << 23);
  const int v0 = (int)((int64_t)sl * nvec / nsl), v1 = (int)((int64_t)(sl + 1) * nvec / nsl);
  const int64_t cstride = (int64_t)a.img_rows * a.kpad;
  uint16_t* out = a.x16 + (int64_t)r * a.kpad;
  for (int i = v0 + tid; i < v1; i += 256) {
    float h[8];
    uint16_t hb[8];
    hvals(i, h, hb);
    if (a.h_dbg) {
      uint32_t w4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) w4[k] = (uint32_t)hb[2 * k] | ((uint32_t)hb[2 * k + 1] << 16);
      *reinterpret_cast<uint4*>(a.h_dbg + (int64_t)p * I + 8 * i) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    if (!has_row) continue;
    uint32_t f4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) f4[k] = pack_f16x2(h[2 * k] * inv, h[2 * k + 1] * inv);
    const uint4 hv = make_uint4(f4[0], f4[1], f4[2], f4[3]);
    for (int cp = 0; cp < a.xcopies; ++cp) *reinterpret_cast<uint4*>(out + cp * cstride + 8 * i) = hv;
  }
  if (has_row && sl == nsl - 1)  // the tail past I (to whole units) is zero
    for (int i = nvec + tid; i < (int)(a.kpad / 8); i += 256)
      for (int cp = 0; cp < a.xcopies; ++cp) *reinterpret_cast<uint4*>(out + cp * cstride + 8 * i) = make_uint4(0, 0, 0, 0);
  if (has_row && sl == 0 && tid == 0) a.tokf[r] = __uint_as_float((uint32_t)(127 + pe) << 23);
  consumer_sync();  // red[] is reused by the next job
}

// MoE routing inside the gate_up launch (softmax top-k, [DSV4] routing and grouped dispatch):
// per token p = softmax(logits) (route_token_warp: fp32 exponentials, a float-float sum), the topk
// experts with the largest logits (equal logits: lower id first) and weights p[ids]
// (renormalised on request); or the given ids and weights.  Then the pairs are grouped by expert
// (increasing id, stable in pair order) and the distinct experts listed in increasing id.  Every
// CTA computes the same routing into its shared memory (ids, first dispatch position per
// expert, distinct experts, their count); CTA 0 also writes it all out.  All threads of the CTA
// call this (E <= 1024, M*topk <= 256).
__device__ inline void s2_route(const Skinny2Args& a, int* s_ids, int* s_cnt, int* s_uniq, int* s_slot, int* s_nu) {
  const int M = a.M, E = a.E, topk = a.topk, P = M * topk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const bool out = blockIdx.x == 0;
  if (a.logits) {
    for (int m = warp; m < M; m += nw) {  // a warp per token
      int id = -1;
      float w = 0.f;
      route_token_warp(a.logits + (int64_t)m * E, E, topk, a.renorm != 0, id, w);
      if (lane < topk) {
        const int pi = m * topk + lane;
        s_ids[pi] = id;
        if (out) {
          a.ids[pi] = id;
          a.wts[pi] = w;
          if (a.ids_dbg) a.ids_dbg[pi] = id;
          if (a.w_dbg) a.w_dbg[pi] = w;
        }
      }
    }
  } else {
    for (int pi = threadIdx.x; pi < P; pi += blockDim.x) {
      int e = a.ids_in[pi];
      if (e < 0 || e >= E) {
        if (out) raise_flag(a.status, 2u);
        e = -1;
      }
      s_ids[pi] = e;
      if (out) {
        a.ids[pi] = e;
        a.wts[pi] = a.w_in[pi];
        if (a.ids_dbg) a.ids_dbg[pi] = e;
        if (a.w_dbg) a.w_dbg[pi] = a.w_in[pi];
      }
    }
  }
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int pi = threadIdx.x; pi < P; pi += blockDim.x)
    if (s_ids[pi] >= 0) atomicAdd(&s_cnt[s_ids[pi]], 1);
  __syncthreads();
  if (warp == 0) {
    // exclusive scans of the counts (dispatch offsets) and of the used flags (slots)
    const int per = (E + 31) / 32, e0 = lane * per;
    int c = 0, u = 0;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      c += s_cnt[e];
      u += s_cnt[e] > 0;
    }
    int ci = c, ui = u;
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
      if (out) a.offsets[e] = run;
      if (n > 0) {
        s_uniq[nu] = e;
        if (out) a.uniq[nu] = e;
        ++nu;
      }
      s_cnt[e] = run;                   // now the expert's first dispatch position
      s_slot[e] = n > 0 ? nu - 1 : -1;  // and its slot
      run += n;
    }
    if (lane == 31) {
      *s_nu = nu;
      if (out) {
        a.offsets[E] = run;
        *a.nuniq = nu;
      }
    }
  }
  __syncthreads();
  if (out)
    for (int pi = threadIdx.x; pi < P; pi += blockDim.x) {
      const int e = s_ids[pi];
      if (e < 0) continue;
      int rank = 0;  // earlier pairs of the same expert
      for (int q = 0; q < pi; ++q) rank += s_ids[q] == e;
      a.pairs[s_cnt[e] + rank] = pi;
      a.rows[s_cnt[e] + rank] = rank < a.slot_rows ? s_slot[e] * a.slot_rows + rank : -1;
    }
}

// shared memory of s2_route: ids [P] int, counts [E+1] int, slot experts [E] int, slot of each
// expert [E] int, count
__host__ __device__ inline size_t s2_route_bytes(int P, int E) {
  return ((size_t)P * 4 + (size_t)(3 * E + 2) * 4 + 15) & ~size_t(15);
}

// the same load with an L2 cache policy (tc::l2_evict_*)
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* m, int x, int y, int z, int w,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, "
      "%4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(tc::smem_u32(bar)), "l"(policy)
      : "memory");
}
// bring a box into L2 only (no shared memory, no barrier), under an L2 cache policy
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* m, int x, int y, int z, int w, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile.L2::cache_hint [%0, {%1, %2, %3, %4}], %5;" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y), "r"(z), "r"(w), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* m, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(tc::smem_u32(bar))
      : "memory");
}

}  // namespace ql
