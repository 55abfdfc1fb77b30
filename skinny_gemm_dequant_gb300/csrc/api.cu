// C ABI of the library (declared in include/qlinear.h): argument validation, workspace
// layout, and the dispatch of each operation to its kernel sequence.
#include <cmath>
#include <cstdio>
#include <cstring>

#include "gemm_i8_tcgen05.h"
#include "gemm_tcgen05.h"
#include "internal.h"
#include "skinny2.cuh"

using namespace ql;

#ifndef QL_CELL_TOKENS
#define QL_CELL_TOKENS 4
#endif
#ifndef QL_LOCAL_MK
#define QL_LOCAL_MK 18432
#endif

namespace {

uint32_t g_wait_limit = 1u << 20;

inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Workspace layout: [0, 256) status word (offset 0) and the skinny GEMM's activation hand-off
// counters (offsets 32 and 36);
// [256, 256 + 4*kMaxTickets) split-K tickets, at the same place for every op and shape, so that
// no call's data region ever overlaps them (the kernels return every counter and ticket to
// zero); op regions follow, carved in order.
constexpr size_t kMaxTickets = 65536;
// the region after the status word that is zero between calls: the split-K tickets (first
// 4*kMaxTickets bytes) or, for INT8 calls of up to kCellTokens tokens, their output cells
// (those calls use no tickets); the kernels leave it zero
constexpr size_t kZeroRegion = size_t(1) << 20;
constexpr size_t kReadyOff = 32, kDoneOff = 36;
// INT8 calls of up to this many tokens settle their outputs through atomic cells (skinny2.cuh,
// s2_cell_*); larger ones through per-CTA partial sums and a waiting settler.  Measured on the
// INT8 decode bench: cells are faster at 1..4 tokens (most at N = 5120, K = 17408, where a row
// block is shared by about 8 CTAs), slower at 8 and 16 (their atomic traffic grows with M)
constexpr int64_t kCellTokens = QL_CELL_TOKENS;
// tokens one launch of the persistent skinny kernel takes: up to 32 for INT8 (four 8-token MMA
// tiles), 16 for the other formats; more tokens run in chunks (INT8: the tcgen05 GEMM)
constexpr int64_t kSkinnyMaxTokens = 32;
inline int64_t skinny_tokens(int fmt) { return fmt == FMT_INT8 ? kSkinnyMaxTokens : 16; }
// dense layers whose M * K is at most this build their activation image inside every CTA
// (each CTA reads the tokens' whole rows, so the cost grows with M * K) instead of sharing one
// through global memory, which takes a grid-wide hand-off per call.  Measured on the INT8 decode
// shapes: the local image wins at 1 token (K = 5120 and 17408) and at 2 tokens with K = 5120;
// the shared one at 2 tokens with K = 17408 (21.7 against 22.3 us) and 4 tokens with K = 5120
// (16.3 against 17.8 us at N = 10240)
constexpr int64_t kLocalMK = QL_LOCAL_MK;
constexpr size_t kTicketOff = 256;
constexpr size_t kRegionsOff = kTicketOff + kZeroRegion;

struct Carver {
  size_t off = kRegionsOff;
  size_t take(size_t bytes) {
    const size_t o = off;
    off += al256(bytes);
    return o;
  }
};

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

ql_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return QL_OK;
  fprintf(stderr, "qlinear: CUDA error %s\n", cudaGetErrorString(e));
  return QL_ERR_CUDA;
}

// ------------------------------------------------------------------ skinny plans
struct SkinnyPlan {
  int mt;
  int64_t nb;  // row blocks
  SplitK sk;
};

SkinnyPlan skinny_plan(int fmt, int64_t M, int64_t N, int64_t K) {
  SkinnyPlan p;
  p.mt = (M <= 8) ? 1 : 2;
  p.nb = cdiv(N, SK_ROWS);
  p.sk = skinny_split(fmt, p.mt, p.nb, K);
  return p;
}

struct DenseLayout {
  size_t counters, part, xq, xs, total;
};

DenseLayout dense_layout(int fmt, int64_t M, int64_t N, int64_t K) {
  const SkinnyPlan p = skinny_plan(fmt, M, N, K);
  Carver c;
  DenseLayout l;
  l.counters = kTicketOff;
  l.part = c.take(p.sk.ks > 1 ? (size_t)p.sk.ks * 16 * N * 4 : 0);
  l.xq = c.take(fmt == FMT_INT8 ? (size_t)M * K : 0);
  l.xs = c.take(fmt == FMT_INT8 ? (size_t)M * 4 : 0);
  l.total = c.off;
  return l;
}

struct Dense2Layout {
  Skinny2Plan p;
  size_t cells, x16, sc, part, total;
  bool cells_clean;  // the cells sit in the zero region (left zero by the kernel)
};

Dense2Layout dense2_layout(int fmt, int64_t Mc, int64_t N, int64_t K, int block_n) {
  Dense2Layout l;
  l.p = skinny2_plan(fmt, Mc, N, K, block_n);
  Carver c;
  const bool cells = fmt == FMT_INT8 && Mc <= kCellTokens;
  // INT8 output cells [M][N]: in the zero region when they fit (no zeroing inside the call),
  // else in a region of their own that the call's activation jobs zero first
  l.cells_clean = cells && (size_t)N * Mc * 8 <= kZeroRegion;
  l.cells = l.cells_clean ? kTicketOff : c.take(cells ? (size_t)N * Mc * 8 : 0);
  l.x16 = c.take((size_t)kXCopies * Mc * l.p.kpad * 2);
  l.sc = c.take(kSkinnyMaxTokens * 4);
  l.part = c.take(cells ? 0 : (size_t)l.p.grid * l.p.mp * S2_ROWS * 4);  // one partial slot per CTA
  l.total = c.off;
  return l;
}

// MoE on the persistent kernel: the router's outputs, gate/up sums, expert outputs, the
// activation image of either stage, per-row factors and per-CTA partial sums
struct Moe2Layout {
  Skinny2Plan gu, dn;
  int slots, slot_rows;
  size_t ids, wts, offsets, pairs, rows, uniq, nuniq, gus, o, x16, tokf, part, total;
};

Moe2Layout moe2_layout(int64_t M, int64_t H, int64_t I, int E, int topk) {
  Moe2Layout l;
  const int64_t P = M * topk;
  l.slots = (int)(P < E ? P : E);
  l.gu = skinny2_plan(FMT_MXFP4, M, 2 * I, H, 0, l.slots);
  l.dn = skinny2_plan(FMT_MXFP4, M, H, I, 0, l.slots);
  l.slot_rows = l.dn.mp;
  Carver c;
  l.ids = c.take(P * 4);
  l.wts = c.take(P * 4);
  l.offsets = c.take((E + 1) * 4);
  l.pairs = c.take(P * 4);
  l.rows = c.take(P * 4);
  l.uniq = c.take((size_t)E * 4);
  l.nuniq = c.take(4);
  l.gus = c.take((size_t)P * 2 * I * 4);
  l.o = c.take((size_t)P * H * 4);
  const size_t img_gu = (size_t)kXCopies * M * l.gu.kpad * 2;
  const size_t img_dn = (size_t)kXCopies * l.slots * l.slot_rows * l.dn.kpad * 2;
  l.x16 = c.take(img_gu > img_dn ? img_gu : img_dn);
  l.tokf = c.take((size_t)(l.slots * l.slot_rows > M ? l.slots * l.slot_rows : M) * 4);
  const int g = l.gu.grid > l.dn.grid ? l.gu.grid : l.dn.grid;
  l.part = c.take((size_t)g * 16 * S2_ROWS * 4);
  l.total = c.off;
  return l;
}

// the persistent kernel takes the MoE when both K's are whole 256-K units (scale rows then
// whole 8-byte groups) and the scale arrays are 8-byte aligned
bool moe2_ok(int64_t H, int64_t I, const void* s13, const void* s2) {
  return H % 256 == 0 && I % 256 == 0 && (reinterpret_cast<uintptr_t>(s13) & 7) == 0 &&
         (reinterpret_cast<uintptr_t>(s2) & 7) == 0;
}

// MXFP4 weights go through the persistent kernel when whole 256-K units and 8-byte scale
// rows allow it; other shapes use the register-streaming kernel.
bool mxfp4_v2_ok(int64_t K, int64_t lds, const void* wsb) {
  return K % 256 == 0 && lds % 8 == 0 && (reinterpret_cast<uintptr_t>(wsb) & 7) == 0;
}

struct Dense2Call {
  int fmt;
  const uint16_t* x;
  int64_t M, K, ldx;
  const uint8_t* w;
  int64_t N, ldw;
  const uint8_t* wsb;
  int64_t lds;
  int block_n, block_k;
  const float* w_scale;
  int64_t w_scale_len;
  const uint16_t* bias;
  uint16_t* y;
  int64_t ldy;
  int32_t* acc_out;
  int8_t* xq_out;
  float* xs_out;
  const float* amax_in;  // INT8 K shard: the tokens' amax over the whole row
  float* y32;            // FP8 / MXFP4 K shard: fp32 partial sums [M, ldy32] instead of y
  int64_t ldy32;
};

ql_status run_dense2(const Dense2Call& d, void* workspace, cudaStream_t st);

struct MoeLayout {
  size_t ids, wts, offsets, pairs, uniq, nuniq, h, o, cnt_gu, part_gu, cnt_dn, part_dn, total;
  int mt, umax;
  SplitK gu, dn;
  int64_t nb_gu, nb_dn;
};

MoeLayout moe_layout(int64_t M, int64_t H, int64_t I, int E, int topk) {
  MoeLayout l;
  const int64_t P = M * topk;
  l.umax = (int)(P < E ? P : E);
  l.mt = (M <= 8) ? 1 : 2;
  l.nb_gu = cdiv(I, 32);
  l.nb_dn = cdiv(H, SK_ROWS);
  l.gu = skinny_split(FMT_MXFP4, l.mt, l.nb_gu * l.umax, H);
  l.dn = skinny_split(FMT_MXFP4, l.mt, l.nb_dn * l.umax, I);
  Carver c;
  l.ids = c.take(P * 4);
  l.wts = c.take(P * 4);
  l.offsets = c.take((E + 1) * 4);
  l.pairs = c.take(P * 4);
  l.uniq = c.take((size_t)E * 4);
  l.nuniq = c.take(4);
  l.h = c.take((size_t)P * I * 2);
  l.o = c.take((size_t)P * H * 4);
  l.cnt_gu = kTicketOff;  // gate_up and down run one after the other and share the tickets
  l.part_gu = c.take(l.gu.ks > 1 ? (size_t)l.umax * l.gu.ks * 16 * (2 * I) * 4 : 0);
  l.cnt_dn = kTicketOff;
  l.part_dn = c.take(l.dn.ks > 1 ? (size_t)l.umax * l.dn.ks * 16 * H * 4 : 0);
  l.total = c.off;
  return l;
}

// grouped MoE for M > 16 on the tcgen05 path: routing, dispatch rows and tile list, the E4M3
// activations of both expert GEMMs by dispatch row, and the fp32 gate/up and down rows by pair
struct Moe3Layout {
  int tt, tiles_max;
  size_t ids, wts, counts, offsets, tiles, ntiles, pairs, pos, q_gu, s_gu, gu, q_dn, s_dn, o, total;
};
Moe3Layout moe3_layout(int64_t M, int64_t H, int64_t I, int E, int topk) {
  Moe3Layout l;
  const int64_t P = M * topk;
  const int64_t used = P < E ? P : E;  // experts that can be routed to
  const int64_t avg = (P + used - 1) / used;
  int tt = (int)((avg + 15) / 16 * 16);
  l.tt = tt < 16 ? 16 : (tt > 128 ? 128 : tt);
  l.tiles_max = (int)((P + l.tt - 1) / l.tt + used);
  Carver c;
  l.ids = c.take((size_t)P * 4);
  l.wts = c.take((size_t)P * 4);
  l.counts = c.take((size_t)E * 4);
  l.offsets = c.take((size_t)(E + 1) * 4);
  l.tiles = c.take((size_t)l.tiles_max * 16);
  l.ntiles = c.take(4);
  l.pairs = c.take((size_t)P * 4);
  l.pos = c.take((size_t)P * 4);
  l.q_gu = c.take((size_t)P * H);
  l.s_gu = c.take((size_t)P * (H / 128));
  l.gu = c.take((size_t)P * 2 * I * 4);
  l.q_dn = c.take((size_t)P * I);
  l.s_dn = c.take((size_t)P * (I / 128));
  l.o = c.take((size_t)P * H * 4);
  l.total = c.off;
  return l;
}

// workspace of the INT8 tcgen05 GEMM (M > 16): f16 activation codes and per-token scales
struct I8Layout {
  size_t img, xs, part, total;
};
I8Layout i8_layout(int64_t M, int64_t N, int64_t K) {
  I8Layout l;
  Carver c;
  l.img = c.take(tc::i8_image_bytes(M, K));
  l.xs = c.take((size_t)M * 4);
  l.part = c.take(tc::i8_part_bytes(M, N, K));  // split-K partial sums (none without a split)
  l.total = c.off;
  return l;
}

// workspace for the tcgen05 path (activation codes and scales) plus the skinny fallbacks
size_t act_quant_ws(int64_t M, int64_t K) {
  Carver c;
  c.take(tc::act_q_bytes(M, K));
  c.take(tc::act_s_bytes(M, K));
  return c.off;
}

bool tc_path(int act_mode) { return act_mode == QL_ACT_E4M3_1X128; }

}  // namespace

uint32_t ql::wait_limit() { return g_wait_limit; }

size_t ql::workspace_zero_bytes() { return kRegionsOff; }

namespace {
ql_status run_dense2(const Dense2Call& d, void* workspace, cudaStream_t st) {
  const int64_t chunk = skinny_tokens(d.fmt);
  for (int64_t m0 = 0; m0 < d.M; m0 += chunk) {
    const int64_t Mc = (d.M - m0) < chunk ? (d.M - m0) : chunk;
    const Dense2Layout l = dense2_layout(d.fmt, Mc, d.N, d.K, d.block_n);
    Skinny2Args a = {};
    a.M = (int)Mc;
    a.N = (int)d.N;
    a.K = (int)d.K;
    a.x = d.x + m0 * d.ldx;
    a.ldx = d.ldx;
    a.x16 = at<uint16_t>(workspace, l.x16);
    a.tokf = at<float>(workspace, l.sc);
    a.img_rows = (int)Mc;
    a.xq_dbg = d.xq_out ? d.xq_out + m0 * d.K : nullptr;
    a.xs_dbg = d.xs_out ? d.xs_out + m0 : nullptr;
    a.ready = at<unsigned>(workspace, kReadyOff);
    a.done = at<unsigned>(workspace, kDoneOff);
    a.wsb = d.wsb;
    a.lds = d.lds;
    a.block_n = d.block_n;
    a.block_k = d.block_k;
    a.w_scale = d.w_scale;
    a.w_scale_len = (int)d.w_scale_len;
    a.y = d.y ? d.y + m0 * d.ldy : nullptr;
    a.ldy = d.ldy;
    a.bias = d.bias;
    a.acc_out = d.acc_out ? d.acc_out + m0 * d.N : nullptr;
    a.amax_in = d.amax_in ? d.amax_in + m0 : nullptr;
    a.y32 = d.y32 ? d.y32 + m0 * d.ldy32 : nullptr;
    a.ldy32 = d.ldy32;
    a.part = at<float>(workspace, l.part);
    a.tickets = at<unsigned>(workspace, kTicketOff);
    a.cells = (d.fmt == FMT_INT8 && Mc <= kCellTokens) ? at<unsigned long long>(workspace, l.cells) : nullptr;
    a.cells_clean = l.cells_clean ? 1 : 0;
    // local activations: no activation jobs run, so INT8 cells must already be clean
    a.local = (d.fmt != FMT_BF16 && Mc * d.K <= kLocalMK && (a.cells == nullptr || a.cells_clean)) ? 1 : 0;
    a.status = at<uint32_t>(workspace, 0);
    a.wait_limit = g_wait_limit;
    const cudaError_t e = launch_skinny2(d.fmt, l.p, a, d.w, d.ldw, st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return QL_OK;
}
}  // namespace

extern "C" {

const char* ql_status_string(ql_status s) {
  switch (s) {
    case QL_OK: return "ok";
    case QL_ERR_INVALID_ARG: return "invalid argument";
    case QL_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case QL_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
    case QL_ERR_WORKSPACE: return "workspace missing or too small";
    case QL_ERR_CUDA: return "CUDA error";
    case QL_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int ql_version(void) { return 1; }

void ql_set_wait_limit(uint32_t polls) { g_wait_limit = polls; }

size_t ql_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int E, int topk) {
  if (M < 0 || N < 0 || K < 0) return 0;
  const int64_t Mc = M < 16 ? M : 16;  // skinny kernels run 16 tokens at a time
  switch (op) {
    case QL_OP_INT8_W8A8: {
      const int64_t Mi = M < kSkinnyMaxTokens ? M : kSkinnyMaxTokens;
      const size_t a = dense2_layout(FMT_INT8, Mi, N, K, 128).total;
      const size_t b = M > kSkinnyMaxTokens ? i8_layout(M, N, K).total : 0;
      return a > b ? a : b;
    }
    case QL_OP_FP8_BLOCK: {
      // block_n is not known here: 16 (the smallest accepted) bounds the scale staging
      size_t a = dense2_layout(FMT_FP8, Mc, N, K, 16).total;
      const size_t a1 = dense_layout(FMT_FP8, Mc, N, K).total;  // block_k not a power of two
      if (a1 > a) a = a1;
      const size_t b = act_quant_ws(M, K);
      return a > b ? a : b;
    }
    case QL_OP_MXFP4: {
      size_t a = dense_layout(FMT_MXFP4, Mc, N, K).total;
      const size_t a2 = dense2_layout(FMT_MXFP4, Mc, N, K, 128).total;
      if (a2 > a) a = a2;
      const size_t b = act_quant_ws(M, K);
      return a > b ? a : b;
    }
    case QL_OP_BF16:
      return dense2_layout(FMT_BF16, Mc, N, K, 128).total;
    case QL_OP_FP8_CHANNEL:
      return dense2_layout(FMT_F8E4C, Mc, N, K, 128).total;  // E4M3 and E5M2 lay out alike
    case QL_OP_MOE_MXFP4: {
      if (E <= 0 || topk <= 0) return 0;
      if (M > 16) return moe3_layout(M, N, K, E, topk).total;
      const size_t a = moe_layout(M, N, K, E, topk).total, b = moe2_layout(M, N, K, E, topk).total;
      return a > b ? a : b;
    }
  }
  return 0;
}

ql_status ql_workspace_init(void* workspace, size_t bytes, ql_stream_t stream) {
  if (!workspace || bytes < 256) return QL_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream));
}

ql_status ql_read_device_status(void* workspace, ql_stream_t stream, int clear, uint32_t* flags_out) {
  if (!workspace) return QL_ERR_WORKSPACE;
  uint32_t flags = 0;
  cudaError_t e = cudaMemcpyAsync(&flags, workspace, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(workspace, 0, 4, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e);
  if (flags_out) *flags_out = flags;
  return (flags & QL_DEV_TIMEOUT) ? QL_ERR_TIMEOUT : QL_OK;
}

}  // extern "C"

namespace {
// the INT8 linear; amax_in (a K shard's whole-row amax) and y == null (acc_out only) serve the
// row-parallel layer
ql_status int8_impl(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const int8_t* w, int64_t N, int64_t ldw,
                    const float* w_scale, int64_t w_scale_len, const uint16_t* bias, uint16_t* y, int64_t ldy,
                    int32_t* acc_out, int8_t* xq_out, float* xs_out, const float* amax_in, void* workspace,
                    size_t workspace_bytes, ql_stream_t stream, int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (!x || !w || (y && !w_scale) || (!y && !acc_out)) return QL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldx < K || ldw < K || (y && ldy < N)) return QL_ERR_INVALID_ARG;
  if (y && w_scale_len != 1 && w_scale_len != N) return QL_ERR_INVALID_ARG;
  if (M > 65535 || N > (1 << 30) || K > 133152) return QL_ERR_UNSUPPORTED;  // |acc| < 2^31
  if (K % 16 != 0) return QL_ERR_UNSUPPORTED;
  if (cdiv(N, SK_ROWS) > (int64_t)kMaxTickets) return QL_ERR_UNSUPPORTED;
  if (!al16(x) || !al16(w) || ldx % 8 != 0 || ldw % 16 != 0) return QL_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < ql_workspace_bytes(QL_OP_INT8_W8A8, M, N, K, 0, 0)) return QL_ERR_WORKSPACE;
  if (!al16(workspace)) return QL_ERR_ALIGNMENT;
  cudaStream_t st = (cudaStream_t)stream;

  if (M > kSkinnyMaxTokens) {
    // prefill-sized batches: one GEMM on the tensor cores streams the weights once
    const I8Layout l = i8_layout(M, N, K);
    tc::I8GemmArgs g = {};
    g.M = (int)M;
    g.N = (int)N;
    g.K = (int)K;
    g.x = x;
    g.ldx = ldx;
    g.w = w;
    g.ldw = ldw;
    g.w_s = w_scale;
    g.w_s_len = (int)w_scale_len;
    g.bias = bias;
    g.y = y;
    g.ldy = ldy;
    g.acc_out = acc_out;
    g.xq_dbg = xq_out;
    g.xs_dbg = xs_out;
    g.img = at<uint16_t>(workspace, l.img);
    g.xs = at<float>(workspace, l.xs);
    g.part = at<int32_t>(workspace, l.part);
    g.tickets = at<unsigned>(workspace, kTicketOff);
    g.status = at<uint32_t>(workspace, 0);
    g.wait_limit = g_wait_limit;
    g.amax_in = amax_in;
    const cudaError_t e = tc::launch_i8_gemm(g, st);
    if (e != cudaSuccess) return cuda_status(e);
    if (path_out) *path_out = QL_PATH_INT8_TCGEN05;
    return QL_OK;
  }

  Dense2Call d = {};
  d.fmt = FMT_INT8;
  d.x = x;
  d.M = M;
  d.K = K;
  d.ldx = ldx;
  d.w = reinterpret_cast<const uint8_t*>(w);
  d.N = N;
  d.ldw = ldw;
  d.w_scale = w_scale;
  d.w_scale_len = w_scale_len;
  d.bias = bias;
  d.y = y;
  d.ldy = ldy;
  d.acc_out = acc_out;
  d.xq_out = xq_out;
  d.xs_out = xs_out;
  d.amax_in = amax_in;
  const ql_status s = run_dense2(d, workspace, st);
  if (s != QL_OK) return s;
  if (path_out) *path_out = QL_PATH_INT8_SKINNY;
  return QL_OK;
}
}  // namespace

extern "C" {

// ------------------------------------------------------------------ INT8 W8A8
ql_status qlinear_int8_w8a8(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const int8_t* w, int64_t N,
                            int64_t ldw, const float* w_scale, int64_t w_scale_len, const uint16_t* bias,
                            uint16_t* y, int64_t ldy, int32_t* acc_out, int8_t* xq_out, float* xs_out,
                            void* workspace, size_t workspace_bytes, ql_stream_t stream, int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (!y) return QL_ERR_INVALID_ARG;
  return int8_impl(x, M, K, ldx, w, N, ldw, w_scale, w_scale_len, bias, y, ldy, acc_out, xq_out, xs_out, nullptr,
                   workspace, workspace_bytes, stream, path_out);
}

// ------------------------------------------------------------------ sharded layers
ql_status ql_token_amax(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float* amax_out, ql_stream_t stream) {
  if (!x || !amax_out) return QL_ERR_INVALID_ARG;
  if (M < 1 || K < 1 || ldx < K) return QL_ERR_INVALID_ARG;
  if (M > 65535 || K > (1 << 30)) return QL_ERR_UNSUPPORTED;
  if (K % 8 != 0) return QL_ERR_UNSUPPORTED;
  if (!al16(x) || ldx % 8 != 0) return QL_ERR_ALIGNMENT;
  return cuda_status(launch_token_amax(x, (int)M, (int)K, ldx, amax_out, (cudaStream_t)stream));
}

ql_status qlinear_int8_w8a8_partial(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const int8_t* w,
                                    int64_t N, int64_t ldw, const float* amax, int32_t* acc_out, int8_t* xq_out,
                                    void* workspace, size_t workspace_bytes, ql_stream_t stream, int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (!amax || !acc_out) return QL_ERR_INVALID_ARG;
  return int8_impl(x, M, K, ldx, w, N, ldw, nullptr, 0, nullptr, nullptr, 0, acc_out, xq_out, nullptr, amax,
                   workspace, workspace_bytes, stream, path_out);
}

ql_status qlinear_int8_epilogue(const int32_t* acc, int64_t M, int64_t N, const float* amax, const float* w_scale,
                                int64_t w_scale_len, const uint16_t* bias, uint16_t* y, int64_t ldy,
                                ql_stream_t stream) {
  if (!acc || !amax || !w_scale || !y) return QL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || ldy < N || (w_scale_len != 1 && w_scale_len != N)) return QL_ERR_INVALID_ARG;
  if (M > 65535 || N > (1 << 30)) return QL_ERR_UNSUPPORTED;
  return cuda_status(launch_int8_epilogue(acc, (int)M, (int)N, amax, w_scale, (int)w_scale_len, bias, y, ldy,
                                          (cudaStream_t)stream));
}

ql_status ql_finish_f32(const float* y32, int64_t M, int64_t N, int64_t ld32, const uint16_t* bias, uint16_t* y,
                        int64_t ldy, ql_stream_t stream) {
  if (!y32 || !y) return QL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || ld32 < N || ldy < N) return QL_ERR_INVALID_ARG;
  if (M > 65535 || N > (1 << 30)) return QL_ERR_UNSUPPORTED;
  return cuda_status(launch_finish_f32(y32, (int)M, (int)N, ld32, bias, y, ldy, (cudaStream_t)stream));
}

// ------------------------------------------------------------------ shared skinny launcher (FP8 / MXFP4, bf16 act)
static ql_status run_skinny_bf16(int fmt, const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* w,
                                 int64_t N, int64_t ldw, const uint8_t* wsb, int64_t lds, int block_n, int block_k,
                                 const uint16_t* bias, uint16_t* y, int64_t ldy, void* workspace, cudaStream_t st) {
  for (int64_t m0 = 0; m0 < M; m0 += 16) {
    const int64_t Mc = (M - m0) < 16 ? (M - m0) : 16;
    const SkinnyPlan p = skinny_plan(fmt, Mc, N, K);
    const DenseLayout l = dense_layout(fmt, Mc, N, K);
    SkinnyArgs a = {};
    a.w = w;
    a.ldw = ldw;
    a.wsb = wsb;
    a.lds = lds;
    a.block_n = block_n;
    a.block_k = block_k;
    a.x = x + m0 * ldx;
    a.ldx = ldx;
    a.M = (int)Mc;
    a.N = (int)N;
    a.K = (int)K;
    a.y = y + m0 * ldy;
    a.ldy = ldy;
    a.bias = bias;
    a.ks = p.sk.ks;
    a.kc = p.sk.kc;
    a.part = at<void>(workspace, l.part);
    a.counters = at<unsigned>(workspace, l.counters);
    a.pdl = 0;
    cudaError_t e = launch_skinny(fmt, p.mt, EPI_LINEAR, a, dim3((unsigned)p.nb, (unsigned)p.sk.ks, 1), st, false);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return QL_OK;
}

// ------------------------------------------------------------------ FP8 block
ql_status qlinear_fp8_block(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* w, int64_t N,
                            int64_t ldw, const uint8_t* w_scale, int block_n, int block_k, int act_mode,
                            const uint16_t* bias, uint16_t* y, int64_t ldy, uint8_t* aq_out, uint8_t* as_out,
                            void* workspace, size_t workspace_bytes, ql_stream_t stream, int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (!x || !w || !w_scale || !y) return QL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldx < K || ldw < K || ldy < N || block_n < 1 || block_k < 1)
    return QL_ERR_INVALID_ARG;
  if (act_mode != QL_ACT_BF16 && act_mode != QL_ACT_E4M3_1X128) return QL_ERR_INVALID_ARG;
  if (M > 65535 || N > (1 << 30) || K > (1 << 30)) return QL_ERR_UNSUPPORTED;
  if (K % 16 != 0 || cdiv(N, SK_ROWS) > (int64_t)kMaxTickets) return QL_ERR_UNSUPPORTED;
  if (!al16(x) || !al16(w) || ldx % 8 != 0 || ldw % 16 != 0) return QL_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < ql_workspace_bytes(QL_OP_FP8_BLOCK, M, N, K, 0, 0)) return QL_ERR_WORKSPACE;
  if (!al16(workspace)) return QL_ERR_ALIGNMENT;
  cudaStream_t st = (cudaStream_t)stream;
  if (!tc_path(act_mode)) {
    if (block_n % 16 != 0 || block_k % 64 != 0) return QL_ERR_UNSUPPORTED;
    if ((block_k & (block_k - 1)) != 0) {
      // the persistent kernel indexes block scales by shift: other block sizes stream through
      // the register kernel
      const ql_status s2 = run_skinny_bf16(FMT_FP8, x, M, K, ldx, w, N, ldw, w_scale, cdiv(K, block_k), block_n,
                                           block_k, bias, y, ldy, workspace, st);
      if (s2 == QL_OK && path_out) *path_out = QL_PATH_FP8_SKINNY;
      return s2;
    }
    Dense2Call d = {};
    d.fmt = FMT_FP8;
    d.x = x;
    d.M = M;
    d.K = K;
    d.ldx = ldx;
    d.w = w;
    d.N = N;
    d.ldw = ldw;
    d.wsb = w_scale;
    d.lds = cdiv(K, block_k);
    d.block_n = block_n;
    d.block_k = block_k;
    d.bias = bias;
    d.y = y;
    d.ldy = ldy;
    const ql_status s = run_dense2(d, workspace, st);
    if (s == QL_OK && path_out) *path_out = QL_PATH_FP8_SKINNY;
    return s;
  }
  if (block_n != 128 || block_k != 128 || K % 128 != 0) return QL_ERR_UNSUPPORTED;
  Carver c;
  const size_t oq = c.take(tc::act_q_bytes(M, K)), os = c.take(tc::act_s_bytes(M, K));
  tc::GemmArgs g = {};
  g.M = (int)M;
  g.N = (int)N;
  g.K = (int)K;
  g.w = w;
  g.ldw = ldw;
  g.ws = w_scale;
  g.lds = cdiv(K, 128);
  g.fp4 = 0;
  g.aq = at<uint8_t>(workspace, oq);
  g.as = at<uint8_t>(workspace, os);
  g.y = y;
  g.ldy = ldy;
  g.bias = bias;
  g.status = at<uint32_t>(workspace, 0);
  g.wait_limit = g_wait_limit;
  cudaError_t e = tc::quantize_activations(x, M, K, ldx, g, aq_out, as_out, st);
  if (e == cudaSuccess) e = tc::launch_gemm(g, st);
  if (e != cudaSuccess) return cuda_status(e);
  if (path_out) *path_out = QL_PATH_FP8_TCGEN05;
  return QL_OK;
}

// a K shard of a row-parallel FP8-block layer: fp32 partial sums, bf16 activations
ql_status qlinear_fp8_block_partial(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* w, int64_t N,
                                    int64_t ldw, const uint8_t* w_scale, int block_n, int block_k, float* y32,
                                    int64_t ldy32, void* workspace, size_t workspace_bytes, ql_stream_t stream,
                                    int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (!x || !w || !w_scale || !y32) return QL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldx < K || ldw < K || ldy32 < N || block_n < 1 || block_k < 1)
    return QL_ERR_INVALID_ARG;
  if (M > 65535 || N > (1 << 30) || K > (1 << 30)) return QL_ERR_UNSUPPORTED;
  if (K % 16 != 0 || cdiv(N, SK_ROWS) > (int64_t)kMaxTickets) return QL_ERR_UNSUPPORTED;
  if (block_n % 16 != 0 || block_k % 64 != 0 || (block_k & (block_k - 1)) != 0) return QL_ERR_UNSUPPORTED;
  if (!al16(x) || !al16(w) || ldx % 8 != 0 || ldw % 16 != 0) return QL_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < ql_workspace_bytes(QL_OP_FP8_BLOCK, M, N, K, 0, 0)) return QL_ERR_WORKSPACE;
  if (!al16(workspace)) return QL_ERR_ALIGNMENT;
  Dense2Call d = {};
  d.fmt = FMT_FP8;
  d.x = x;
  d.M = M;
  d.K = K;
  d.ldx = ldx;
  d.w = w;
  d.N = N;
  d.ldw = ldw;
  d.wsb = w_scale;
  d.lds = cdiv(K, block_k);
  d.block_n = block_n;
  d.block_k = block_k;
  d.y32 = y32;
  d.ldy32 = ldy32;
  const ql_status s = run_dense2(d, workspace, (cudaStream_t)stream);
  if (s == QL_OK && path_out) *path_out = QL_PATH_FP8_SKINNY;
  return s;
}

// ------------------------------------------------------------------ FP8 per channel / per tensor
ql_status qlinear_fp8(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* w, int64_t N, int64_t ldw,
                      int w_fmt, const float* w_scale, int64_t w_scale_len, const uint16_t* bias, uint16_t* y,
                      int64_t ldy, void* workspace, size_t workspace_bytes, ql_stream_t stream, int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (!x || !w || !w_scale || !y) return QL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldx < K || ldw < K || ldy < N) return QL_ERR_INVALID_ARG;
  if (w_fmt != QL_FP8_E4M3 && w_fmt != QL_FP8_E5M2) return QL_ERR_INVALID_ARG;
  if (w_scale_len != 1 && w_scale_len != N) return QL_ERR_INVALID_ARG;
  if (M > 65535 || N > (1 << 30) || K > (1 << 28)) return QL_ERR_UNSUPPORTED;
  if (K % 16 != 0 || cdiv(N, S2_ROWS) > (int64_t)kMaxTickets) return QL_ERR_UNSUPPORTED;
  if (!al16(x) || !al16(w) || ldx % 8 != 0 || ldw % 16 != 0) return QL_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < ql_workspace_bytes(QL_OP_FP8_CHANNEL, M, N, K, 0, 0)) return QL_ERR_WORKSPACE;
  if (!al16(workspace)) return QL_ERR_ALIGNMENT;
  Dense2Call d = {};
  d.fmt = w_fmt == QL_FP8_E4M3 ? FMT_F8E4C : FMT_F8E5C;
  d.x = x;
  d.M = M;
  d.K = K;
  d.ldx = ldx;
  d.w = w;
  d.N = N;
  d.ldw = ldw;
  d.w_scale = w_scale;
  d.w_scale_len = w_scale_len;
  d.bias = bias;
  d.y = y;
  d.ldy = ldy;
  const ql_status s = run_dense2(d, workspace, (cudaStream_t)stream);
  if (s == QL_OK && path_out) *path_out = QL_PATH_FP8_CHANNEL_SKINNY;
  return s;
}

// ------------------------------------------------------------------ BF16 dense
ql_status qlinear_bf16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint16_t* w, int64_t N,
                       int64_t ldw, const uint16_t* bias, uint16_t* y, int64_t ldy, void* workspace,
                       size_t workspace_bytes, ql_stream_t stream, int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (!x || !w || !y) return QL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldx < K || ldw < K || ldy < N) return QL_ERR_INVALID_ARG;
  if (M > 65535 || N > (1 << 30) || K > (1 << 28)) return QL_ERR_UNSUPPORTED;
  if (K % 8 != 0 || cdiv(N, S2_ROWS) > (int64_t)kMaxTickets) return QL_ERR_UNSUPPORTED;
  if (!al16(x) || !al16(w) || ldx % 8 != 0 || ldw % 8 != 0) return QL_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < ql_workspace_bytes(QL_OP_BF16, M, N, K, 0, 0)) return QL_ERR_WORKSPACE;
  if (!al16(workspace)) return QL_ERR_ALIGNMENT;
  Dense2Call d = {};
  d.fmt = FMT_BF16;
  d.x = x;
  d.M = M;
  d.K = K;
  d.ldx = ldx;
  d.w = reinterpret_cast<const uint8_t*>(w);
  d.N = N;
  d.ldw = ldw * 2;  // bytes
  d.bias = bias;
  d.y = y;
  d.ldy = ldy;
  const ql_status s = run_dense2(d, workspace, (cudaStream_t)stream);
  if (s == QL_OK && path_out) *path_out = QL_PATH_BF16_SKINNY;
  return s;
}

// ------------------------------------------------------------------ MXFP4 dense
ql_status qlinear_mxfp4(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* w, int64_t N,
                        int64_t ldw_bytes, const uint8_t* w_scale, int64_t lds, int act_mode, const uint16_t* bias,
                        uint16_t* y, int64_t ldy, uint8_t* aq_out, uint8_t* as_out, void* workspace,
                        size_t workspace_bytes, ql_stream_t stream, int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (!x || !w || !w_scale || !y) return QL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldx < K || ldw_bytes * 2 < K || lds * 32 < K || ldy < N) return QL_ERR_INVALID_ARG;
  if (act_mode != QL_ACT_BF16 && act_mode != QL_ACT_E4M3_1X128) return QL_ERR_INVALID_ARG;
  if (M > 65535 || N > (1 << 30) || K > (1 << 30)) return QL_ERR_UNSUPPORTED;
  if (K % 32 != 0 || cdiv(N, SK_ROWS) > (int64_t)kMaxTickets) return QL_ERR_UNSUPPORTED;
  if (!al16(x) || !al16(w) || ldx % 8 != 0 || ldw_bytes % 16 != 0) return QL_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < ql_workspace_bytes(QL_OP_MXFP4, M, N, K, 0, 0)) return QL_ERR_WORKSPACE;
  if (!al16(workspace)) return QL_ERR_ALIGNMENT;
  cudaStream_t st = (cudaStream_t)stream;
  if (!tc_path(act_mode)) {
    if (lds % 4 != 0 || (reinterpret_cast<uintptr_t>(w_scale) & 3) != 0) return QL_ERR_ALIGNMENT;
    ql_status s;
    if (mxfp4_v2_ok(K, lds, w_scale)) {
      Dense2Call d = {};
      d.fmt = FMT_MXFP4;
      d.x = x;
      d.M = M;
      d.K = K;
      d.ldx = ldx;
      d.w = w;
      d.N = N;
      d.ldw = ldw_bytes;
      d.wsb = w_scale;
      d.lds = lds;
      d.bias = bias;
      d.y = y;
      d.ldy = ldy;
      s = run_dense2(d, workspace, st);
    } else {
      s = run_skinny_bf16(FMT_MXFP4, x, M, K, ldx, w, N, ldw_bytes, w_scale, lds, 0, 0, bias, y, ldy, workspace, st);
    }
    if (s == QL_OK && path_out) *path_out = QL_PATH_MXFP4_SKINNY;
    return s;
  }
  if (K % 128 != 0) return QL_ERR_UNSUPPORTED;
  if (lds % 16 != 0 || !al16(w_scale)) return QL_ERR_ALIGNMENT;
  Carver c;
  const size_t oq = c.take(tc::act_q_bytes(M, K)), os = c.take(tc::act_s_bytes(M, K));
  tc::GemmArgs g = {};
  g.M = (int)M;
  g.N = (int)N;
  g.K = (int)K;
  g.w = w;
  g.ldw = ldw_bytes;
  g.ws = w_scale;
  g.lds = lds;
  g.fp4 = 1;
  g.aq = at<uint8_t>(workspace, oq);
  g.as = at<uint8_t>(workspace, os);
  g.y = y;
  g.ldy = ldy;
  g.bias = bias;
  g.status = at<uint32_t>(workspace, 0);
  g.wait_limit = g_wait_limit;
  cudaError_t e = tc::quantize_activations(x, M, K, ldx, g, aq_out, as_out, st);
  if (e == cudaSuccess) e = tc::launch_gemm(g, st);
  if (e != cudaSuccess) return cuda_status(e);
  if (path_out) *path_out = QL_PATH_MXFP4_TCGEN05;
  return QL_OK;
}

// ------------------------------------------------------------------ MoE
// a K shard of a row-parallel MXFP4 layer: fp32 partial sums, bf16 activations
ql_status qlinear_mxfp4_partial(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* w, int64_t N,
                                int64_t ldw_bytes, const uint8_t* w_scale, int64_t lds, float* y32, int64_t ldy32,
                                void* workspace, size_t workspace_bytes, ql_stream_t stream, int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (!x || !w || !w_scale || !y32) return QL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldx < K || ldw_bytes * 2 < K || lds * 32 < K || ldy32 < N) return QL_ERR_INVALID_ARG;
  if (M > 65535 || N > (1 << 30) || K > (1 << 30)) return QL_ERR_UNSUPPORTED;
  if (cdiv(N, SK_ROWS) > (int64_t)kMaxTickets) return QL_ERR_UNSUPPORTED;
  if (!mxfp4_v2_ok(K, lds, w_scale)) return QL_ERR_UNSUPPORTED;  // whole 256-K units, 8-byte scale rows
  if (!al16(x) || !al16(w) || ldx % 8 != 0 || ldw_bytes % 16 != 0) return QL_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < ql_workspace_bytes(QL_OP_MXFP4, M, N, K, 0, 0)) return QL_ERR_WORKSPACE;
  if (!al16(workspace)) return QL_ERR_ALIGNMENT;
  Dense2Call d = {};
  d.fmt = FMT_MXFP4;
  d.x = x;
  d.M = M;
  d.K = K;
  d.ldx = ldx;
  d.w = w;
  d.N = N;
  d.ldw = ldw_bytes;
  d.wsb = w_scale;
  d.lds = lds;
  d.y32 = y32;
  d.ldy32 = ldy32;
  const ql_status s = run_dense2(d, workspace, (cudaStream_t)stream);
  if (s == QL_OK && path_out) *path_out = QL_PATH_MXFP4_SKINNY;
  return s;
}

ql_status moe_mxfp4_grouped(const uint16_t* x, int64_t M, int64_t H, const uint16_t* router_logits,
                            const int32_t* topk_ids_in, const float* topk_w_in, int E, int topk, int renormalize,
                            const uint8_t* w13, const uint8_t* s13, const uint8_t* w2, const uint8_t* s2, int64_t I,
                            float swiglu_alpha, float swiglu_limit, int32_t* topk_ids_out, float* topk_w_out,
                            uint16_t* h_out, uint16_t* y, void* workspace, size_t workspace_bytes,
                            ql_stream_t stream, int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (!x || !w13 || !s13 || !w2 || !s2 || !y) return QL_ERR_INVALID_ARG;
  if (!std::isfinite(swiglu_alpha) || std::isnan(swiglu_limit) || swiglu_limit < 0.f) return QL_ERR_INVALID_ARG;
  if ((router_logits == nullptr) == (topk_ids_in == nullptr)) return QL_ERR_INVALID_ARG;
  if (topk_ids_in && !topk_w_in) return QL_ERR_INVALID_ARG;
  if (M < 1 || H < 1 || I < 1 || E < 1 || topk < 1) return QL_ERR_INVALID_ARG;
  if (M > 65535 || topk > 16 || topk > E || E > 1024) return QL_ERR_UNSUPPORTED;
  if (H % 128 != 0 || I % 128 != 0 || H > (1 << 20) || I > (1 << 20)) return QL_ERR_UNSUPPORTED;
  if (!al16(x) || !al16(w13) || !al16(w2) || (reinterpret_cast<uintptr_t>(s13) & 3) ||
      (reinterpret_cast<uintptr_t>(s2) & 3))
    return QL_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < ql_workspace_bytes(QL_OP_MOE_MXFP4, M, H, I, E, topk)) return QL_ERR_WORKSPACE;
  if (!al16(workspace)) return QL_ERR_ALIGNMENT;
  cudaStream_t st = (cudaStream_t)stream;
  if (M > 16) {
    // larger batches: grouped tcgen05 GEMMs over the routed experts, 1x128 E4M3 activations
    const Moe3Layout l = moe3_layout(M, H, I, E, topk);
    MoeGroupArgs a = {};
    a.logits = router_logits;
    a.ids_in = topk_ids_in;
    a.w_in = topk_w_in;
    a.M = (int)M;
    a.E = E;
    a.topk = topk;
    a.renorm = renormalize;
    a.ids = at<int32_t>(workspace, l.ids);
    a.wts = at<float>(workspace, l.wts);
    a.counts = at<int32_t>(workspace, l.counts);
    a.ids_dbg = topk_ids_out;
    a.w_dbg = topk_w_out;
    a.status = at<uint32_t>(workspace, 0);
    a.tt = l.tt;
    a.offsets = at<int32_t>(workspace, l.offsets);
    a.tiles = at<int4>(workspace, l.tiles);
    a.ntiles = at<int32_t>(workspace, l.ntiles);
    a.pairs = at<int32_t>(workspace, l.pairs);
    a.pos_of_pair = at<int32_t>(workspace, l.pos);
    a.x = x;
    a.ldx = H;
    a.H = (int)H;
    a.I = (int)I;
    a.q_gu = at<uint8_t>(workspace, l.q_gu);
    a.s_gu = at<uint8_t>(workspace, l.s_gu);
    a.gu = at<float>(workspace, l.gu);
    a.q_dn = at<uint8_t>(workspace, l.q_dn);
    a.s_dn = at<uint8_t>(workspace, l.s_dn);
    a.h_dbg = h_out;
    a.act_alpha = swiglu_alpha;
    a.act_limit = swiglu_limit;
    cudaError_t e = launch_moe_grouped_prologue(a, st);
    if (e != cudaSuccess) return cuda_status(e);
    const int P = (int)(M * topk);
    tc::GemmArgs g = {};
    g.grouped = 1;
    g.fp4 = 1;
    g.experts = E;
    g.tiles = a.tiles;
    g.ntiles = a.ntiles;
    g.tiles_max = l.tiles_max;
    g.tt = l.tt;
    g.pairs = a.pairs;
    g.status = a.status;
    g.wait_limit = g_wait_limit;
    // gate_up: rows [0, 2I) of W13[e] against the dispatch rows' x codes, fp32 rows per pair
    g.M = P;
    g.N = (int)(2 * I);
    g.K = (int)H;
    g.w = w13;
    g.ldw = H / 2;
    g.w_estride = 2 * I * (H / 2);
    g.ws = s13;
    g.lds = H / 32;
    g.s_estride = 2 * I * (H / 32);
    g.aq = a.q_gu;
    g.as = a.s_gu;
    g.out = a.gu;
    g.ld_out = 2 * I;
    e = tc::launch_gemm(g, st);
    if (e == cudaSuccess) e = launch_moe_h_quant(a, st);
    if (e != cudaSuccess) return cuda_status(e);
    // down: rows [0, H) of W2[e] against the dispatch rows' h codes, fp32 rows per pair
    g.N = (int)H;
    g.K = (int)I;
    g.w = w2;
    g.ldw = I / 2;
    g.w_estride = H * (I / 2);
    g.ws = s2;
    g.lds = I / 32;
    g.s_estride = H * (I / 32);
    g.aq = a.q_dn;
    g.as = a.s_dn;
    g.out = at<float>(workspace, l.o);
    g.ld_out = H;
    e = tc::launch_gemm(g, st);
    if (e == cudaSuccess) e = launch_moe_combine(g.out, a.ids, a.wts, (int)M, topk, (int)H, y, st);
    if (e != cudaSuccess) return cuda_status(e);
    if (path_out) *path_out = QL_PATH_MOE_MXFP4_TCGEN05;
    return QL_OK;
  }
  if (M > 8 && moe2_ok(H, I, s13, s2)) {
    // 9..16 tokens: two calls, tokens [0, 8) and [8, M).  Tokens are independent in the layer,
    // and one 8-token MMA tile per call is cheaper than two tiles per expert: the second tile
    // doubles the consumers' MMA and scale-fold work for every routed expert, while the split
    // streams only the experts both halves route to twice (measured at 9 tokens: 8 + 1 tokens
    // took 215 us against 245 us in one call)
    ql_status r = moe_mxfp4_grouped(x, 8, H, router_logits, topk_ids_in, topk_w_in, E, topk, renormalize, w13, s13,
                                    w2, s2, I, swiglu_alpha, swiglu_limit, topk_ids_out, topk_w_out, h_out, y,
                                    workspace, workspace_bytes, stream, path_out);
    if (r != QL_OK) return r;
    const int64_t P8 = (int64_t)8 * topk;
    return moe_mxfp4_grouped(x + 8 * H, M - 8, H, router_logits ? router_logits + 8 * (int64_t)E : nullptr,
                             topk_ids_in ? topk_ids_in + P8 : nullptr, topk_w_in ? topk_w_in + P8 : nullptr, E, topk,
                             renormalize, w13, s13, w2, s2, I, swiglu_alpha, swiglu_limit,
                             topk_ids_out ? topk_ids_out + P8 : nullptr, topk_w_out ? topk_w_out + P8 : nullptr,
                             h_out ? h_out + P8 * I : nullptr, y + 8 * H, workspace, workspace_bytes, stream, path_out);
  }
  if (moe2_ok(H, I, s13, s2)) {
    const Moe2Layout l = moe2_layout(M, H, I, E, topk);
    if ((int64_t)l.slots * (l.gu.nb > l.dn.nb ? l.gu.nb : l.dn.nb) > (int64_t)kMaxTickets) return QL_ERR_UNSUPPORTED;
    cudaError_t e;
    Skinny2Args a = {};
    a.x16 = at<uint16_t>(workspace, l.x16);
    a.tokf = at<float>(workspace, l.tokf);
    a.ready = at<unsigned>(workspace, kReadyOff);
    a.done = at<unsigned>(workspace, kDoneOff);
    a.part = at<float>(workspace, l.part);
    a.tickets = at<unsigned>(workspace, kTicketOff);
    a.status = at<uint32_t>(workspace, 0);
    a.wait_limit = g_wait_limit;
    // routing: done by the gate_up launch (CTA 0 writes the results for down and the combine)
    a.logits = router_logits;
    a.ids_in = topk_ids_in;
    a.w_in = topk_w_in;
    a.renorm = renormalize;
    a.ids_dbg = topk_ids_out;
    a.w_dbg = topk_w_out;
    a.wts = at<float>(workspace, l.wts);
    a.nuniq = at<int32_t>(workspace, l.nuniq);
    a.uniq = at<int32_t>(workspace, l.uniq);
    a.offsets = at<int32_t>(workspace, l.offsets);
    a.pairs = at<int32_t>(workspace, l.pairs);
    a.rows = at<int32_t>(workspace, l.rows);
    a.ids = at<int32_t>(workspace, l.ids);
    a.topk = topk;
    a.E = E;
    a.I = (int)I;
    a.gu = at<float>(workspace, l.gus);
    a.slot_rows = l.slot_rows;
    a.act_alpha = swiglu_alpha;
    a.act_limit = swiglu_limit;
    a.M = (int)M;
    // stage 1: gate and up rows of W13[e] against every token's x
    a.N = (int)(2 * I);
    a.K = (int)H;
    a.x = x;
    a.ldx = H;
    a.img_rows = (int)M;
    a.wsb = s13;
    a.lds = H / 32;
    a.s_estride = 2 * I * (H / 32);
    e = launch_moe2(S2_MOE_GU, l.gu, a, w13, H / 2, 2 * I * (H / 2), E, st);
    if (e != cudaSuccess) return cuda_status(e);
    // stage 2: rows of W2[e] against the gathered h = bf16(swiglu(g, u)) of its pairs
    a.N = (int)H;
    a.K = (int)I;
    a.x = nullptr;
    a.img_rows = l.slots * l.slot_rows;
    a.wsb = s2;
    a.lds = I / 32;
    a.s_estride = H * (I / 32);
    a.h_dbg = h_out;
    a.o = at<float>(workspace, l.o);
    e = launch_moe2(S2_MOE_DN, l.dn, a, w2, I / 2, H * (I / 2), E, st);
    if (e != cudaSuccess) return cuda_status(e);
    e = launch_moe_combine(a.o, a.ids, a.wts, (int)M, topk, (int)H, y, st);
    if (e != cudaSuccess) return cuda_status(e);
    if (path_out) *path_out = QL_PATH_MOE_MXFP4;
    return QL_OK;
  }
  const MoeLayout l = moe_layout(M, H, I, E, topk);
  if ((int64_t)l.umax * (l.nb_gu > l.nb_dn ? l.nb_gu : l.nb_dn) > (int64_t)kMaxTickets) return QL_ERR_UNSUPPORTED;

  MoeRouteArgs r = {};
  r.logits = router_logits;
  r.ids_in = topk_ids_in;
  r.w_in = topk_w_in;
  r.M = (int)M;
  r.E = E;
  r.topk = topk;
  r.renorm = renormalize;
  r.ids = at<int32_t>(workspace, l.ids);
  r.wts = at<float>(workspace, l.wts);
  r.offsets = at<int32_t>(workspace, l.offsets);
  r.pairs = at<int32_t>(workspace, l.pairs);
  r.uniq = at<int32_t>(workspace, l.uniq);
  r.nuniq = at<int32_t>(workspace, l.nuniq);
  r.ids_dbg = topk_ids_out;
  r.w_dbg = topk_w_out;
  r.status = at<uint32_t>(workspace, 0);
  cudaError_t e = launch_moe_route(r, st);
  if (e != cudaSuccess) return cuda_status(e);

  SkinnyArgs a = {};
  a.offsets = r.offsets;
  a.pairs = r.pairs;
  a.uniq = r.uniq;
  a.nuniq = r.nuniq;
  a.topk = topk;
  a.I = (int)I;
  a.h = at<uint16_t>(workspace, l.h);
  a.h_dbg = h_out;
  a.act_alpha = swiglu_alpha;
  a.act_limit = swiglu_limit;
  a.o = at<float>(workspace, l.o);
  a.pdl = 1;
  // gate_up: rows 2I of W13[e], K = H, activations x[m]
  a.w = w13;
  a.ldw = H / 2;
  a.w_estride = 2 * I * (H / 2);
  a.wsb = s13;
  a.lds = H / 32;
  a.s_estride = 2 * I * (H / 32);
  a.x = x;
  a.ldx = H;
  a.M = (int)M;
  a.N = (int)(2 * I);
  a.K = (int)H;
  a.ks = l.gu.ks;
  a.kc = l.gu.kc;
  a.part = at<void>(workspace, l.part_gu);
  a.counters = at<unsigned>(workspace, l.cnt_gu);
  e = launch_skinny(FMT_MXFP4, l.mt, EPI_GATEUP, a, dim3((unsigned)l.nb_gu, (unsigned)l.gu.ks, (unsigned)l.umax), st,
                    true);
  if (e != cudaSuccess) return cuda_status(e);
  // down: rows H of W2[e], K = I, activations h[pair]
  a.w = w2;
  a.ldw = I / 2;
  a.w_estride = H * (I / 2);
  a.wsb = s2;
  a.lds = I / 32;
  a.s_estride = H * (I / 32);
  a.x = at<uint16_t>(workspace, l.h);
  a.ldx = I;
  a.N = (int)H;
  a.K = (int)I;
  a.ks = l.dn.ks;
  a.kc = l.dn.kc;
  a.part = at<void>(workspace, l.part_dn);
  a.counters = at<unsigned>(workspace, l.cnt_dn);
  e = launch_skinny(FMT_MXFP4, l.mt, EPI_DOWN, a, dim3((unsigned)l.nb_dn, (unsigned)l.dn.ks, (unsigned)l.umax), st,
                    true);
  if (e != cudaSuccess) return cuda_status(e);
  e = launch_moe_combine(at<float>(workspace, l.o), r.ids, r.wts, (int)M, topk, (int)H, y, st);
  if (e != cudaSuccess) return cuda_status(e);
  if (path_out) *path_out = QL_PATH_MOE_MXFP4;
  return QL_OK;
}

}  // extern "C"
