/*
 * qlinear.h - C ABI of the GB300 (sm_103a) quantized decode linear layer.
 *
 * Three weight formats of the decode-time weight-quantized linear layer (skinny GEMM,
 * M = 1..256 tokens), as described by the two source pages:
 *   [Z100] "Hygon Z100 (gfx906) vLLM adaptation: full record of optimisation and operator
 *          development (condensed)", chapter 二 (self-written operators) and chapter 三 §2;
 *   [DSV4] "vLLM 0.27.x port: DeepSeek V4 Flash FP4 on Hygon DCU - full report".
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer (cudaMalloc / PyTorch CUDA memory) owned by
 *     the caller; the library never allocates, frees or synchronises, and enqueues all work
 *     on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *   - bf16 tensors are passed as uint16_t bit patterns; fp8 E4M3, packed fp4 E2M1 and
 *     UE8M0 scales as uint8_t bytes.  All matrices are row-major with an explicit leading
 *     dimension (elements for bf16/int8/fp8, BYTES for packed fp4).
 *   - Every argument is validated on the host before any launch.  An invalid call returns
 *     an error status and launches nothing: no device assert, no silent copy ([Z100] §二.2.4
 *     "non-unit inner stride is an explicit error"; [Z100] chapter 四 on skinny kernels that
 *     device-asserted on unsupported sizes).
 *   - `workspace` is caller-owned device scratch of at least ql_workspace_bytes(...) bytes,
 *     16-byte aligned.  It must be zeroed once after allocation (ql_workspace_init); the
 *     kernels leave it reusable.  Calls that share a workspace must not overlap in time.
 *   - `path_out` (nullable HOST pointer) receives the QL_PATH_* code of the kernel sequence
 *     that ran: a dispatch marker, so tests can assert which path was taken.
 *   - Kernels that wait on barriers bound every wait; a wait that runs out sets a flag in
 *     the workspace status word (read it with ql_read_device_status) and the kernel exits
 *     cleanly.  Such a call's outputs are undefined.
 */
#ifndef QLINEAR_H
#define QLINEAR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QL_API __attribute__((visibility("default")))
#else
#define QL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ql_stream_t; /* identical to cudaStream_t */

typedef enum {
  QL_OK = 0,
  QL_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size            */
  QL_ERR_UNSUPPORTED = 2, /* valid but not implemented (shape, block size, mode)      */
  QL_ERR_ALIGNMENT = 3,   /* base pointer / leading dimension not 16-byte aligned     */
  QL_ERR_WORKSPACE = 4,   /* workspace null or smaller than ql_workspace_bytes()      */
  QL_ERR_CUDA = 5,        /* a CUDA runtime call failed (launch error)                */
  QL_ERR_TIMEOUT = 6      /* a bounded device-side wait ran out (ql_read_device_status)*/
} ql_status;

/* operation ids for ql_workspace_bytes */
enum { QL_OP_INT8_W8A8 = 1, QL_OP_FP8_BLOCK = 2, QL_OP_MXFP4 = 3, QL_OP_MOE_MXFP4 = 4, QL_OP_BF16 = 5,
       QL_OP_FP8_CHANNEL = 6 };

/* FP8 weight code formats of qlinear_fp8 */
enum { QL_FP8_E4M3 = 0 /* e4m3fn: bias 7, no infinities, S.1111.111 is NaN */,
       QL_FP8_E5M2 = 1 /* e5m2: bias 15, IEEE-style infinities and NaNs      */ };

/* activation modes of the FP8-block and MXFP4 linears */
enum {
  QL_ACT_BF16 = 0,      /* bf16 activations used as they are (a_s = 1)                        */
  QL_ACT_E4M3_1X128 = 1 /* activations quantised per token and per 128-K group to E4M3 with a
                           UE8M0 power-of-two scale (smallest 2^e with amax <= 448*2^e),
                           [DSV4] §3.3 quant_config "activation_scheme: dynamic, fmt e4m3,
                           scale_fmt ue8m0"                                                   */
};

/* dispatch markers written to *path_out */
enum {
  QL_PATH_NONE = 0,
  QL_PATH_INT8_SKINNY = 1,     /* skinny tensor-core GEMM, per-token INT8 quant in the launch */
  QL_PATH_FP8_SKINNY = 2,      /* FP8 block skinny GEMM, bf16 activations                   */
  QL_PATH_FP8_TCGEN05 = 3,     /* 1x128 act quant + tcgen05 block-scaled GEMM (FP8 x FP8)   */
  QL_PATH_MXFP4_SKINNY = 4,    /* MXFP4 skinny GEMM, bf16 activations                       */
  QL_PATH_MXFP4_TCGEN05 = 5,   /* 1x128 act quant + tcgen05 block-scaled GEMM (E4M3 x E2M1) */
  QL_PATH_MOE_MXFP4 = 6,       /* routing + dispatch + gate_up/SiLU + down + combine         */
  QL_PATH_BF16_SKINNY = 7,     /* BF16 skinny GEMM (unquantised weights)                    */
  QL_PATH_FP8_CHANNEL_SKINNY = 8, /* FP8 skinny GEMM, per-channel / per-tensor fp32 scale    */
  QL_PATH_INT8_TCGEN05 = 9,      /* per-token INT8 quant + tcgen05 GEMM on exact f16 images  */
  QL_PATH_MOE_MXFP4_TCGEN05 = 10 /* M > 16: routing + grouped tcgen05 GEMMs, 1x128 E4M3 act  */
};

/* device status flags (bitmask) */
enum { QL_DEV_TIMEOUT = 1u };

QL_API const char* ql_status_string(ql_status s);
QL_API int ql_version(void);

/*
 * Bytes of workspace the op needs for these sizes.  Every layout starts with the same
 * 256 + 1 MiB: the device status word and counters, then a region that is zero between calls
 * (split-K tickets, or the output cells of INT8 calls of up to 4 tokens), so one workspace can
 * serve calls of any op and shape in turn.  M, N, K as in the op; for
 * QL_OP_MOE_MXFP4: M tokens, N = H (hidden), K = I (expert intermediate), E experts and
 * topk routed experts per token.  Returns 0 for an unknown op or negative sizes.
 */
QL_API size_t ql_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int E, int topk);

/* Zero `bytes` of workspace on `stream` (cudaMemsetAsync).  Call once after allocating. */
QL_API ql_status ql_workspace_init(void* workspace, size_t bytes, ql_stream_t stream);

/*
 * Read (and, if clear != 0, reset) the device status word of `workspace`; synchronises
 * `stream`.  *flags_out receives the QL_DEV_* bits.  Returns QL_ERR_TIMEOUT if the timeout
 * bit was set, QL_OK otherwise.  Test and debugging aid: the compute calls never read it.
 */
QL_API ql_status ql_read_device_status(void* workspace, ql_stream_t stream, int clear, uint32_t* flags_out);

/*
 * Iteration cap of every bounded device wait (default 1<<20 polls).  A test knob: a small
 * cap makes waits run out so the timeout path can be exercised without a hung GPU.
 */
QL_API void ql_set_wait_limit(uint32_t polls);

/*
 * INT8 W8A8 linear with dynamic per-token activation quantisation
 * ([Z100] §二.2 operator table "INT8 W8A8 sdot4" and §二.2.1):
 *   x_s[m]  = max_k |x[m,k]| / 127                       (fp32 IEEE division)
 *   x_q[m,k]= clamp(round_half_even(x[m,k] / x_s[m]), -127, 127)   (0 if x_s == 0)
 *   acc[m,n]= sum_k x_q[m,k] * w[n,k]                    (exact int32)
 *   y[m,n]  = bf16((acc * x_s[m]) * w_s[n])  then, if bias, y = bf16(y + bias[n])
 * x: bf16 [M, ldx] (K used); w: int8 [N, ldw], K-contiguous, used as stored (no transpose,
 * no dequantised copy); w_scale: fp32 [N] (per channel) or [1] (per tensor, w_scale_len == 1);
 * bias: nullable bf16 [N]; y: bf16 [M, ldy].
 * Debug outputs (nullable): acc_out int32 [M, N] (dense, ld N), xq_out int8 [M, K] (ld K),
 * xs_out fp32 [M].
 * Paths: M <= 32 -> the persistent skinny kernel (quantisation fused in, one launch);
 *        M > 32  -> a quantisation launch + the tcgen05 GEMM (kind::f16 MMAs on the exact f16
 *                   values of the codes and weights, drained to int32 every 512 K).
 * Requires: M >= 1, N >= 1, K >= 16, K % 16 == 0, ldx >= K, ldw >= K, ldw % 16 == 0,
 * ldy >= N, 16-byte aligned x and w, |acc| < 2^31 (always true for K <= 133152).
 */
QL_API ql_status qlinear_int8_w8a8(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                            const int8_t* w, int64_t N, int64_t ldw,
                            const float* w_scale, int64_t w_scale_len,
                            const uint16_t* bias, uint16_t* y, int64_t ldy,
                            int32_t* acc_out, int8_t* xq_out, float* xs_out,
                            void* workspace, size_t workspace_bytes, ql_stream_t stream,
                            int* path_out);

/*
 * FP8 E4M3 weights with block UE8M0 scales ([Z100] §二.2.4 "block-scaled (128x128) FP8
 * extension"; chapter 三 §2):
 *   y[m,n] = bf16( sum_kb a_s[m,kb] * 2^(w_scale[n/block_n, kb] - 127)
 *                        * sum_{k in kb} a[m,k] * e4m3(w[n,k]) )   (+ bias after the cast)
 * act_mode QL_ACT_BF16: a = x (bf16), a_s = 1.  QL_ACT_E4M3_1X128: a = e4m3 codes and a_s
 * their UE8M0 scales from the 1x128 quantisation of x (block_k must then be 128).
 * x: bf16 [M, ldx]; w: E4M3 bytes [N, ldw] (padded rows allowed, e.g. ldw = K + 256);
 * w_scale: UE8M0 [ceil(N/block_n), ceil(K/block_k)] row-major; y: bf16 [M, ldy].
 * Debug outputs (nullable, act_mode 1 only): aq_out E4M3 [M, K], as_out UE8M0 [M, ceil(K/128)].
 * Paths: act_mode 0 -> skinny tensor-core kernel (block_n % 16 == 0, block_k % 64 == 0);
 *        act_mode 1 -> tcgen05 block-scaled GEMM (block_n == block_k == 128).
 * Requires K % 16 == 0 (act_mode 1: K % 128 == 0), ldw % 16 == 0, 16-byte aligned x and w.
 */
QL_API ql_status qlinear_fp8_block(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                            const uint8_t* w, int64_t N, int64_t ldw,
                            const uint8_t* w_scale, int block_n, int block_k, int act_mode,
                            const uint16_t* bias, uint16_t* y, int64_t ldy,
                            uint8_t* aq_out, uint8_t* as_out,
                            void* workspace, size_t workspace_bytes, ql_stream_t stream,
                            int* path_out);

/*
 * MXFP4 weights: E2M1 codes packed two per byte (element 2i in the LOW nibble of byte i)
 * with one UE8M0 scale per 32 consecutive K elements of a row ([DSV4] §9.3, MXFP4 expert
 * weights kept in checkpoint format and dequantised on demand):
 *   y[m,n] = bf16( sum_k a[m,k] * e2m1(w[n,k]) * 2^(w_scale[n, k/32] - 127) ) (+ bias)
 * act_mode QL_ACT_BF16: a = x.  QL_ACT_E4M3_1X128: a = e4m3(q[m,k]) * 2^(s[m,k/128]-127).
 * w: [N, ldw_bytes] (K/2 bytes used); w_scale: [N, lds] (K/32 used).
 * Paths: act_mode 0 -> skinny tensor-core kernel; act_mode 1 -> tcgen05 GEMM.
 * Requires K % 32 == 0 (act_mode 1: K % 128 == 0), ldw_bytes % 16 == 0, 16-byte aligned
 * x and w, lds >= K/32 (act_mode 1: lds % 16 == 0 and 16-byte aligned w_scale).
 */
QL_API ql_status qlinear_mxfp4(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                        const uint8_t* w, int64_t N, int64_t ldw_bytes,
                        const uint8_t* w_scale, int64_t lds, int act_mode,
                        const uint16_t* bias, uint16_t* y, int64_t ldy,
                        uint8_t* aq_out, uint8_t* as_out,
                        void* workspace, size_t workspace_bytes, ql_stream_t stream,
                        int* path_out);

/*
 * FP8 weights with one fp32 scale per output channel or per tensor ([Z100] §二.2.2, the
 * emulated FP8 GEMV: e4m3fn or e5m2 codes widened exactly, the scale applied once to the
 * finished dot product):
 *   y[m,n] = bf16( w_scale[n or 0] * sum_k x[m,k] * fp8(w[n,k]) ) (+ bias, added after the
 *   cast and rounded again)
 * x: bf16 [M, ldx] (device); w: FP8 codes [N, ldw] (device, K used, padded rows allowed);
 * w_fmt: QL_FP8_E4M3 or QL_FP8_E5M2; w_scale: fp32 [w_scale_len] (device), w_scale_len = N
 * (per channel) or 1 (per tensor); bias: bf16 [N] or null; y: bf16 [M, ldy] (device).  The
 * caller owns every buffer; nothing is retained after the call returns.  Codes must be finite
 * (NaN / infinity codes propagate through the sum).  Runs the persistent skinny kernel 16
 * tokens at a time, bf16 activations.
 * Requires K % 16 == 0, ldx % 8 == 0, ldw % 16 == 0, 16-byte aligned x and w, ldy >= N;
 * returns QL_ERR_INVALID_ARG / QL_ERR_ALIGNMENT / QL_ERR_UNSUPPORTED before any launch
 * otherwise.  workspace: ql_workspace_bytes(QL_OP_FP8_CHANNEL, M, N, K, 0, 0) bytes, zeroed once.
 */
QL_API ql_status qlinear_fp8(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                      const uint8_t* w, int64_t N, int64_t ldw, int w_fmt,
                      const float* w_scale, int64_t w_scale_len,
                      const uint16_t* bias, uint16_t* y, int64_t ldy,
                      void* workspace, size_t workspace_bytes, ql_stream_t stream,
                      int* path_out);

/*
 * BF16 dense decode GEMV, unquantised weights ([Z100] §二.2.3, the bf16 route: bf16 widened to
 * fp32 exactly, products summed in fp32):
 *   y[m,n] = bf16( sum_k x[m,k] * w[n,k] ) (+ bias, added after the cast and rounded again)
 * x: bf16 [M, ldx] (device), w: bf16 [N, ldw] (device, K used, padded rows allowed), bias:
 * bf16 [N] or null, y: bf16 [M, ldy] (device).  The caller owns every buffer; nothing is
 * retained after the call returns.  Runs the persistent skinny kernel 16 tokens at a time.
 * Requires K % 8 == 0, ldx % 8 == 0, ldw % 8 == 0, 16-byte aligned x and w, ldy >= N; returns
 * QL_ERR_INVALID_ARG / QL_ERR_ALIGNMENT / QL_ERR_UNSUPPORTED before any launch otherwise.
 * workspace: ql_workspace_bytes(QL_OP_BF16, M, N, K, 0, 0) bytes, zeroed once.
 */
QL_API ql_status qlinear_bf16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                       const uint16_t* w, int64_t N, int64_t ldw, const uint16_t* bias,
                       uint16_t* y, int64_t ldy, void* workspace, size_t workspace_bytes,
                       ql_stream_t stream, int* path_out);

/*
 * MXFP4 mixture-of-experts decode layer ([DSV4] §0.1 "M=1 MoE routing Q1", §0.3 grouped
 * batch MoE, §9.3 MXFP4 emulation experts):
 *   routing : p = softmax(router_logits[m, :E]); ids = the topk largest logits (ties go to
 *             the lower expert id), ordered by decreasing logit; weights = p[ids]
 *             (divided by their sum if renormalize != 0).  Alternatively the caller passes
 *             topk_ids_in / topk_w_in and router_logits = NULL (exactly one of the two).
 *             The weights are fp32 exponentials over a float-float sum: within a few fp32
 *             ulps of the exact softmax; the ids depend on logit comparisons only.
 *   dispatch: (token, slot) pairs grouped by expert, pairs of one expert in pair order.
 *   gate_up : for pair (m,j) with expert e: g = W13[e][0:I] x_m, u = W13[e][I:2I] x_m,
 *             h = bf16( silu(alpha * min(g, limit)) * clamp(u, -limit, limit) )
 *             (the clamped SwiGLU of [DSV4] §6.6 / §9.4, alpha = swiglu_alpha, limit =
 *             swiglu_limit; limit = +infinity with alpha = 1 is the plain silu(g) * u)
 *   down    : y[m] = bf16( sum_j weight[m,j] * W2[e_(m,j)] h_(m,j) )
 * x: bf16 [M, H]; router_logits: bf16 [M, E]; topk_ids_in int32 [M, topk];
 * topk_w_in fp32 [M, topk]; w13: [E, 2I, H/2] packed E2M1, s13: [E, 2I, H/32] UE8M0;
 * w2: [E, H, I/2], s2: [E, H, I/32]; y: bf16 [M, H] (dense).
 * Debug outputs (nullable): topk_ids_out int32 [M, topk], topk_w_out fp32 [M, topk],
 * h_out bf16 [M*topk, I] (row m*topk + j).
 * swiglu_alpha must be finite; swiglu_limit >= 0 (+infinity allowed), else QL_ERR_INVALID_ARG.
 * Paths: M <= 16: the persistent skinny kernel with bf16 activations (routing fused into the
 *        gate_up launch), QL_PATH_MOE_MXFP4; 9..16 tokens run as two such calls, tokens
 *        [0, 8) and [8, M) (tokens are independent; one 8-token tile per call is cheaper);
 *        M > 16: grouped tcgen05 GEMMs over the routed experts ([DSV4] §0.3 grouped batch MoE),
 *        QL_PATH_MOE_MXFP4_TCGEN05: x and h are quantised per token and 128-K group to E4M3 with
 *        a UE8M0 scale before their GEMMs (the activation format of qlinear_mxfp4's act_mode 1).
 * Requires 1 <= M <= 65535, 1 <= topk <= min(E, 16), E <= 1024, H % 128 == 0, I % 128 == 0,
 * 16-byte aligned weight pointers.
 */
QL_API ql_status moe_mxfp4_grouped(const uint16_t* x, int64_t M, int64_t H,
                            const uint16_t* router_logits, const int32_t* topk_ids_in,
                            const float* topk_w_in, int E, int topk, int renormalize,
                            const uint8_t* w13, const uint8_t* s13,
                            const uint8_t* w2, const uint8_t* s2, int64_t I,
                            float swiglu_alpha, float swiglu_limit,
                            int32_t* topk_ids_out, float* topk_w_out, uint16_t* h_out,
                            uint16_t* y, void* workspace, size_t workspace_bytes,
                            ql_stream_t stream, int* path_out);

/*
 * Sharded (tensor-parallel) layers.  The pages run these linears split over 2, 4 or 8 GPUs
 * ([Z100] chapter 一 §5, communication and parallelism under TP = 2/4/8; [DSV4] §0, TP = 4/8):
 *   - column-parallel (N split): every shard is a plain call of the entry points above on its
 *     rows of W (FP8 block scales: shard boundaries on whole block_n rows); the concatenated
 *     outputs are the unsharded layer's outputs, bit for bit.
 *   - row-parallel (K split): every shard holds a K range of W and of x (FP8 block: whole
 *     block_k ranges; MXFP4: whole 256-K units, so its scale rows stay whole bytes per shard).
 *     INT8: each shard's ql_token_amax, an all-reduce MAX across shards, then
 *     qlinear_int8_w8a8_partial on each shard with that amax (its codes are then exactly the
 *     unsharded codes), an all-reduce SUM of the int32 sums (exact) and qlinear_int8_epilogue:
 *     the result equals the unsharded call's bit for bit.  FP8 / MXFP4: each shard's fp32
 *     partial sums (the *_partial entry points), an all-reduce SUM, then ql_finish_f32 rounds
 *     once to bf16 and adds the bias.  The collectives are the caller's (NCCL, gloo, ...).
 * Pointers are device pointers owned by the caller; nothing is allocated or retained.
 */

/* Per-token amax of a K shard: amax_out[m] = max_k |x[m,k]| (fp32 [M]).  K % 8 == 0,
 * 16-byte aligned x, ldx % 8 == 0. */
QL_API ql_status ql_token_amax(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float* amax_out,
                               ql_stream_t stream);

/* A K shard of a row-parallel INT8 W8A8 layer: x_s[m] = amax[m] / 127 (amax: the tokens'
 * amax over the whole row, fp32 [M]), codes as in qlinear_int8_w8a8, and the exact int32
 * sums over this shard's K written to acc_out [M, N] (dense, required); no epilogue, no y.
 * xq_out (nullable) receives the codes.  Same requirements and workspace as
 * qlinear_int8_w8a8. */
QL_API ql_status qlinear_int8_w8a8_partial(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                           const int8_t* w, int64_t N, int64_t ldw, const float* amax,
                                           int32_t* acc_out, int8_t* xq_out, void* workspace,
                                           size_t workspace_bytes, ql_stream_t stream, int* path_out);

/* The INT8 epilogue on int32 sums added over the shards: y = bf16((acc * x_s) * w_s) (+ bias
 * after the cast), x_s = amax / 127 (IEEE fp32 division), acc int32 [M, N] dense. */
QL_API ql_status qlinear_int8_epilogue(const int32_t* acc, int64_t M, int64_t N, const float* amax,
                                       const float* w_scale, int64_t w_scale_len, const uint16_t* bias,
                                       uint16_t* y, int64_t ldy, ql_stream_t stream);

/* A K shard of a row-parallel FP8-block layer (bf16 activations): y32[m,n] = the fp32 sum of
 * this shard's scaled block products (no bias), [M, ldy32].  block_k a power of two >= 64,
 * block_n % 16 == 0; otherwise as qlinear_fp8_block with act_mode QL_ACT_BF16. */
QL_API ql_status qlinear_fp8_block_partial(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                           const uint8_t* w, int64_t N, int64_t ldw, const uint8_t* w_scale,
                                           int block_n, int block_k, float* y32, int64_t ldy32,
                                           void* workspace, size_t workspace_bytes, ql_stream_t stream,
                                           int* path_out);

/* A K shard of a row-parallel MXFP4 layer (bf16 activations): fp32 partial sums into y32
 * [M, ldy32], no bias.  K % 256 == 0, lds % 8 == 0 and 8-byte aligned w_scale (else
 * QL_ERR_UNSUPPORTED); otherwise as qlinear_mxfp4 with act_mode QL_ACT_BF16. */
QL_API ql_status qlinear_mxfp4_partial(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                       const uint8_t* w, int64_t N, int64_t ldw_bytes, const uint8_t* w_scale,
                                       int64_t lds, float* y32, int64_t ldy32, void* workspace,
                                       size_t workspace_bytes, ql_stream_t stream, int* path_out);

/* One bf16 rounding of fp32 sums added over the shards, then + bias (after the cast, rounded
 * again): y[m,n] = bf16(bf16(y32[m,n]) + bias[n]). */
QL_API ql_status ql_finish_f32(const float* y32, int64_t M, int64_t N, int64_t ld32, const uint16_t* bias,
                               uint16_t* y, int64_t ldy, ql_stream_t stream);

/*
 * INT8 W8A8 linear that allocates nothing and takes no workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot give the library device
 * memory - hosts without a device allocator of their own, plugins inside a framework that
 * has reserved all GPU memory for its pool and forbids new cudaMalloc calls, and latency-
 * critical paths that must not call cudaMalloc/cudaFree because those can synchronise the
 * device.  It computes exactly what qlinear_int8_w8a8 computes (same arguments, minus the
 * workspace) and takes its scratch from a 16 MiB array in the library's own device memory,
 * held on every GPU that loads the library until the process exits.
 *   - The first call on each device looks up that array's device address (with the device
 *     current) and caches it; make that first call before any stream capture.
 *   - Sizes whose scratch need (ql_workspace_bytes(QL_OP_INT8_W8A8, M, N, K, 0, 0)) exceeds
 *     16 MiB are rejected with QL_ERR_WORKSPACE; nothing is launched.
 *   - All calls on a device share the array: each call clears what must start at zero on its
 *     stream, and calls that overlap on the GPU (unordered streams) race on it.
 *   - It never calls cudaMalloc, cudaFree or any allocating routine.
 */
QL_API ql_status qlinear_int8_w8a8_noalloc(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                           const int8_t* w, int64_t N, int64_t ldw,
                                           const float* w_scale, int64_t w_scale_len,
                                           const uint16_t* bias, uint16_t* y, int64_t ldy,
                                           int32_t* acc_out, int8_t* xq_out, float* xs_out,
                                           ql_stream_t stream, int* path_out);

#ifdef __cplusplus
}
#endif
#endif /* QLINEAR_H */
