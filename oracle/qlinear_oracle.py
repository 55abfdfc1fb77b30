"""Plain CPU oracle of the quantized decode linear layer (INT8 W8A8, FP8 128x128 block,
MXFP4 MoE, 1x128 E4M3 activation quantisation).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module.  It shares no code with the CUDA library: the two
meet only through the seeded inputs of ``synth``.

Each function is the definition from the pages written out directly in fp64 (or in the
precision the definition fixes), with a numpy matmul as the only library step; no blocking,
fusion or reordering beyond what the definition states.  Sources:
  [Z100]  "Hygon Z100 (gfx906) vLLM adaptation: full record of optimisation and operator
          development (condensed)"
  [DSV4]  "vLLM 0.27.x port: DeepSeek V4 Flash FP4 on Hygon DCU - full report"

Readings taken where the pages are silent (each is listed with its reason in the design
notes of the repository):
  * INT8 activation scale and quotient are IEEE fp32 divisions, rounding half-to-even,
    clamp to +-127, all-zero token -> scale 0 and codes 0.
  * 1x128 activation scale = smallest power of two 2^e with amax <= 448 * 2^e (so no code
    saturates), e clamped to >= -127; codes round to nearest even, signed zeros kept.
  * MXFP4: low nibble = even K index; W13 rows [0, I) are gate, [I, 2I) are up.
  * Routing: softmax over all experts, top-k by logit value with ties to the lower expert
    index, weights = softmax probabilities, no renormalisation unless asked.
  * The expert intermediate h is rounded to bf16 (the pages compute experts in BF16).
Parity pins: every function below is checked by ``tests/test_oracle_*.py`` against values
fixed by the pages or by mathematics (closed forms, brute force, special cases).
"""
from __future__ import annotations

import numpy as np

from .formats import (
    bf16_to_f32,
    bf16_to_f64,
    e2m1_decode,
    e4m3_decode,
    e4m3_encode_rne_sat,
    e5m2_decode,
    round_to_bf16,
    unpack_e2m1,
    ue8m0_decode,
)

INT32_MAX = 2 ** 31 - 1


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


# ----------------------------------------------------------------------------------------
# INT8 W8A8 ([Z100] §二.2.1 "INT8 W8A8 sdot4" and the operator table of §二.2)
# ----------------------------------------------------------------------------------------


def quant_int8_per_token(x_bits, amax=None):
    """Dynamic symmetric per-token INT8 quantisation of bf16 activations.

    For each token m: amax = max_k |x[m,k]| (exact in fp32), x_s = amax / 127 and
    x_q = round_half_even(x / x_s) clamped to [-127, 127], both divisions IEEE fp32.
    A token whose amax is 0 gets x_s = 0 and x_q = 0.  Returns (x_q int8 [M,K], x_s fp32 [M]).
    ``amax`` (optional, fp32 [M]) is the tokens' amax taken over a wider K than ``x_bits``
    holds: a K slice of a row-parallel layer quantises with the whole row's scale.
    """
    xf = bf16_to_f32(x_bits)
    if amax is None:
        amax = np.max(np.abs(xf), axis=1).astype(np.float32)
    amax = np.asarray(amax, dtype=np.float32).reshape(-1)
    xs = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(xs > 0, xs, np.float32(1.0)).astype(np.float32)
    quo = (xf / safe[:, None]).astype(np.float32)
    q = np.clip(np.rint(quo), -127, 127)
    q = np.where(xs[:, None] > 0, q, 0).astype(np.int8)
    return q, xs


def int8_accumulate(x_q, w):
    """acc[m,n] = sum_k x_q[m,k] * w[n,k] as an exact integer (int64), checked to fit int32
    (the pages accumulate in int32 exactly)."""
    acc = np.asarray(x_q, dtype=np.int64) @ np.asarray(w, dtype=np.int64).T
    assert np.all(np.abs(acc) <= INT32_MAX), "int32 accumulator would overflow"
    return acc


def int8_epilogue(acc, x_s, w_s, bias_bits=None):
    """y = bf16((acc * x_s) * w_s), then + bias after the cast ([Z100] §二.2: the epilogue
    order "(acc*x_s)*w_s -> cast -> +bias").  x_s is [M] or [1], w_s is [N] or [1].
    Evaluated exactly in fp64 from the fp32 factors, rounded once to bf16."""
    acc = np.asarray(acc, dtype=np.float64)
    xs = np.asarray(x_s, dtype=np.float32).astype(np.float64).reshape(-1)
    ws = np.asarray(w_s, dtype=np.float32).astype(np.float64).reshape(-1)
    y = (acc * xs[:, None]) * ws[None, :]
    yb = round_to_bf16(y)
    if bias_bits is not None:
        yb = round_to_bf16(bf16_to_f64(yb) + bf16_to_f64(bias_bits)[None, :])
    return yb


def int8_w8a8(x_bits, w, w_s, bias_bits=None, rows=None, amax=None):
    """Whole INT8 W8A8 linear: quantise x, accumulate exactly, epilogue.

    ``rows`` (optional) restricts the computation to those output columns n; ``amax``
    (optional) is the per-token amax to quantise with (see quant_int8_per_token).
    Returns dict with x_q, x_s, acc [M,len(rows)], y bits, and the error scale
    sum_k |x_deq * w_deq| used by the float tolerance."""
    w = np.asarray(w, dtype=np.int8)
    w_s = np.asarray(w_s, dtype=np.float32).reshape(-1)
    if rows is not None:
        rows = np.asarray(rows)
        w = w[rows]
        w_s = w_s[rows] if w_s.size > 1 else w_s
        if bias_bits is not None:
            bias_bits = np.asarray(bias_bits)[rows]
    x_q, x_s = quant_int8_per_token(x_bits, amax)
    acc = int8_accumulate(x_q, w)
    y = int8_epilogue(acc, x_s, w_s, bias_bits)
    abs_acc = np.abs(x_q.astype(np.int64)) @ np.abs(w.astype(np.int64)).T
    ws64 = w_s.astype(np.float64)
    err_scale = abs_acc * x_s.astype(np.float64)[:, None] * (ws64[None, :] if ws64.size > 1 else ws64[0])
    return {"x_q": x_q, "x_s": x_s, "acc": acc, "y": y, "abs_sum": err_scale}


# ----------------------------------------------------------------------------------------
# FP8 E4M3 weights with 128x128 UE8M0 block scales ([Z100] §二.2.4 "block-scaled (128x128)
# FP8 extension" and chapter 三 §2): out[m,n] = sum_kb (sum_{k in kb} a[m,k] w[n,k])
#                                                      * a_s[m,kb] * w_s[n // block_n, kb]
# ----------------------------------------------------------------------------------------


def fp8_block(x, w_codes, w_scale_bytes, K, block_n=128, block_k=128, a_scale=None, rows=None):
    """Block-scaled FP8 linear, evaluated block by block exactly as the formula reads.

    x: activations as fp64 values [M, K] (bf16 activations decoded exactly, or E4M3 codes
       already decoded);
    w_codes: E4M3 bytes [N, ldw] (only the first K columns are used: padded rows allowed);
    w_scale_bytes: UE8M0 [ceil(N/block_n), ceil(K/block_k)], row-major;
    a_scale: optional fp64 [M, ceil(K/block_k)] per-token per-block activation scales
             (absent = 1, the bf16-activation case).
    Returns (y fp64 [M, len(rows)], abs_sum fp64 [M, len(rows)]) where abs_sum is
    sum_k |x*w*scales|, the error scale of the float tolerance.
    """
    x = np.asarray(x, dtype=np.float64)
    M = x.shape[0]
    w_codes = np.asarray(w_codes, dtype=np.uint8)
    N = w_codes.shape[0]
    rows = np.arange(N) if rows is None else np.asarray(rows)
    wv = e4m3_decode(w_codes[rows, :K])              # [R, K]
    sb = np.asarray(w_scale_bytes, dtype=np.uint8)
    nkb = _cdiv(K, block_k)
    y = np.zeros((M, rows.size))
    a = np.zeros((M, rows.size))
    for kb in range(nkb):
        ks = slice(kb * block_k, min(K, (kb + 1) * block_k))
        part = x[:, ks] @ wv[:, ks].T
        apart = np.abs(x[:, ks]) @ np.abs(wv[:, ks]).T
        ws = ue8m0_decode(sb[rows // block_n, kb])    # [R]
        asc = np.ones(M) if a_scale is None else np.asarray(a_scale, dtype=np.float64)[:, kb]
        y += part * ws[None, :] * asc[:, None]
        a += apart * ws[None, :] * asc[:, None]
    return y, a


# ----------------------------------------------------------------------------------------
# FP8 weights with per-tensor / per-channel scales ([Z100] §二.2.2, the emulated FP8 GEMV:
# e4m3fn or e5m2 codes, one fp32 scale per output channel or for the whole tensor, applied a
# single time to the finished dot product).
#   y[m, n] = w_s[n] * sum_k x[m, k] * fp8(w[n, k])
# ----------------------------------------------------------------------------------------


def fp8_channel(x_bits, w_codes, w_fmt, w_s, K, rows=None):
    """x_bits: bf16 [M, K]; w_codes: FP8 bytes [N, ldw] (first K used); w_fmt: "e4m3" or
    "e5m2"; w_s: fp32 [N] (per channel) or [1] (per tensor).  Returns (y fp64 [M, R],
    abs_sum fp64 [M, R]) with abs_sum = |w_s| sum_k |x w|, the float tolerance's scale."""
    x = bf16_to_f64(np.asarray(x_bits)[:, :K])
    w_codes = np.asarray(w_codes, dtype=np.uint8)
    rows = np.arange(w_codes.shape[0]) if rows is None else np.asarray(rows)
    dec = e4m3_decode if w_fmt == "e4m3" else e5m2_decode
    w = dec(w_codes[rows, :K])
    ws = np.asarray(w_s, dtype=np.float64)
    s = ws[rows] if ws.size > 1 else np.full(rows.size, ws[0])
    return (x @ w.T) * s[None, :], (np.abs(x) @ np.abs(w).T) * np.abs(s)[None, :]


# ----------------------------------------------------------------------------------------
# BF16 dense decode GEMV ([Z100] §二.2.3, the bf16 route: bf16 values widen to fp32 exactly and
# are multiplied and summed).  y[m, n] = sum_k x[m, k] w[n, k], both operands bf16.
# ----------------------------------------------------------------------------------------


def bf16_linear(x_bits, w_bits, K, rows=None):
    """Unquantised linear on bf16 operands, exact in fp64.

    x_bits: bf16 bits [M, K]; w_bits: bf16 bits [N, ldw] (only the first K columns are used:
    padded rows allowed).  Returns (y fp64 [M, len(rows)], abs_sum fp64 [M, len(rows)]) with
    abs_sum = sum_k |x w|, the error scale of the float tolerance."""
    x = bf16_to_f64(np.asarray(x_bits)[:, :K])
    w_bits = np.asarray(w_bits)
    rows = np.arange(w_bits.shape[0]) if rows is None else np.asarray(rows)
    w = bf16_to_f64(w_bits[rows, :K])
    return x @ w.T, np.abs(x) @ np.abs(w).T


# ----------------------------------------------------------------------------------------
# 1x128 dynamic E4M3 activation quantisation with UE8M0 scales ([DSV4] §3.3 quant_config:
# activation_scheme dynamic, fmt e4m3, scale_fmt ue8m0; [Z100] §二.2.4 a_s[m, kb]).
# ----------------------------------------------------------------------------------------


def ue8m0_exponent_for(amax):
    """Smallest integer e with amax <= 448 * 2^e (exact comparison), clamped to >= -127.
    amax == 0 gives e = 0 (scale byte 127)."""
    amax = np.asarray(amax, dtype=np.float64)
    pos = amax > 0
    safe = np.where(pos, amax, 448.0)
    _, e0 = np.frexp(safe / 448.0)                # estimate; corrected by exact tests below
    e = e0.astype(np.int64)
    for _ in range(3):
        too_small = safe > 448.0 * np.ldexp(1.0, e)          # needs a larger scale
        e = np.where(too_small, e + 1, e)
    for _ in range(3):
        fits_lower = safe <= 448.0 * np.ldexp(1.0, e - 1)    # a smaller scale still fits
        e = np.where(fits_lower, e - 1, e)
    e = np.where(pos, e, 0)
    return np.maximum(e, -127)


def quant_e4m3_1x128(x_bits, group=128):
    """Per-token, per-128-K-group E4M3 quantisation with a UE8M0 (power-of-two) scale.

    Returns (q E4M3 bytes [M, K], s UE8M0 bytes [M, ceil(K/group)])."""
    x = bf16_to_f64(x_bits)
    M, K = x.shape
    ng = _cdiv(K, group)
    q = np.zeros((M, K), dtype=np.uint8)
    s = np.zeros((M, ng), dtype=np.uint8)
    for g in range(ng):
        ks = slice(g * group, min(K, (g + 1) * group))
        amax = np.max(np.abs(x[:, ks]), axis=1)
        e = ue8m0_exponent_for(amax)
        s[:, g] = (127 + e).astype(np.uint8)
        q[:, ks] = e4m3_encode_rne_sat(np.ldexp(x[:, ks], -e[:, None]))
    return q, s


def fp8_block_act_quant(x_bits, w_codes, w_scale_bytes, K, block_n=128, block_k=128, rows=None):
    """FP8 block linear with 1x128 E4M3 activations: quantise, then the block formula with
    a_s[m, kb] = 2^(s[m,kb] - 127)."""
    q, s = quant_e4m3_1x128(x_bits, block_k)
    y, a = fp8_block(e4m3_decode(q), w_codes, w_scale_bytes, K, block_n, block_k,
                     a_scale=ue8m0_decode(s), rows=rows)
    return {"q": q, "s": s, "y_f64": y, "abs_sum": a, "y": round_to_bf16(y)}


# ----------------------------------------------------------------------------------------
# MXFP4 dense linear: E2M1 weights with one UE8M0 scale per 32 K-elements per row
# ([DSV4] §9.3 MXFP4 experts kept in checkpoint format and dequantised on demand).
# ----------------------------------------------------------------------------------------


def mxfp4_dequant(w_packed, w_scale_bytes):
    """Packed E2M1 [R, K/2] + UE8M0 [R, K/32] -> fp64 [R, K]: e2m1(code) * 2^(s[r, k//32]-127)."""
    codes = unpack_e2m1(w_packed)
    v = e2m1_decode(codes)
    sc = ue8m0_decode(np.asarray(w_scale_bytes, dtype=np.uint8))
    return v * np.repeat(sc, 32, axis=1)[:, : v.shape[1]]


def mxfp4_act_quant(x_bits, w_packed, w_scale_bytes, rows=None, group=128):
    """MXFP4-weight linear with 1x128 E4M3 activations:
    y[m,n] = sum_k (e4m3(q[m,k]) * 2^(s_a[m, k//128]-127)) * w_deq[n,k]."""
    q, s = quant_e4m3_1x128(x_bits, group)
    wp = np.asarray(w_packed, dtype=np.uint8)
    ws = np.asarray(w_scale_bytes, dtype=np.uint8)
    if rows is not None:
        wp, ws = wp[rows], ws[rows]
    K = q.shape[1]
    a = e4m3_decode(q) * np.repeat(ue8m0_decode(s), group, axis=1)[:, :K]
    w = mxfp4_dequant(wp, ws)
    y = a @ w.T
    absum = np.abs(a) @ np.abs(w).T
    return {"q": q, "s": s, "y_f64": y, "abs_sum": absum, "y": round_to_bf16(y)}


# ----------------------------------------------------------------------------------------
# MoE: softmax top-k routing ([DSV4] §0.1 "M=1 MoE routing Q1"; the formula is the plain
# softmax-then-top-k reading), then MXFP4 experts gate_up -> SiLU*mul -> down, weighted sum.
# The clamped SwiGLU of [DSV4] §6.6 (J09, the SwiGLU fallback fix) and §9.4 (SwiGLU parameters
# matching the model config, alpha = 1.0 and limit = 10.0) is the optional activation: the gate
# is capped from above at limit, up is clipped to [-limit, limit], and the activation is
# silu(alpha * gate) * up.  Without a limit (and alpha = 1) it is the plain SiLU*mul.
# ----------------------------------------------------------------------------------------


def route_topk(logits_bits, topk, renormalize=False):
    """p = softmax(logits) in fp64; ids = the topk largest logits (ties -> lower expert id),
    ordered by decreasing logit; weights = p[ids] (divided by their sum if renormalize)."""
    lg = bf16_to_f64(logits_bits)
    M, E = lg.shape
    mx = lg.max(axis=1, keepdims=True)
    ex = np.exp(lg - mx)
    p = ex / ex.sum(axis=1, keepdims=True)
    ids = np.zeros((M, topk), dtype=np.int32)
    for m in range(M):
        order = sorted(range(E), key=lambda e: (-lg[m, e], e))
        ids[m] = order[:topk]
    w = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return ids, w


def dispatch(ids, num_experts):
    """Group (token, slot) pairs by expert: offsets [E+1] and pair list (pair = m*topk + j),
    pairs of one expert in increasing pair order (a stable counting sort)."""
    flat = np.asarray(ids).reshape(-1)
    counts = np.bincount(flat, minlength=num_experts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    pairs = np.argsort(flat, kind="stable").astype(np.int32)
    return offsets, pairs


def silu(g):
    return g / (1.0 + np.exp(-g))


def swiglu(g, u, alpha=1.0, limit=None):
    """silu(alpha * min(g, limit)) * clip(u, -limit, limit); limit None: no clamp."""
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    if limit is not None:
        g = np.minimum(g, limit)
        u = np.clip(u, -limit, limit)
    return silu(alpha * g) * u


def moe_gate_up(x_bits, ids, w13, s13, I, pairs=None, cols=None, alpha=1.0, limit=None):
    """Stage 1 for each (token m, slot j) pair: gu = W13[e] x_m with the dequantised expert,
    g = gu[:I], u = gu[I:], h = bf16(swiglu(g, u, alpha, limit)) (plain silu(g) * u by default).

    pairs: optional list of pair indices p = m*topk + j to evaluate (default all);
    cols:  optional intermediate indices i to evaluate (default all I).
    Returns dict of fp64 g, u, h_f64, bits h, and the error scales G = sum|w1 x|,
    U = sum|w3 x| per entry; arrays are [len(pairs), len(cols)]."""
    x = bf16_to_f64(x_bits)
    M, topk = ids.shape
    pairs = np.arange(M * topk) if pairs is None else np.asarray(pairs)
    cols = np.arange(I) if cols is None else np.asarray(cols)
    rows = np.concatenate([cols, I + cols])
    out = {k: np.zeros((pairs.size, cols.size)) for k in ("g", "u", "G", "U")}
    cache = {}
    for pi, p in enumerate(pairs):
        m, j = divmod(int(p), topk)
        e = int(ids[m, j])
        if e not in cache:
            cache = {e: mxfp4_dequant(np.asarray(w13[e])[rows], np.asarray(s13[e])[rows])}
        W = cache[e]
        gu = W @ x[m]
        au = np.abs(W) @ np.abs(x[m])
        n = cols.size
        out["g"][pi], out["u"][pi] = gu[:n], gu[n:]
        out["G"][pi], out["U"][pi] = au[:n], au[n:]
    out["h_f64"] = swiglu(out["g"], out["u"], alpha, limit)
    out["h"] = round_to_bf16(out["h_f64"])
    return out


def moe_down_combine(h_bits, ids, weights, w2, s2, rows=None):
    """Stage 2: o_p = W2[e_p] h_p for each pair, y[m] = bf16(sum_j weights[m,j] * o_(m,j)).

    h_bits: bf16 [M*topk, I] (pair-major, pair = m*topk + j); rows: optional output
    indices n.  Returns (y bits [M, R], y fp64, abs_sum = sum_j |w_j| sum_i |W2 h|)."""
    h = bf16_to_f64(h_bits)
    M, topk = ids.shape
    H = np.asarray(w2[0]).shape[0]
    rows = np.arange(H) if rows is None else np.asarray(rows)
    y = np.zeros((M, rows.size))
    a = np.zeros((M, rows.size))
    for m in range(M):
        for j in range(topk):
            e = int(ids[m, j])
            W = mxfp4_dequant(np.asarray(w2[e])[rows], np.asarray(s2[e])[rows])
            hp = h[m * topk + j]
            y[m] += weights[m, j] * (W @ hp)
            a[m] += abs(weights[m, j]) * (np.abs(W) @ np.abs(hp))
    return round_to_bf16(y), y, a


def moe_mxfp4(x_bits, logits_bits, w13, s13, w2, s2, I, topk, renormalize=False, alpha=1.0, limit=None):
    """Whole MoE layer at a size the oracle finishes quickly (all pairs, all outputs)."""
    ids, w = route_topk(logits_bits, topk, renormalize)
    st1 = moe_gate_up(x_bits, ids, w13, s13, I, alpha=alpha, limit=limit)
    y, y64, a = moe_down_combine(st1["h"], ids, w, w2, s2)
    return {"ids": ids, "weights": w, "stage1": st1, "y": y, "y_f64": y64, "abs_sum": a}


# ----------------------------------------------------------------------------------------
# Grouped MoE for larger batches with 1x128 E4M3 activations ([DSV4] §0.3, the grouped batch
# MoE path, with the activation format of the block-scaled GEMM): routing as above; each routed
# token's x quantised per 128-K group to E4M3 with a UE8M0 scale; gate/up sums on those
# activations; h = bf16(swiglu(g, u)); h itself quantised per 128-K group; down on that; the
# weighted combine.
# ----------------------------------------------------------------------------------------


def moe_mxfp4_act_quant(x_bits, logits_bits, w13, s13, w2, s2, I, topk, renormalize=False, alpha=1.0,
                        limit=None, ids=None, weights=None):
    """Whole layer with quantised activations at both GEMMs.  Returns routing, the stage-1
    values (g, u fp64 and their error scales G, U, h bits and fp64), and the stage-2 results
    (y bits, y fp64, abs_sum) computed from the oracle's own h."""
    if ids is None:
        ids, weights = route_topk(logits_bits, topk, renormalize)
    st1 = moe_gate_up_act_quant(x_bits, ids, w13, s13, I, alpha=alpha, limit=limit)
    yb, y64, a = moe_down_combine_act_quant(st1["h"], ids, weights, w2, s2)
    return {"ids": ids, "weights": weights, "stage1": st1, "y": yb, "y_f64": y64, "abs_sum": a}


def moe_gate_up_act_quant(x_bits, ids, w13, s13, I, pairs=None, cols=None, alpha=1.0, limit=None):
    """Stage 1 on 1x128-quantised activations: a = e4m3(q) * 2^(s-127) per token, then for each
    (token m, slot j) pair g = W13[e][:I] a_m, u = W13[e][I:] a_m and h = bf16(swiglu(g, u))."""
    q, s = quant_e4m3_1x128(x_bits)
    H = q.shape[1]
    a = e4m3_decode(q) * np.repeat(ue8m0_decode(s), 128, axis=1)[:, :H]
    M, topk = ids.shape
    pairs = np.arange(M * topk) if pairs is None else np.asarray(pairs)
    cols = np.arange(I) if cols is None else np.asarray(cols)
    rows = np.concatenate([cols, I + cols])
    out = {k: np.zeros((pairs.size, cols.size)) for k in ("g", "u", "G", "U")}
    for pi, p in enumerate(pairs):
        m, j = divmod(int(p), topk)
        W = mxfp4_dequant(np.asarray(w13[int(ids[m, j])])[rows], np.asarray(s13[int(ids[m, j])])[rows])
        gu, au = W @ a[m], np.abs(W) @ np.abs(a[m])
        n = cols.size
        out["g"][pi], out["u"][pi] = gu[:n], gu[n:]
        out["G"][pi], out["U"][pi] = au[:n], au[n:]
    out["h_f64"] = swiglu(out["g"], out["u"], alpha, limit)
    out["h"] = round_to_bf16(out["h_f64"])
    out["q"], out["s"] = q, s
    return out


def moe_down_combine_act_quant(h_bits, ids, weights, w2, s2, rows=None):
    """Stage 2 on 1x128-quantised h: o_p = W2[e_p] a2_p with a2 = e4m3(q) * 2^(s-127) of each
    pair's h row, y[m] = bf16(sum_j weights[m,j] o_(m,j)).  Returns (y bits, y fp64, abs_sum)."""
    q, s = quant_e4m3_1x128(h_bits)
    I = q.shape[1]
    a2 = e4m3_decode(q) * np.repeat(ue8m0_decode(s), 128, axis=1)[:, :I]
    M, topk = ids.shape
    H = np.asarray(w2[0]).shape[0]
    rows = np.arange(H) if rows is None else np.asarray(rows)
    weights = np.asarray(weights, dtype=np.float64)
    y = np.zeros((M, rows.size))
    ab = np.zeros((M, rows.size))
    for m in range(M):
        for j in range(topk):
            e = int(ids[m, j])
            W = mxfp4_dequant(np.asarray(w2[e])[rows], np.asarray(s2[e])[rows])
            hp = a2[m * topk + j]
            y[m] += weights[m, j] * (W @ hp)
            ab[m] += abs(weights[m, j]) * (np.abs(W) @ np.abs(hp))
    return round_to_bf16(y), y, ab
