"""Number formats used by the quantized decode linear layer, decoded from their definitions.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module; only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.

Sources (page titles as cited throughout the oracle):
  [Z100]  "Hygon Z100 (gfx906) vLLM adaptation: full record of optimisation and operator
          development (condensed)", chapter 二 (self-written HIP operators).
  [DSV4]  "vLLM 0.27.x port: DeepSeek V4 Flash FP4 on Hygon DCU - full report".

Every function here is the plain definition, vectorised with numpy, evaluated in fp64
(all values involved are exactly representable in fp64).
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------------------
# bfloat16
# ----------------------------------------------------------------------------------------


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values (bf16 is the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def round_to_bf16(v) -> np.ndarray:
    """Round exact fp64 values to bf16 (round to nearest, ties to even); returns bit patterns.

    bf16 keeps 8 significant bits; normal exponents reach down to 2^-126 and the subnormal
    quantum is 2^-133.  The value is divided by its quantum (a power of two, exact), rounded
    half-to-even with ``np.rint`` and scaled back.  Results of magnitude >= 2^128 overflow to
    infinity, as round-to-nearest does.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.float64)
    fin = np.isfinite(v)
    a = np.abs(np.where(fin, v, 0.0))
    _, e = np.frexp(a)                     # a = f * 2^e, f in [0.5, 1)
    q_exp = np.maximum(e - 1 - 7, -133)    # quantum of the 8-bit significand
    r = np.rint(np.ldexp(np.where(fin, v, 0.0), -q_exp))
    out = np.ldexp(r, q_exp)
    out = np.where(np.abs(out) >= 2.0 ** 128, np.copysign(np.inf, out), out)
    out = np.where(fin, out, v)
    f32 = out.astype(np.float32)           # exact: every value here is a bf16 value
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(v)
    if np.any(nan):
        bits = np.where(nan, np.uint16(0x7FC0), bits)
    return bits


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 values at |v| (the unit in the last place of an 8-bit significand)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(a)
    return np.ldexp(1.0, np.maximum(e - 1, -126) - 7)


# ----------------------------------------------------------------------------------------
# OCP FP8 E4M3 ("E4M3FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities,
# S.1111.111 is NaN, largest finite 448.  [DSV4] names the format ("manual OCP E4M3 decode"),
# [Z100] §二.2.2 warns that exponent-0 codes are subnormal and break shift-and-rebias tricks.
# ----------------------------------------------------------------------------------------


def e4m3_value(code: int) -> float:
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** -6
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


# ----------------------------------------------------------------------------------------
# OCP FP8 E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits, IEEE-style: exponent 31 with
# mantissa 0 is infinity, otherwise NaN; largest finite 57344.  [Z100] §二.2.2 names both
# e4m3fn and e5m2 weights for the per-tensor / per-channel FP8 GEMV.
# ----------------------------------------------------------------------------------------


def e5m2_value(code: int) -> float:
    s = (code >> 7) & 1
    e = (code >> 2) & 0x1F
    m = code & 0x3
    if e == 0x1F:
        mag = float("inf") if m == 0 else float("nan")
    elif e == 0:
        mag = (m / 4.0) * 2.0 ** -14
    else:
        mag = (1.0 + m / 4.0) * 2.0 ** (e - 15)
    return -mag if s else mag


E5M2_TABLE = np.array([e5m2_value(c) for c in range(256)], dtype=np.float64)


def e5m2_decode(codes) -> np.ndarray:
    return E5M2_TABLE[np.asarray(codes, dtype=np.uint8)]


# non-negative finite magnitudes in code order 0x00..0x7E (monotone increasing)
_E4M3_POS = E4M3_TABLE[:0x7F].copy()


def e4m3_encode_rne_sat(t) -> np.ndarray:
    """Nearest E4M3 code to each fp64 value (ties to the even code), saturating at +-448.

    Brute force over the 127 non-negative finite magnitudes: the candidate just below and
    just above |t| are compared and the closer one is taken; on an exact tie the code with a
    zero mantissa LSB (the even code) wins.  The sign bit follows the sign of t, so negative
    values that round to zero give 0x80 (IEEE-style signed zero).
    """
    t = np.asarray(t, dtype=np.float64)
    a = np.minimum(np.abs(t), 448.0)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_hi = np.abs(_E4M3_POS[hi] - a)
    d_lo = np.abs(a - _E4M3_POS[lo])
    pick = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    pick = np.where(tie, np.where(lo % 2 == 0, lo, hi), pick)
    sign = np.signbit(t).astype(np.uint8) << np.uint8(7)
    return (pick.astype(np.uint8) | sign).astype(np.uint8)


# ----------------------------------------------------------------------------------------
# FP4 E2M1 (the MXFP4 element): 1 sign, 2 exponent (bias 1), 1 mantissa bit.  Values
# {0, 0.5, 1, 1.5, 2, 3, 4, 6} and their negatives.  [DSV4] §9.3 names MXFP4 experts but
# gives no bit layout; this is the OCP microscaling definition.
# ----------------------------------------------------------------------------------------


def e2m1_value(code: int) -> float:
    s = (code >> 3) & 1
    e = (code >> 1) & 0x3
    m = code & 0x1
    mag = m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def unpack_e2m1(packed) -> np.ndarray:
    """Packed FP4 bytes [..., K/2] -> codes [..., K]; element 2i is the LOW nibble of byte i."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def e2m1_decode(codes) -> np.ndarray:
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8)]


# ----------------------------------------------------------------------------------------
# UE8M0 scale byte: an unsigned power-of-two exponent, value 2^(b - 127); 255 is NaN.
# [DSV4], "KV cache layout root cause": scale = exp2(byte - 127), 118 -> 2^-9, 119 -> 2^-8.
# ----------------------------------------------------------------------------------------


def ue8m0_decode(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.int64)
    v = np.ldexp(1.0, b - 127)
    return np.where(b == 255, np.nan, v)
