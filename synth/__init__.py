"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module only draws random numbers with the shapes and distributions of the decode
workloads; it holds none of the layer's arithmetic (no quantisation, decoding or
contraction).  Random streams come from numpy's counter-based Philox generator keyed by
(seed, stream id), so every tensor of a case is reproducible on its own.
"""
from __future__ import annotations

import numpy as np

# stream ids: one independent Philox key per tensor role
_X, _W, _WS, _BIAS, _LOGITS, _W13, _S13, _W2, _S2, _IDS = range(10)


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=(int(seed) << 16) | int(stream)))


def f32_to_bf16_bits(v) -> np.ndarray:
    """Round fp32 samples to bf16 bit patterns (nearest, ties to even) for finite inputs.
    In uint32: the largest finite pattern plus 0x8000 stays below 2^32."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF)
    r += (u >> np.uint32(16)) & np.uint32(1)
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_normal(g: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(g.standard_normal(size=shape, dtype=np.float32))


def random_bytes(g: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return np.frombuffer(g.bytes(n), dtype=np.uint8).reshape(shape).copy()


# the 254 finite E4M3 codes (0x7F and 0xFF are NaN)
_E4M3_FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def e4m3_finite_codes(g: np.random.Generator, shape) -> np.ndarray:
    return _E4M3_FINITE[g.integers(0, _E4M3_FINITE.size, size=shape)]


def ue8m0_uniform(g: np.random.Generator, shape, lo: int, hi: int) -> np.ndarray:
    return g.integers(lo, hi + 1, size=shape).astype(np.uint8)


# ---------------------------------------------------------------- INT8 W8A8 cases
def int8_case(M, N, K, seed=0, ldw=None):
    """INT8 W8A8: w ~ U{-127..127} int8 [N, ldw], per-channel w_s ~ U[0.001, 0.01] fp32,
    x ~ N(0,1) rounded to bf16 [M, K]."""
    ldw = K if ldw is None else ldw
    w = rng(seed, _W).integers(-127, 128, size=(N, ldw), dtype=np.int64).astype(np.int8)
    ws = rng(seed, _WS).uniform(0.001, 0.01, size=N).astype(np.float32)
    x = bf16_normal(rng(seed, _X), (M, K))
    return {"x": x, "w": w, "w_s": ws}


# ---------------------------------------------------------------- FP8 block cases
def fp8_block_case(M, N, K, seed=0, ldw=None, block_n=128, block_k=128, s_lo=118, s_hi=122):
    """FP8 E4M3 weights uniform over the finite codes [N, ldw] (padding columns hold 0xFF,
    a NaN code, so a kernel that reads past K shows it), UE8M0 block scales uniform in
    [s_lo, s_hi] of shape [ceil(N/block_n), ceil(K/block_k)], x ~ N(0,1) bf16 [M, K]."""
    ldw = K if ldw is None else ldw
    w = np.full((N, ldw), 0xFF, dtype=np.uint8)
    w[:, :K] = e4m3_finite_codes(rng(seed, _W), (N, K))
    s = ue8m0_uniform(rng(seed, _WS), (-(-N // block_n), -(-K // block_k)), s_lo, s_hi)
    x = bf16_normal(rng(seed, _X), (M, K))
    return {"x": x, "w": w, "s": s}


# ---------------------------------------------------------------- MXFP4 cases
# the 248 finite E5M2 codes (exponent 31 is infinity or NaN)
_E5M2_FINITE = np.array([c for c in range(256) if ((c >> 2) & 0x1F) != 0x1F], dtype=np.uint8)


def fp8_channel_case(M, N, K, seed=0, ldw=None, w_fmt="e4m3", per_channel=True):
    """FP8 weights with fp32 scales: codes uniform over the finite codes of the format [N, ldw]
    (padding columns hold 0xFF, a NaN code in both formats), scales ~ U[2^-10, 2^-6] per channel
    (or one per tensor), x ~ N(0,1) bf16 [M, K]."""
    ldw = K if ldw is None else ldw
    w = np.full((N, ldw), 0xFF, dtype=np.uint8)
    table = _E4M3_FINITE if w_fmt == "e4m3" else _E5M2_FINITE
    w[:, :K] = table[rng(seed, _W).integers(0, table.size, size=(N, K))]
    ws = rng(seed, _WS).uniform(2.0 ** -10, 2.0 ** -6, size=N if per_channel else 1).astype(np.float32)
    x = bf16_normal(rng(seed, _X), (M, K))
    return {"x": x, "w": w, "w_s": ws}


def bf16_dense_case(M, N, K, seed=0, ldw=None):
    """BF16 dense weights: w ~ N(0, 0.05^2) bf16 [N, ldw] (padding columns hold a NaN, so a
    kernel that reads past K shows it), x ~ N(0,1) bf16 [M, K]."""
    ldw = K if ldw is None else ldw
    w = np.full((N, ldw), 0x7FC0, dtype=np.uint16)
    w[:, :K] = f32_to_bf16_bits(0.05 * rng(seed, _W).standard_normal(size=(N, K), dtype=np.float32))
    x = bf16_normal(rng(seed, _X), (M, K))
    return {"x": x, "w": w}


def mxfp4_dense_case(M, N, K, seed=0, s_lo=120, s_hi=127):
    """MXFP4 weights: uniform random E2M1 codes packed two per byte [N, K/2], UE8M0 per 32
    along K uniform in [s_lo, s_hi] [N, K/32]; x ~ N(0,1) bf16 [M, K]."""
    w = random_bytes(rng(seed, _W), (N, K // 2))
    s = ue8m0_uniform(rng(seed, _WS), (N, K // 32), s_lo, s_hi)
    x = bf16_normal(rng(seed, _X), (M, K))
    return {"x": x, "w": w, "s": s}


def moe_case(M, E=256, H=4096, I=2048, seed=0, s_lo=120, s_hi=127):
    """MXFP4 MoE decode: x ~ N(0,1) bf16 [M, H], router logits ~ N(0,1) bf16 [M, E],
    W13 codes [E, 2I, H/2] with UE8M0 [E, 2I, H/32], W2 codes [E, H, I/2] with UE8M0
    [E, H, I/32]; codes uniform, scale exponents uniform in [s_lo, s_hi]."""
    return {
        "x": bf16_normal(rng(seed, _X), (M, H)),
        "logits": bf16_normal(rng(seed, _LOGITS), (M, E)),
        "w13": random_bytes(rng(seed, _W13), (E, 2 * I, H // 2)),
        "s13": ue8m0_uniform(rng(seed, _S13), (E, 2 * I, H // 32), s_lo, s_hi),
        "w2": random_bytes(rng(seed, _W2), (E, H, I // 2)),
        "s2": ue8m0_uniform(rng(seed, _S2), (E, H, I // 32), s_lo, s_hi),
    }


def moe_weights_only(E, H, I, seed=0, s_lo=120, s_hi=127):
    c = moe_case(1, E, H, I, seed, s_lo, s_hi)
    return {k: c[k] for k in ("w13", "s13", "w2", "s2")}


def moe_tokens(M, E, H, seed=0):
    return {"x": bf16_normal(rng(seed, _X), (M, H)),
            "logits": bf16_normal(rng(seed, _LOGITS), (M, E))}
