"""Pins for the INT8 W8A8, FP8 block and 1x128 quantisation parts of the oracle:
hand-worked values, exact rational brute force, special cases and invariants.  CPU only."""
import os
from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import formats as F
from oracle import qlinear_oracle as Q


def _parse_golden(path):
    d = {}
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        k, v = line.split(":")
        d[k.strip()] = [float(t) for t in v.split()]
    return d


def _bits(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, np.float32))


# --------------------------------------------------------------------------------- INT8
def test_int8_hand_worked(golden_dir):
    g = _parse_golden(os.path.join(golden_dir, "int8_w8a8_hand_3x8.txt"))
    x = _bits([g[f"x {i}"] for i in range(3)])
    w = np.array([g["w 0"], g["w 1"]], dtype=np.int8)
    ws = np.array(g["w_s"], np.float32)
    r = Q.int8_w8a8(x, w, ws)
    assert r["x_s"].tolist() == g["x_s"]
    for i in range(3):
        assert r["x_q"][i].tolist() == g[f"x_q {i}"]
        assert r["acc"][i].tolist() == g[f"acc {i}"]
        assert F.bf16_to_f64(r["y"][i]).tolist() == g[f"y {i}"]


def test_int8_brute_force_python_ints():
    c = synth.int8_case(3, 5, 96, seed=7)
    r = Q.int8_w8a8(c["x"], c["w"], c["w_s"])
    xf = F.bf16_to_f32(c["x"])
    for m in range(3):
        amax = max(abs(float(v)) for v in xf[m])
        xs = np.float32(np.float32(amax) / np.float32(127))
        assert r["x_s"][m] == xs
        for n in range(5):
            acc = sum(int(r["x_q"][m, k]) * int(c["w"][n, k]) for k in range(96))
            assert r["acc"][m, n] == acc
            exact = Fraction(acc) * Fraction(float(xs)) * Fraction(float(c["w_s"][n]))
            assert F.round_to_bf16(float(exact)) == r["y"][m, n]


def test_int8_quant_ties_and_extremes():
    # amax 127 gives x_s exactly 1, so x/x_s = x and ties are visible
    x = _bits([[127, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, -127]])
    q, s = Q.quant_int8_per_token(x)
    assert s[0] == 1.0
    assert q[0].tolist() == [127, 0, 2, 2, 0, -2, -2, -127]
    q0, s0 = Q.quant_int8_per_token(np.zeros((1, 16), np.uint16))
    assert s0[0] == 0 and not q0.any()


def test_int8_bias_after_cast():
    x = _bits([[127, 0, 0, 0]])
    w = np.array([[1, 0, 0, 0]], np.int8)
    r = Q.int8_w8a8(x, w, np.array([1.0], np.float32), bias_bits=_bits([1.0]))
    assert F.bf16_to_f64(r["y"]).tolist() == [[128.0]]


# ----------------------------------------------------------------------------- FP8 block
def _exact_fp8_block(xv, wc, sb, K, bn, bk, a_s=None):
    M, N = xv.shape[0], wc.shape[0]
    y = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for kb in range(-(-K // bk)):
                part = sum(Fraction(float(xv[m, k])) * Fraction(float(F.e4m3_decode(wc[n, k])))
                           for k in range(kb * bk, min(K, (kb + 1) * bk)))
                sc = Fraction(2) ** (int(sb[n // bn, kb]) - 127)
                if a_s is not None:
                    sc *= Fraction(float(a_s[m, kb]))
                tot += part * sc
            y[m][n] = tot
    return y


def test_fp8_block_exact_rational_with_ragged_tail():
    # N and K not multiples of the 32x64 block: ceil-div indexing of the scale grid
    c = synth.fp8_block_case(2, 37, 150, seed=3, ldw=160, block_n=32, block_k=64)
    xv = F.bf16_to_f64(c["x"])
    y, _ = Q.fp8_block(xv, c["w"], c["s"], 150, 32, 64)
    ex = _exact_fp8_block(xv, c["w"], c["s"], 150, 32, 64)
    for m in range(2):
        for n in range(37):
            assert abs(y[m, n] - float(ex[m][n])) <= 1e-12 * (abs(float(ex[m][n])) + 1e-30)


def test_fp8_block_unit_scales_is_dequant_matmul():
    c = synth.fp8_block_case(3, 256, 384, seed=4)
    s1 = np.full_like(c["s"], 127)
    xv = F.bf16_to_f64(c["x"])
    y, _ = Q.fp8_block(xv, c["w"], s1, 384)
    ref = xv @ F.e4m3_decode(c["w"]).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_fp8_block_scale_grid_orientation():
    """One scale block raised by 2^3 must scale exactly the (n-block 1, k-block 0) share of
    the outputs n in [128, 256): a transposed scale index fails this."""
    c = synth.fp8_block_case(2, 256, 384, seed=5)
    s = np.full((2, 3), 127, np.uint8)
    xv = F.bf16_to_f64(c["x"])
    base, _ = Q.fp8_block(xv, c["w"], s, 384)
    s2 = s.copy()
    s2[1, 0] = 130
    y, _ = Q.fp8_block(xv, c["w"], s2, 384)
    wv = F.e4m3_decode(c["w"])
    blk = xv[:, :128] @ wv[128:, :128].T
    assert np.allclose(y[:, :128], base[:, :128], rtol=1e-13)
    assert np.allclose(y[:, 128:], base[:, 128:] + 7 * blk, rtol=1e-12, atol=1e-12)


def test_fp8_block_scale_fold_identity():
    # sum_t sum_kb p[t,kb] s[kb] == sum_kb s[kb] sum_t p[t,kb]   (Z100 record, §二.2.4)
    g = np.random.default_rng(0)
    p = g.standard_normal((64, 40))
    s = 2.0 ** g.integers(-9, -4, 40)
    assert np.isclose((p * s).sum(), (s * p.sum(axis=0)).sum(), rtol=1e-13)


def test_fp8_block_ignores_row_padding():
    c = synth.fp8_block_case(1, 8, 128, seed=6, ldw=256)   # padding holds NaN codes
    y, _ = Q.fp8_block(F.bf16_to_f64(c["x"]), c["w"], c["s"], 128)
    assert np.all(np.isfinite(y))


# ---------------------------------------------------------------- 1x128 E4M3 activations
def test_ue8m0_exponent_hand_values():
    e = Q.ue8m0_exponent_for(np.array([448.0, 449.0, 224.0, 224.5, 1.0, 0.0, 2.0 ** -140]))
    assert e.tolist() == [0, 1, -1, 0, -8, 0, -127]


def test_quant_e4m3_1x128_invariants():
    c = synth.fp8_block_case(4, 1, 1000, seed=8)
    q, s = Q.quant_e4m3_1x128(c["x"])
    x = F.bf16_to_f64(c["x"])
    qv = F.e4m3_decode(q)
    assert np.all(np.abs(qv) <= 448)
    for g in range(s.shape[1]):
        ks = slice(g * 128, min(1000, (g + 1) * 128))
        amax = np.abs(x[:, ks]).max(axis=1)
        sc = F.ue8m0_decode(s[:, g])
        r = amax / sc
        assert np.all((r > 224) & (r <= 448))
        # nearest-code property: error at most half the E4M3 spacing at that magnitude
        t = x[:, ks] / sc[:, None]
        err = np.abs(qv[:, ks] - t)
        a = np.abs(t)
        spacing = np.where(a < 2 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(a, 2 ** -6))) - 3))
        assert np.all(err <= spacing / 2 + 1e-300)


def test_quant_e4m3_all_zero_group():
    q, s = Q.quant_e4m3_1x128(np.zeros((1, 256), np.uint16))
    assert s.tolist() == [[127, 127]] and not q.any()


def test_planted_transposed_scale_index_is_caught(monkeypatch):
    """Negative control: an oracle that indexes the block scales as [kb, n//bn] must fail
    the grid-orientation pin."""
    orig = Q.fp8_block

    def transposed(x, w, s, K, bn=128, bk=128, a_scale=None, rows=None):
        st = np.asarray(s).T.copy()
        st = np.resize(st, np.asarray(s).shape)
        return orig(x, w, st, K, bn, bk, a_scale, rows)

    monkeypatch.setattr(Q, "fp8_block", transposed)
    with pytest.raises(AssertionError):
        test_fp8_block_scale_grid_orientation()


# ------------------------------------------------------------------ BF16 dense GEMV
def test_bf16_linear_exact_rational():
    # every bf16 value is a dyadic rational: the oracle's fp64 sums of these small cases are
    # exact, so they must equal the Fraction dot products
    c = synth.bf16_dense_case(3, 5, 24, seed=3)
    y, a = Q.bf16_linear(c["x"], c["w"], 24)
    xv = F.bf16_to_f64(c["x"])
    wv = F.bf16_to_f64(c["w"][:, :24])
    for m in range(3):
        for n in range(5):
            ref = sum(Fraction(float(xv[m, k])) * Fraction(float(wv[n, k])) for k in range(24))
            aref = sum(abs(Fraction(float(xv[m, k])) * Fraction(float(wv[n, k]))) for k in range(24))
            assert Fraction(float(y[m, n])) == ref
            assert Fraction(float(a[m, n])) == aref


def test_bf16_linear_identity_and_padding():
    # W = I picks the activations; NaN padding past K is never read
    K = 16
    x = synth.bf16_dense_case(2, 1, K, seed=4)["x"]
    w = np.full((K, K + 8), 0x7FC0, np.uint16)
    w[:, :K] = 0
    w[np.arange(K), np.arange(K)] = 0x3F80  # bf16 1.0
    y, a = Q.bf16_linear(x, w, K)
    assert np.array_equal(y, F.bf16_to_f64(x))
    assert np.array_equal(a, np.abs(F.bf16_to_f64(x)))


def test_bf16_linear_row_subset_and_transpose():
    # rows= selects output columns; a wrong operand orientation would break the shape or values
    c = synth.bf16_dense_case(2, 7, 32, seed=5)
    y, _ = Q.bf16_linear(c["x"], c["w"], 32)
    ys, _ = Q.bf16_linear(c["x"], c["w"], 32, rows=[6, 1])
    assert y.shape == (2, 7) and np.array_equal(ys, y[:, [6, 1]])
    # a planted mistake (w used without the transpose on a square case) must not agree
    sq = synth.bf16_dense_case(3, 3, 3, seed=6)
    yy, _ = Q.bf16_linear(sq["x"], sq["w"], 3)
    wrong = F.bf16_to_f64(sq["x"]) @ F.bf16_to_f64(sq["w"])
    assert not np.allclose(yy, wrong)


# ------------------------------------------------------------------ FP8 per-tensor / per-channel
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_channel_rational_brute_force(fmt):
    # exact rational dot products; the oracle's fp64 evaluation may round only within the
    # fp64 summation bound (E5M2's 31-binade range can exceed 53 bits in a 16-term sum)
    c = synth.fp8_channel_case(2, 4, 16, seed=11, w_fmt=fmt)
    y, a = Q.fp8_channel(c["x"], c["w"], fmt, c["w_s"], 16)
    dec = F.e4m3_decode if fmt == "e4m3" else F.e5m2_decode
    xv, wv = F.bf16_to_f64(c["x"]), dec(c["w"][:, :16])
    for m in range(2):
        for n in range(4):
            s = Fraction(float(c["w_s"][n]))
            terms = [Fraction(float(xv[m, k])) * Fraction(float(wv[n, k])) for k in range(16)]
            ref = s * sum(terms)
            bound = 18 * Fraction(2) ** -53 * abs(s) * sum(abs(t) for t in terms)
            assert abs(Fraction(float(y[m, n])) - ref) <= bound
            assert abs(Fraction(float(a[m, n])) - abs(s) * sum(abs(t) for t in terms)) <= bound


def test_fp8_channel_per_tensor_is_uniform_per_channel():
    c = synth.fp8_channel_case(3, 6, 40, seed=12, per_channel=False)
    y1, a1 = Q.fp8_channel(c["x"], c["w"], "e4m3", c["w_s"], 40)
    y2, a2 = Q.fp8_channel(c["x"], c["w"], "e4m3", np.full(6, c["w_s"][0], np.float32), 40)
    assert np.array_equal(y1, y2) and np.array_equal(a1, a2)


def test_fp8_channel_unit_scale_is_block_path_with_unit_blocks():
    # with every scale 1 the per-channel formula equals the 128x128 block formula at scale 2^0
    c = synth.fp8_channel_case(2, 130, 300, seed=13)
    y, _ = Q.fp8_channel(c["x"], c["w"], "e4m3", np.ones(130, np.float32), 300)
    sb = np.full((2, 3), 127, np.uint8)
    yb, _ = Q.fp8_block(F.bf16_to_f64(c["x"]), c["w"], sb, 300)
    assert np.allclose(y, yb, rtol=1e-13, atol=0)


def test_fp8_channel_scale_index_and_padding():
    # a scale on one channel changes only that output column; padding past K is never read
    c = synth.fp8_channel_case(2, 5, 24, seed=14, ldw=40, w_fmt="e5m2")
    ws = np.ones(5, np.float32)
    y0, _ = Q.fp8_channel(c["x"], c["w"], "e5m2", ws, 24)
    ws[3] = 4.0
    y1, _ = Q.fp8_channel(c["x"], c["w"], "e5m2", ws, 24)
    assert np.array_equal(y1[:, [0, 1, 2, 4]], y0[:, [0, 1, 2, 4]])
    assert np.array_equal(y1[:, 3], 4.0 * y0[:, 3])
    assert np.all(np.isfinite(y0))
