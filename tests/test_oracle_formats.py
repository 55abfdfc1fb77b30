"""Pins for the oracle's number formats: exhaustive decodes against closed forms and an
independent library, the pages' worked UE8M0 example, and rounding against reference
conversions.  CPU only."""
import math
import os

import numpy as np
import pytest

from oracle import formats as F


def _ref_e4m3(code):
    # closed form written independently of the oracle: value = sign * 2^E * mantissa
    sign = -1.0 if code & 0x80 else 1.0
    mag = code & 0x7F
    if mag == 0x7F:
        return math.nan
    e, m = mag >> 3, mag & 7
    return sign * (math.ldexp(m, -9) if e == 0 else math.ldexp(8 + m, e - 10))


def test_e4m3_exhaustive_closed_form():
    for c in range(256):
        want, got = _ref_e4m3(c), F.e4m3_decode(np.uint8(c))
        if math.isnan(want):
            assert np.isnan(got), c
        else:
            assert got == want, (c, got, want)
    fin = F.E4M3_TABLE[np.isfinite(F.E4M3_TABLE)]
    assert fin.size == 254
    assert fin.max() == 448.0 and fin.min() == -448.0
    assert F.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9      # smallest subnormal
    assert F.e4m3_decode(np.uint8(0x08)) == 2.0 ** -6      # smallest normal
    assert F.e4m3_decode(np.uint8(0x38)) == 1.0


def test_e4m3_exhaustive_vs_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    codes = np.arange(256, dtype=np.uint8)
    lib = codes.view(ml.float8_e4m3fn).astype(np.float64)
    ours = F.e4m3_decode(codes)
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], ours[ok])


def _ref_e5m2(code):
    # closed form written independently: E5M2 is the top byte of an IEEE binary16
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 2) & 0x1F, code & 3
    if e == 31:
        return sign * math.inf if m == 0 else math.nan
    return sign * (math.ldexp(m, -16) if e == 0 else math.ldexp(4 + m, e - 17))


def test_e5m2_exhaustive_closed_form():
    for c in range(256):
        want, got = _ref_e5m2(c), F.e5m2_decode(np.uint8(c))
        if math.isnan(want):
            assert np.isnan(got), c
        else:
            assert got == want, (c, got, want)
    fin = F.E5M2_TABLE[np.isfinite(F.E5M2_TABLE)]
    assert fin.size == 248 and fin.max() == 57344.0
    assert F.e5m2_decode(np.uint8(0x01)) == 2.0 ** -16     # smallest subnormal
    assert F.e5m2_decode(np.uint8(0x3C)) == 1.0


def test_e5m2_is_the_high_byte_of_float16():
    # an independent library route: code c is the binary16 with bits c << 8
    codes = np.arange(256, dtype=np.uint16)
    lib = (codes << 8).astype(np.uint16).view(np.float16).astype(np.float64)
    ours = F.e5m2_decode(codes.astype(np.uint8))
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], ours[ok])


def test_e5m2_vs_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e5m2"):
        pytest.skip("torch without float8_e5m2")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e5m2).to(torch.float64).numpy()
    ours = F.e5m2_decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], ours[ok])


def test_e2m1_exhaustive():
    want = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(F.E2M1_TABLE[:8]) == want
    assert list(F.E2M1_TABLE[8:]) == [-v for v in want]


def test_e2m1_vs_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    if not hasattr(ml, "float4_e2m1fn"):
        pytest.skip("ml_dtypes without float4_e2m1fn")
    vals = np.array(F.E2M1_TABLE, dtype=np.float32)
    back = vals.astype(ml.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(back, F.E2M1_TABLE)


def test_unpack_e2m1_low_nibble_first():
    b = np.array([[0x21, 0xF0]], dtype=np.uint8)
    assert F.unpack_e2m1(b).tolist() == [[1, 2, 0, 15]]


def test_ue8m0_worked_example(golden_dir):
    rows = [l.split() for l in open(os.path.join(golden_dir, "ue8m0_kv_scale_example.txt"))
            if l.strip() and not l.startswith("#")]
    for byte, ex, val in rows:
        got = F.ue8m0_decode(int(byte))
        assert got == 2.0 ** int(ex) == float(val)


def test_ue8m0_exhaustive():
    for b in range(255):
        assert F.ue8m0_decode(b) == math.ldexp(1.0, b - 127)
    assert np.isnan(F.ue8m0_decode(255))


def test_bf16_round_vs_torch():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(1)
    v = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(1000),
        (g.standard_normal(2000) * 1e-39).astype(np.float32),          # bf16 subnormals
        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.3e38, -3.3e38], np.float32),
    ])
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = F.round_to_bf16(v.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_round_ties_even_exact_f64():
    # 1 + 2^-8 is exactly halfway between 1 and 1 + 2^-7: ties to the even significand (1.0)
    assert F.round_to_bf16(1.0 + 2 ** -8) == 0x3F80
    assert F.round_to_bf16(1.0 + 2 ** -8 + 2 ** -40) == 0x3F81   # just above the tie
    assert F.round_to_bf16(-(1.0 + 3 * 2 ** -8)) == 0xBF82
    assert F.round_to_bf16(2.0 ** 128) == 0x7F80


def test_e4m3_encode_roundtrip_and_ties():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = F.e4m3_decode(codes)
    back = F.e4m3_encode_rne_sat(vals)
    # +0 and -0 are distinct codes and both survive
    assert np.array_equal(back, codes)
    # tie between 1.0 (0x38, even) and 1.125 (0x39): goes to 1.0; 1.1875 -> 1.25 (0x3A)
    assert F.e4m3_encode_rne_sat(1.0625) == 0x38
    assert F.e4m3_encode_rne_sat(1.1875) == 0x3A
    assert F.e4m3_encode_rne_sat(-1e-9) == 0x80
    assert F.e4m3_encode_rne_sat(1000.0) == 0x7E


def test_e4m3_encode_vs_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8")
    g = np.random.default_rng(2)
    v = np.concatenate([g.uniform(-448, 448, 20000), g.standard_normal(20000) * 2 ** -7,
                        F.E4M3_TABLE[:0x7F] + 2 ** -12]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.e4m3_encode_rne_sat(v.astype(np.float64))
    assert np.array_equal(got, want)


def test_planted_mistake_caught_by_exhaustive_decode(monkeypatch):
    """Negative control: a subnormal decoded with the normal formula (the shift-and-rebias
    mistake the Z100 record warns about) must fail the closed-form check."""
    bad = F.E4M3_TABLE.copy()
    bad[0x03] = (1 + 3 / 8) * 2.0 ** -7
    monkeypatch.setattr(F, "E4M3_TABLE", bad)
    with pytest.raises(AssertionError):
        test_e4m3_exhaustive_closed_form()
