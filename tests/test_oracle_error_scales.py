"""Pins for the oracle parts that the float parity bar rests on but that no other pin reaches:
the error scales sum_k |w x| (the denominators of the tolerance) of every linear and of both
MoE stages, the block formula with non-unit 1x128 activation scales, the routing weights
against an independent high-precision softmax, and the weighted combine over several experts.

Each pin compares the oracle with exact rational arithmetic (Fraction) or with mpmath at 40
digits on tiny inputs, i.e. with the definition evaluated a different way, and each has a
negative control: the same check applied to a plausible mistake (a signed sum for an absolute
one, one activation scale for every K group, renormalised weights, swapped combine weights)
must fail.  CPU only."""
from fractions import Fraction

import mpmath
import numpy as np
import pytest

import synth
from oracle import formats as F
from oracle import qlinear_oracle as Q


def _fr(v):
    return Fraction(float(v))


def _e4m3(code):
    return _fr(F.e4m3_decode(np.uint8(code)))


def _p2(e):
    return Fraction(2) ** int(e)


def _mx(packed, scales, r, k):
    """Exact MXFP4 weight: E2M1 code (low nibble = even k) times 2^(s - 127)."""
    byte = int(packed[r, k // 2])
    code = (byte & 0xF) if k % 2 == 0 else (byte >> 4)
    return _fr(F.E2M1_TABLE[code]) * _p2(int(scales[r, k // 32]) - 127)


def _close(got, exact, rel=1e-13):
    """got (fp64) within rel of the exact rational (and exactly 0 when it is 0)."""
    ex = float(exact)
    assert abs(float(got) - ex) <= rel * abs(ex) + 1e-300, (float(got), ex)


def _check_matrix(got, exact, rel=1e-13):
    got = np.asarray(got)
    for idx in np.ndindex(got.shape):
        _close(got[idx], exact[idx[0]][idx[1]], rel)


# ------------------------------------------------------------------------------ INT8
def _int8_abs_exact(r, w, w_s):
    M, N = r["acc"].shape
    ws = np.asarray(w_s, np.float32).reshape(-1)
    return [[sum(abs(int(r["x_q"][m, k]) * int(w[n, k])) for k in range(w.shape[1]))
             * _fr(r["x_s"][m]) * _fr(ws[n] if ws.size > 1 else ws[0]) for n in range(N)] for m in range(M)]


def test_int8_abs_sum_exact():
    """abs_sum[m,n] = x_s[m] w_s[n] sum_k |x_q[m,k] w[n,k]|, per channel and per tensor."""
    c = synth.int8_case(3, 6, 80, seed=21)
    r = Q.int8_w8a8(c["x"], c["w"], c["w_s"])
    _check_matrix(r["abs_sum"], _int8_abs_exact(r, c["w"], c["w_s"]))
    r1 = Q.int8_w8a8(c["x"], c["w"], c["w_s"][:1])
    _check_matrix(r1["abs_sum"], _int8_abs_exact(r1, c["w"], c["w_s"][:1]))


def test_int8_abs_sum_negative_control():
    c = synth.int8_case(2, 4, 64, seed=22)
    r = Q.int8_w8a8(c["x"], c["w"], c["w_s"])
    signed = np.abs(r["acc"].astype(np.float64)) * r["x_s"][:, None].astype(np.float64) \
        * c["w_s"][None, :].astype(np.float64)            # |sum| instead of sum |.|
    with pytest.raises(AssertionError):
        _check_matrix(signed, _int8_abs_exact(r, c["w"], c["w_s"]))


# ------------------------------------------------------------------------------ FP8 block
def _fp8_exact(xv, wc, sb, K, bn, bk, a_s=None):
    """(y, abs_sum) of the block formula as Fractions; a_s: fp64 [M, nkb] activation scales."""
    M, N = xv.shape[0], wc.shape[0]
    y = [[Fraction(0)] * N for _ in range(M)]
    a = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            for kb in range(-(-K // bk)):
                ks = range(kb * bk, min(K, (kb + 1) * bk))
                terms = [_fr(xv[m, k]) * _e4m3(wc[n, k]) for k in ks]
                sc = _p2(int(sb[n // bn, kb]) - 127) * (1 if a_s is None else _fr(a_s[m, kb]))
                y[m][n] += sum(terms) * sc
                a[m][n] += sum(abs(t) for t in terms) * abs(sc)
    return y, a


def test_fp8_block_abs_sum_exact_ragged():
    c = synth.fp8_block_case(2, 37, 150, seed=23, ldw=160, block_n=32, block_k=64)
    xv = F.bf16_to_f64(c["x"])
    y, a = Q.fp8_block(xv, c["w"], c["s"], 150, 32, 64)
    ye, ae = _fp8_exact(xv, c["w"], c["s"], 150, 32, 64)
    _check_matrix(y, ye, 1e-12)
    _check_matrix(a, ae)


def _act_quant_case():
    """x with a different 1x128 scale in each K group (group 1 is 2^5 larger) and a ragged
    last group (K = 200: groups [0,128) and [128,200))."""
    c = synth.fp8_block_case(2, 37, 200, seed=24, ldw=208, block_n=32, block_k=128)
    x = F.bf16_to_f32(c["x"]).copy()
    x[:, 128:] *= 32.0
    c["x"] = synth.f32_to_bf16_bits(x)
    return c


def _act_quant_exact(c):
    q, s = Q.quant_e4m3_1x128(c["x"])           # the quantisation has its own pins
    qv = F.e4m3_decode(q)
    a_s = F.ue8m0_decode(s)
    return _fp8_exact(qv, c["w"], c["s"], 200, 32, 128, a_s=a_s), s


def test_fp8_block_act_quant_exact_with_group_scales():
    """The 1x128-activation FP8 linear (the tcgen05 path's definition): a_s[m, kb] scales
    exactly the K group kb of token m, in y and in abs_sum."""
    c = _act_quant_case()
    r = Q.fp8_block_act_quant(c["x"], c["w"], c["s"], 200, 32, 128)
    (ye, ae), s = _act_quant_exact(c)
    assert len(set(s[0].tolist())) == 2          # two different activation scales per token
    _check_matrix(r["y_f64"], ye, 1e-12)
    _check_matrix(r["abs_sum"], ae)


def test_fp8_block_act_quant_negative_control(monkeypatch):
    """An oracle applying the first group's activation scale to every K group must fail."""
    orig = Q.fp8_block

    def first_group_only(x, w, s, K, bn=128, bk=128, a_scale=None, rows=None):
        if a_scale is not None:
            a_scale = np.repeat(np.asarray(a_scale)[:, :1], np.asarray(a_scale).shape[1], axis=1)
        return orig(x, w, s, K, bn, bk, a_scale, rows)

    monkeypatch.setattr(Q, "fp8_block", first_group_only)
    with pytest.raises(AssertionError):
        test_fp8_block_act_quant_exact_with_group_scales()


# ------------------------------------------------------------------------------ FP8 per channel / BF16
def test_fp8_channel_and_bf16_abs_sum_signs():
    """abs_sum is unchanged when every activation changes sign, while y changes sign: a
    signed sum in place of the absolute one fails this."""
    c = synth.fp8_channel_case(2, 5, 48, seed=25)
    neg = c["x"] ^ np.uint16(0x8000)
    y, a = Q.fp8_channel(c["x"], c["w"], "e4m3", c["w_s"], 48)
    yn, an = Q.fp8_channel(neg, c["w"], "e4m3", c["w_s"], 48)
    assert np.array_equal(a, an) and np.array_equal(y, -yn) and np.all(a >= np.abs(y))
    b = synth.bf16_dense_case(2, 5, 48, seed=26)
    y, a = Q.bf16_linear(b["x"], b["w"], 48)
    yn, an = Q.bf16_linear(b["x"] ^ np.uint16(0x8000), b["w"], 48)
    assert np.array_equal(a, an) and np.array_equal(y, -yn) and np.all(a >= np.abs(y))


# ------------------------------------------------------------------------------ MXFP4, 1x128 activations
def test_mxfp4_act_quant_abs_sum_exact():
    c = synth.mxfp4_dense_case(2, 3, 256, seed=27)
    r = Q.mxfp4_act_quant(c["x"], c["w"], c["s"])
    for m in range(2):
        for n in range(3):
            tot = Fraction(0)
            for k in range(256):
                av = _e4m3(r["q"][m, k]) * _p2(int(r["s"][m, k // 128]) - 127)
                tot += abs(av * _mx(c["w"], c["s"], n, k))
            _close(r["abs_sum"][m, n], tot)


# ------------------------------------------------------------------------------ MoE error scales
def _gate_up_exact(x, w13, s13, e, I, i):
    """(g, u, G, U) of intermediate i of expert e for activations x (exact rationals)."""
    g = sum(_mx(w13[e], s13[e], i, k) * _fr(x[k]) for k in range(len(x)))
    u = sum(_mx(w13[e], s13[e], I + i, k) * _fr(x[k]) for k in range(len(x)))
    G = sum(abs(_mx(w13[e], s13[e], i, k) * _fr(x[k])) for k in range(len(x)))
    U = sum(abs(_mx(w13[e], s13[e], I + i, k) * _fr(x[k])) for k in range(len(x)))
    return g, u, G, U


@pytest.mark.parametrize("act_quant", [False, True])
def test_moe_gate_up_error_scales_exact(act_quant):
    """G = sum_k |W13[e][i,k] a_k| and U = sum_k |W13[e][I+i,k] a_k| per pair, with a = x (bf16
    path) or the 1x128 E4M3 dequantised x (grouped path)."""
    M, E, H, I, topk = 2, 3, 128, 32, 2
    c = synth.moe_case(M, E=E, H=H, I=I, seed=28)
    ids = np.array([[2, 0], [1, 2]], np.int32)
    cols = np.array([0, 5, 31])
    if act_quant:
        st = Q.moe_gate_up_act_quant(c["x"], ids, c["w13"], c["s13"], I, cols=cols)
        xa = F.e4m3_decode(st["q"]) * np.repeat(F.ue8m0_decode(st["s"]), 128, axis=1)[:, :H]
    else:
        st = Q.moe_gate_up(c["x"], ids, c["w13"], c["s13"], I, cols=cols)
        xa = F.bf16_to_f64(c["x"])
    for p in range(M * topk):
        m, j = divmod(p, topk)
        for ci, i in enumerate(cols):
            g, u, G, U = _gate_up_exact(xa[m], c["w13"], c["s13"], int(ids[m, j]), I, int(i))
            _close(st["g"][p, ci], g, 1e-12)
            _close(st["u"][p, ci], u, 1e-12)
            _close(st["G"][p, ci], G)
            _close(st["U"][p, ci], U)


def test_moe_gate_up_error_scales_negative_control():
    """G with the gate and up rows exchanged (U in place of G) fails the same check."""
    c = synth.moe_case(1, E=1, H=64, I=32, seed=29)
    ids = np.zeros((1, 1), np.int32)
    st = Q.moe_gate_up(c["x"], ids, c["w13"], c["s13"], 32, cols=np.array([3]))
    _, _, G, U = _gate_up_exact(F.bf16_to_f64(c["x"])[0], c["w13"], c["s13"], 0, 32, 3)
    assert G != U
    with pytest.raises(AssertionError):
        _close(st["U"][0, 0], G)


# ------------------------------------------------------------------------------ MoE combine, top-k > 1
def _combine_exact(hv, ids, wts, w2, s2, rows):
    """y[m][n] and abs_sum[m][n] of sum_j w_(m,j) W2[e_(m,j)] h_(m,j), as Fractions; hv: fp64
    activations per pair [M*topk, I]."""
    M, topk = ids.shape
    I = hv.shape[1]
    y = [[Fraction(0)] * len(rows) for _ in range(M)]
    a = [[Fraction(0)] * len(rows) for _ in range(M)]
    for m in range(M):
        for j in range(topk):
            e, wj = int(ids[m, j]), _fr(wts[m, j])
            for ni, n in enumerate(rows):
                terms = [_mx(w2[e], s2[e], n, i) * _fr(hv[m * topk + j, i]) for i in range(I)]
                y[m][ni] += wj * sum(terms)
                a[m][ni] += abs(wj) * sum(abs(t) for t in terms)
    return y, a


def _combine_case():
    M, E, H, I, topk = 2, 3, 64, 128, 3
    c = synth.moe_case(M, E=E, H=H, I=I, seed=30)
    ids = np.array([[2, 0, 1], [1, 2, 0]], np.int32)
    wts = np.array([[0.625, 0.25, 0.125], [0.5, 0.375, -0.0625]])  # distinct, dyadic (exact)
    h = synth.bf16_normal(synth.rng(30, 9), (M * topk, I))
    return c, ids, wts, h, [0, 7, 63]


@pytest.mark.parametrize("act_quant", [False, True])
def test_moe_down_combine_topk_exact(act_quant):
    """Stage 2 with three experts per token and unequal weights: y and its error scale equal
    the exact weighted sum over the pairs (h used as bf16 values, or 1x128-quantised)."""
    c, ids, wts, h, rows = _combine_case()
    if act_quant:
        _, y64, ab = Q.moe_down_combine_act_quant(h, ids, wts, c["w2"], c["s2"], rows=rows)
        q, s = Q.quant_e4m3_1x128(h)
        hv = F.e4m3_decode(q) * np.repeat(F.ue8m0_decode(s), 128, axis=1)[:, :h.shape[1]]
    else:
        _, y64, ab = Q.moe_down_combine(h, ids, wts, c["w2"], c["s2"], rows=rows)
        hv = F.bf16_to_f64(h)
    ye, ae = _combine_exact(hv, ids, wts, c["w2"], c["s2"], rows)
    _check_matrix(y64, ye, 1e-12)
    _check_matrix(ab, ae, 1e-12)


def test_moe_down_combine_negative_control():
    """Weights paired with the wrong slot (j -> topk-1-j) fail the exact combine pin."""
    c, ids, wts, h, rows = _combine_case()
    _, y64, _ = Q.moe_down_combine(h, ids, wts[:, ::-1].copy(), c["w2"], c["s2"], rows=rows)
    ye, _ = _combine_exact(F.bf16_to_f64(h), ids, wts, c["w2"], c["s2"], rows)
    with pytest.raises(AssertionError):
        _check_matrix(y64, ye, 1e-12)


# ------------------------------------------------------------------------------ routing weights
mpmath.mp.dps = 40


def _softmax_mp(logits):
    ex = [mpmath.e ** mpmath.mpf(v) for v in logits]
    tot = mpmath.fsum(ex)
    return [e / tot for e in ex]


ROUTE_LOGITS = [2.0, 1.0, 0.0, -1.0, 0.5, -3.0, 1.0, 0.25]   # exact in bf16


def test_routing_weights_vs_high_precision_softmax():
    """Weights = softmax probabilities of the chosen experts, against mpmath at 40 digits:
    p_i = e^(l_i) / sum_j e^(l_j).  Top-4 of the logits above: ids 0, 1, 6 (tie with 1,
    the higher id second), 4."""
    lg = synth.f32_to_bf16_bits(np.array([ROUTE_LOGITS], np.float32))
    ids, w = Q.route_topk(lg, 4)
    assert ids[0].tolist() == [0, 1, 6, 4]
    p = _softmax_mp(ROUTE_LOGITS)
    for j, e in enumerate(ids[0]):
        assert abs(w[0, j] - float(p[e])) <= 4e-16 * float(p[e])
    # hand value of the largest: e^2 / (e^2 + 2e + 1 + e^-1 + e^0.5 + e^-3 + e^0.25)
    hand = mpmath.e ** 2 / (mpmath.e ** 2 + 2 * mpmath.e + 1 + mpmath.e ** -1 + mpmath.e ** 0.5
                            + mpmath.e ** -3 + mpmath.e ** 0.25)
    assert abs(w[0, 0] - float(hand)) <= 4e-16


def test_routing_renormalised_weights_vs_high_precision():
    lg = synth.f32_to_bf16_bits(np.array([ROUTE_LOGITS], np.float32))
    ids, w = Q.route_topk(lg, 3, renormalize=True)
    sel = _softmax_mp([ROUTE_LOGITS[e] for e in ids[0]])
    for j in range(3):
        assert abs(w[0, j] - float(sel[j])) <= 4e-16 * float(sel[j])


def test_routing_weights_negative_control(monkeypatch):
    """An oracle that renormalises when not asked fails the unrenormalised pin."""
    orig = Q.route_topk
    monkeypatch.setattr(Q, "route_topk", lambda lg, k, renormalize=False: orig(lg, k, True))
    with pytest.raises(AssertionError):
        test_routing_weights_vs_high_precision_softmax()
