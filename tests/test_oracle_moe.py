"""Pins for the MXFP4 and MoE parts of the oracle: exact rational brute force, routing
against a library sort, special cases and invariants.  CPU only."""
from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import formats as F
from oracle import qlinear_oracle as Q


def _dequant_exact(packed, scales, r, k):
    byte = int(packed[r, k // 2])
    code = (byte & 0xF) if k % 2 == 0 else (byte >> 4)
    return Fraction(float(F.E2M1_TABLE[code])) * Fraction(2) ** (int(scales[r, k // 32]) - 127)


def test_mxfp4_dequant_exact_brute_force():
    c = synth.mxfp4_dense_case(1, 3, 64, seed=1)
    d = Q.mxfp4_dequant(c["w"], c["s"])
    for r in range(3):
        for k in range(64):
            assert d[r, k] == float(_dequant_exact(c["w"], c["s"], r, k))


def test_mxfp4_dense_act_quant_exact():
    c = synth.mxfp4_dense_case(2, 4, 256, seed=2)
    r = Q.mxfp4_act_quant(c["x"], c["w"], c["s"])
    for m in range(2):
        for n in range(4):
            tot = Fraction(0)
            for k in range(256):
                a = Fraction(float(F.e4m3_decode(r["q"][m, k]))) * Fraction(2) ** (int(r["s"][m, k // 128]) - 127)
                tot += a * _dequant_exact(c["w"], c["s"], n, k)
            assert abs(r["y_f64"][m, n] - float(tot)) <= 1e-12 * abs(float(tot)) + 1e-300


def test_routing_vs_stable_argsort():
    lg = synth.bf16_normal(synth.rng(3, 0), (9, 256))
    ids, w = Q.route_topk(lg, 8)
    v = F.bf16_to_f64(lg)
    for m in range(9):
        want = np.argsort(-v[m], kind="stable")[:8]
        assert ids[m].tolist() == want.tolist()
    p = np.exp(v - v.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    assert np.allclose(w, np.take_along_axis(p, ids.astype(int), 1), rtol=1e-14)


def test_routing_ties_go_to_lower_index():
    lg = synth.f32_to_bf16_bits(np.array([[1.0, 2.0, 2.0, 0.5, 2.0, 1.0]], np.float32))
    ids, w = Q.route_topk(lg, 4)
    assert ids[0].tolist() == [1, 2, 4, 0]
    assert w[0, 0] == w[0, 1] == w[0, 2]


def test_routing_full_topk_weights_sum_to_one():
    lg = synth.bf16_normal(synth.rng(4, 0), (3, 16))
    _, w = Q.route_topk(lg, 16)
    assert np.allclose(w.sum(1), 1.0, rtol=1e-14)
    _, wr = Q.route_topk(lg, 4, renormalize=True)
    assert np.allclose(wr.sum(1), 1.0, rtol=1e-14)


def test_routing_signed_zeros_tie():
    # -0 and +0 compare equal: among equal logits the lower expert id comes first
    lg = np.array([[0x8000, 0x0000, 0xBF80, 0x8000, 0x0000]], np.uint16)  # -0, +0, -1, -0, +0
    ids, w = Q.route_topk(lg, 4)
    assert ids[0].tolist() == [0, 1, 3, 4]
    assert np.all(w[0] == w[0, 0])


def test_routing_renormalised_is_softmax_over_the_chosen():
    # p_k / sum_{chosen} p_j: the softmax taken over the chosen logits alone
    lg = synth.bf16_normal(synth.rng(5, 0), (4, 64))
    ids, wr = Q.route_topk(lg, 6, renormalize=True)
    v = F.bf16_to_f64(lg)
    for m in range(4):
        sel = v[m, ids[m].astype(int)]
        e = np.exp(sel - sel.max())
        assert np.allclose(wr[m], e / e.sum(), rtol=1e-14)


def test_dispatch_groups_pairs():
    ids = np.array([[3, 1], [1, 0], [3, 2]], np.int32)
    off, pairs = Q.dispatch(ids, 5)
    assert off.tolist() == [0, 1, 3, 4, 6, 6]
    assert pairs.tolist() == [3, 1, 2, 5, 0, 4]


def _moe_exact(c, ids, w, I, topk):
    """Exact rational gate_up / down (silu in fp64), independent of the oracle code."""
    x = F.bf16_to_f64(c["x"])
    M, H = x.shape
    y = np.zeros((M, H))
    for m in range(M):
        for j in range(topk):
            e = int(ids[m, j])
            g = [sum(_dequant_exact(c["w13"][e], c["s13"][e], i, k) * Fraction(float(x[m, k])) for k in range(H)) for i in range(I)]
            u = [sum(_dequant_exact(c["w13"][e], c["s13"][e], I + i, k) * Fraction(float(x[m, k])) for k in range(H)) for i in range(I)]
            gf = np.array([float(v) for v in g])
            h = F.bf16_to_f64(F.round_to_bf16(gf / (1 + np.exp(-gf)) * np.array([float(v) for v in u])))
            for n in range(H):
                o = sum(_dequant_exact(c["w2"][e], c["s2"][e], n, i) * Fraction(float(h[i])) for i in range(I))
                y[m, n] += w[m, j] * float(o)
    return y


def test_moe_small_exact():
    c = synth.moe_case(2, E=6, H=64, I=32, seed=5)
    r = Q.moe_mxfp4(c["x"], c["logits"], c["w13"], c["s13"], c["w2"], c["s2"], I=32, topk=2)
    ye = _moe_exact(c, r["ids"], r["weights"], 32, 2)
    assert np.allclose(r["y_f64"], ye, rtol=1e-10, atol=1e-12)


def test_moe_gate_up_order():
    """W13 rows [0, I) are the gate (through SiLU), rows [I, 2I) are up: build weights with
    g = 6*x0 and u = x0 and check h = silu(g)*u, not silu(u)*g."""
    E, H, I = 1, 32, 32
    w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    s13 = np.full((E, 2 * I, 1), 127, np.uint8)
    w13[0, :I, 0] = 0x07      # code 7 = 6.0 at k=0 (low nibble)
    w13[0, I:, 0] = 0x02      # code 2 = 1.0 at k=0
    x = synth.f32_to_bf16_bits(np.array([[1.0] + [0.0] * (H - 1)], np.float32))
    st = Q.moe_gate_up(x, np.zeros((1, 1), np.int32), w13, s13, I)
    assert np.allclose(st["h_f64"], 6.0 / (1 + np.exp(-6.0)) * 1.0)


def test_moe_expert_relabel_invariance():
    c = synth.moe_case(3, E=5, H=64, I=32, seed=6)
    r = Q.moe_mxfp4(c["x"], c["logits"], c["w13"], c["s13"], c["w2"], c["s2"], I=32, topk=2)
    perm = np.array([2, 4, 0, 1, 3])          # new slot of old expert e is perm[e]
    inv = np.argsort(perm)
    c2 = {k: (v[inv] if k in ("w13", "s13", "w2", "s2") else v) for k, v in c.items()}
    c2["logits"] = c["logits"][:, inv]
    r2 = Q.moe_mxfp4(c2["x"], c2["logits"], c2["w13"], c2["s13"], c2["w2"], c2["s2"], I=32, topk=2)
    assert np.array_equal(r["y"], r2["y"])


def test_moe_single_expert_is_two_dense_gemvs():
    c = synth.moe_case(1, E=1, H=64, I=32, seed=7)
    r = Q.moe_mxfp4(c["x"], c["logits"], c["w13"], c["s13"], c["w2"], c["s2"], I=32, topk=1)
    assert r["weights"][0, 0] == 1.0
    x = F.bf16_to_f64(c["x"])[0]
    W13 = Q.mxfp4_dequant(c["w13"][0], c["s13"][0])
    gu = W13 @ x
    h = F.bf16_to_f64(F.round_to_bf16(gu[:32] / (1 + np.exp(-gu[:32])) * gu[32:]))
    y = Q.mxfp4_dequant(c["w2"][0], c["s2"][0]) @ h
    assert np.array_equal(r["y"][0], F.round_to_bf16(y))


def test_planted_swapped_nibbles_caught(monkeypatch):
    """Negative control: a high-nibble-first unpack must fail the exact dequant pin."""
    def swapped(p):
        p = np.asarray(p, np.uint8)
        out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
        out[..., 0::2], out[..., 1::2] = p >> 4, p & 0xF
        return out
    monkeypatch.setattr(Q, "unpack_e2m1", swapped)
    with pytest.raises(AssertionError):
        test_mxfp4_dequant_exact_brute_force()


# ------------------------------------------------------------------ clamped SwiGLU
def test_swiglu_alpha_closed_form():
    """sigmoid(ln 3) = 3/4, so silu(ln 3) = (3/4) ln 3.  With alpha = 2 and g = ln(3)/2 the
    activation is (3/4) ln 3 * u; alpha outside the SiLU or dropped gives another number."""
    g, u = np.log(3.0) / 2, 4.0
    assert Q.swiglu(g, u, alpha=2.0, limit=10.0) == pytest.approx(0.75 * np.log(3.0) * 4.0, rel=1e-15)
    assert Q.swiglu(np.log(3.0), u) == pytest.approx(3.0 * np.log(3.0), rel=1e-15)


@pytest.mark.parametrize("alpha", [1.0, 1.702, 0.5])
def test_swiglu_odd_part_is_alpha_g_u(alpha):
    """silu(z) - silu(-z) = z (sigmoid(z) + sigmoid(-z) = 1): h(g) - h(-g) = alpha g u while
    |g| stays inside the clamp."""
    g = np.linspace(-9.5, 9.5, 39)
    u = np.linspace(-7.0, 7.0, 39)
    d = Q.swiglu(g, u, alpha, 10.0) - Q.swiglu(-g, u, alpha, 10.0)
    assert np.allclose(d, alpha * g * u, rtol=1e-12, atol=1e-12)


def test_swiglu_gate_capped_from_above_only():
    u = np.array([3.0, -2.5, 0.75])
    for g in (10.0, 10.5, 20.0, 1e6):  # at or above the limit the gate no longer matters
        assert np.array_equal(Q.swiglu(g, u, 1.0, 10.0), Q.swiglu(10.0, u))
    # no lower cap: a gate of -20 is used as it is, not raised to -10
    assert np.array_equal(Q.swiglu(-20.0, u, 1.0, 10.0), Q.swiglu(-20.0, u))
    assert not np.allclose(Q.swiglu(-20.0, u, 1.0, 10.0), Q.swiglu(-10.0, u))


def test_swiglu_up_clipped_both_ways():
    g = np.array([0.3, -1.0, 4.0])
    assert np.array_equal(Q.swiglu(g, 25.0, 1.0, 10.0), Q.swiglu(g, 10.0))
    assert np.array_equal(Q.swiglu(g, -25.0, 1.0, 10.0), Q.swiglu(g, -10.0))
    assert np.array_equal(Q.swiglu(g, 9.0, 1.0, 10.0), Q.swiglu(g, 9.0))
    # roles not swapped: gate -25 kept, up -25 clipped to -10
    assert Q.swiglu(-25.0, -25.0, 1.0, 10.0) == Q.swiglu(-25.0, -10.0)


def test_swiglu_no_limit_is_silu_mul():
    rng = np.random.default_rng(3)
    g, u = rng.normal(0, 8, 64), rng.normal(0, 8, 64)
    assert np.array_equal(Q.swiglu(g, u), Q.silu(g) * u)
    assert np.array_equal(Q.swiglu(g, u, 1.0, 1e300), Q.swiglu(g, u))


def test_moe_gate_up_passes_the_clamp_through():
    """Expert weights giving g = 12 (code 6.0 at scale 2^1) and u = 12 under limit 10 equal,
    in the clamped stage, an expert giving g = u = 10 exactly (6 + 4) with no clamp."""
    E, H, I = 1, 32, 32
    x = synth.f32_to_bf16_bits(np.array([[1.0, 1.0] + [0.0] * (H - 2)], np.float32))
    big = np.zeros((E, 2 * I, H // 2), np.uint8)
    big[0, :, 0] = 0x07                          # k=0: 6.0, k=1: 0
    s_big = np.full((E, 2 * I, 1), 128, np.uint8)  # 2^1
    ten = np.zeros((E, 2 * I, H // 2), np.uint8)
    ten[0, :, 0] = 0x67                          # k=0: 6.0 (low nibble), k=1: 4.0 (high nibble)
    s_one = np.full((E, 2 * I, 1), 127, np.uint8)
    ids = np.zeros((1, 1), np.int32)
    a = Q.moe_gate_up(x, ids, big, s_big, I, limit=10.0)
    b = Q.moe_gate_up(x, ids, ten, s_one, I)
    assert np.all(a["g"] == 12.0) and np.all(b["g"] == 10.0)
    assert np.array_equal(a["h"], b["h"])
    assert not np.array_equal(Q.moe_gate_up(x, ids, big, s_big, I)["h"], b["h"])


# ------------------------------------------------------------------ grouped MoE, 1x128 E4M3 activations
def test_moe_act_quant_single_expert_is_the_dense_act_quant_linear():
    """E = 1, top-1: stage 1 is the dense MXFP4 linear with 1x128 E4M3 activations on W13 and
    stage 2 the same on W2 with h as the activations (a different oracle path, pinned itself)."""
    c = synth.moe_case(5, E=1, H=256, I=128, seed=41)
    r = Q.moe_mxfp4_act_quant(c["x"], c["logits"], c["w13"], c["s13"], c["w2"], c["s2"], I=128, topk=1)
    d1 = Q.mxfp4_act_quant(c["x"], c["w13"][0], c["s13"][0])
    assert np.array_equal(r["stage1"]["g"], d1["y_f64"][:, :128])
    assert np.array_equal(r["stage1"]["u"], d1["y_f64"][:, 128:])
    d2 = Q.mxfp4_act_quant(r["stage1"]["h"], c["w2"][0], c["s2"][0])
    assert np.array_equal(r["y_f64"], d2["y_f64"])


def test_moe_act_quant_lossless_x_matches_bf16_stage1():
    """x whose every 128-group is E4M3 codes times one power of two quantises losslessly, so
    stage 1 equals the bf16-activation MoE's stage 1."""
    E, H, I, M, topk = 6, 256, 128, 3, 2
    c = synth.moe_case(M, E=E, H=H, I=I, seed=42)
    rng = np.random.default_rng(42)
    vals = F.e4m3_decode(rng.integers(0, 0x7F, size=(M, H)).astype(np.uint8))  # finite, >= 0
    vals = vals * np.where(rng.random((M, H)) < 0.5, -1.0, 1.0)
    vals[:, ::128] = 448.0  # group amax 448: the UE8M0 scale is 2^0
    x = synth.f32_to_bf16_bits((vals * 2.0 ** -4).astype(np.float32))  # exact in bf16
    ids, _ = Q.route_topk(c["logits"], topk)
    a = Q.moe_gate_up_act_quant(x, ids, c["w13"], c["s13"], I)
    b = Q.moe_gate_up(x, ids, c["w13"], c["s13"], I)
    assert np.array_equal(a["g"], b["g"]) and np.array_equal(a["u"], b["u"])
    assert np.array_equal(a["h"], b["h"])


def test_moe_act_quant_clamp_passes_through():
    c = synth.moe_case(4, E=4, H=256, I=128, seed=43)
    ids, _ = Q.route_topk(c["logits"], 2)
    a = Q.moe_gate_up_act_quant(c["x"], ids, c["w13"], c["s13"], 128, limit=10.0)
    assert np.array_equal(a["h_f64"], Q.swiglu(a["g"], a["u"], 1.0, 10.0))
    assert np.any(a["g"] > 10.0)
