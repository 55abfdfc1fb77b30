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
