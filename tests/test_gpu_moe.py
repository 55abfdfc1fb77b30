"""MXFP4 dense (bf16 activations) and MXFP4 MoE parity: CUDA path vs the oracle.
Routing ids bit-exact; weights to 1e-6 relative; h and y stage by stage within the float
tolerance propagated through SiLU*mul (see test docstrings)."""
import numpy as np
import pytest
import torch

import synth
from _util import bits_of, check_float, gpu_lib, h_tolerance, sample_rows, to_bf16_tensor
from oracle import formats as F
from oracle import qlinear_oracle as Q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ql():
    return gpu_lib()


# ------------------------------------------------------------------ MXFP4 dense, bf16 activations
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (7, 130, 1024), (16, 512, 4096), (3, 64, 96), (2, 2048, 8192),
                                   (1, 1000, 40960)])
def test_mxfp4_dense_bf16(ql, M, N, K):
    c = synth.mxfp4_dense_case(M, N, K, seed=M + N)
    x = to_bf16_tensor(c["x"])
    # scale rows padded to a multiple of 4 bytes with NaN scales (255): never read
    lds = -(-(K // 32) // 4) * 4
    sp = np.full((N, lds), 255, np.uint8)
    sp[:, : K // 32] = c["s"]
    y, _, _, path = ql.qlinear_mxfp4(x, torch.from_numpy(c["w"]).cuda(), torch.from_numpy(sp).cuda(), debug=True)
    torch.cuda.synchronize()
    assert path == "mxfp4_skinny"
    w = Q.mxfp4_dequant(c["w"], c["s"])
    xv = F.bf16_to_f64(c["x"])
    check_float(bits_of(y), xv @ w.T, np.abs(xv) @ np.abs(w).T)


# ------------------------------------------------------------------ MoE
def run_moe(ql, c, wdev, topk, ids=None, wts=None, alpha=1.0, limit=None):
    x = to_bf16_tensor(c["x"])
    kw = {}
    if ids is None:
        kw["router_logits"] = to_bf16_tensor(c["logits"])
    else:
        kw["topk_ids"] = torch.from_numpy(ids).cuda()
        kw["topk_weights"] = torch.from_numpy(wts).cuda()
    y, gi, gw, h, path = ql.moe_mxfp4_grouped(x, *wdev, topk=topk, swiglu_alpha=alpha, swiglu_limit=limit,
                                              debug=True, **kw)
    torch.cuda.synchronize()
    assert path == "moe_mxfp4"
    return bits_of(y), gi.cpu().numpy(), gw.cpu().numpy(), bits_of(h)


def check_moe(c, got, I, topk, cols=None, rows=None, ids=None, wts=None, alpha=1.0, limit=None):
    y, gi, gw, h = got
    if ids is None:
        ids, wts = Q.route_topk(c["logits"], topk)
        assert np.array_equal(gi, ids), "routing ids differ"
        assert np.allclose(gw, wts, rtol=1e-6, atol=0), "routing weights differ"
    M = c["x"].shape[0]
    cols = np.arange(I) if cols is None else cols
    st = Q.moe_gate_up(c["x"], ids, c["w13"], c["s13"], I, cols=cols, alpha=alpha, limit=limit)
    hv = F.bf16_to_f64(h[:, cols])
    err = np.abs(hv - F.bf16_to_f64(st["h"]))
    tol = h_tolerance(st, alpha, limit)
    assert np.all(err <= tol), f"h: {np.sum(err > tol)} entries outside tolerance"
    # stage 2 on the kernel's own h: y within 1e-3 * sum_j |w_j| sum_i |W2 h| + 1 ulp
    yb, y64, a = Q.moe_down_combine(h, ids, np.asarray(gw, np.float64), c["w2"], c["s2"], rows=rows)
    sl = slice(None) if rows is None else rows
    check_float(y[:, sl], y64, a)
    return st


@pytest.mark.parametrize("M", [1, 3, 9, 16])
def test_moe_small(ql, M):
    E, H, I, topk = 16, 256, 128, 4
    c = synth.moe_case(M, E, H, I, seed=M)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    check_moe(c, run_moe(ql, c, wdev, topk), I, topk)


@pytest.mark.parametrize("M,E,topk", [(1, 16, 4), (3, 16, 4), (9, 16, 4), (16, 16, 4), (16, 4, 2), (8, 64, 8)])
def test_moe_small_persistent_kernel(ql, M, E, topk):
    # H and I whole 256-K units: both expert GEMVs run on the persistent TMA kernel; (16, 4, 2)
    # puts 8 pairs on each expert on average (up to all 16 tokens on one)
    H, I = 512, 256
    c = synth.moe_case(M, E, H, I, seed=40 + M + E)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    check_moe(c, run_moe(ql, c, wdev, topk), I, topk)


def test_moe_persistent_given_ids(ql):
    E, H, I, topk = 8, 256, 512, 2
    c = synth.moe_case(4, E, H, I, seed=33)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    ids = np.array([[0, 7], [7, 0], [3, 4], [5, 6]], np.int32)
    wts = np.array([[0.25, 0.75], [1.0, 0.5], [0.1, 0.2], [0.3, 0.3]], np.float32)
    got = run_moe(ql, c, wdev, topk, ids=ids, wts=wts)
    assert np.array_equal(got[1], ids)
    check_moe(c, got, I, topk, ids=ids, wts=wts)


def test_moe_persistent_given_ids_more_than_8_tokens(ql):
    # 9..16 tokens run as two calls of 8 and M - 8 tokens: the given ids and weights, the debug
    # outputs and y of the second call sit at row 8 of every array
    E, H, I, topk, M = 8, 256, 512, 3, 13
    c = synth.moe_case(M, E, H, I, seed=34)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    r = synth.rng(34, 7)
    ids = np.stack([r.permutation(E)[:topk] for _ in range(M)]).astype(np.int32)
    wts = r.uniform(0.05, 1.0, (M, topk)).astype(np.float32)
    got = run_moe(ql, c, wdev, topk, ids=ids, wts=wts)
    assert np.array_equal(got[1], ids)
    check_moe(c, got, I, topk, ids=ids, wts=wts)


def test_moe_given_ids_and_renormalised_routing(ql):
    E, H, I, topk = 8, 128, 128, 2
    c = synth.moe_case(4, E, H, I, seed=31)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    ids = np.array([[0, 7], [7, 0], [3, 3 + 1], [5, 6]], np.int32)
    wts = np.array([[0.25, 0.75], [1.0, 0.5], [0.1, 0.2], [0.3, 0.3]], np.float32)
    got = run_moe(ql, c, wdev, topk, ids=ids, wts=wts)
    assert np.array_equal(got[1], ids)
    check_moe(c, got, I, topk, ids=ids, wts=wts)
    x = to_bf16_tensor(c["x"])
    _, gi, gw, _, _ = ql.moe_mxfp4_grouped(x, *wdev, router_logits=to_bf16_tensor(c["logits"]), topk=topk,
                                          renormalize=True, debug=True)
    rid, rw = Q.route_topk(c["logits"], topk, renormalize=True)
    assert np.array_equal(gi.cpu().numpy(), rid)
    assert np.allclose(gw.cpu().numpy(), rw, rtol=1e-6)


def test_moe_routing_ties(ql):
    E, H, I, topk = 32, 128, 128, 8
    c = synth.moe_case(2, E, H, I, seed=32)
    c["logits"][0] = synth.f32_to_bf16_bits(np.round(np.linspace(-2, 2, E)).astype(np.float32))  # many ties
    c["logits"][1] = 0
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    check_moe(c, run_moe(ql, c, wdev, topk), I, topk)


@pytest.fixture(scope="module")
def moe_full():
    E, H, I = 256, 4096, 2048
    w = synth.moe_weights_only(E, H, I, seed=0)
    dev = [torch.from_numpy(w[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    return w, dev


@pytest.mark.parametrize("M", [1, 2, 5, 9])
def test_moe_full_size_sampled(ql, moe_full, M):
    E, H, I, topk = 256, 4096, 2048, 8
    w, dev = moe_full
    c = dict(w, **synth.moe_tokens(M, E, H, seed=0))
    got = run_moe(ql, c, dev, topk)
    check_moe(c, got, I, topk, cols=sample_rows(I, 24, seed=M), rows=sample_rows(H, 24, seed=M + 1))


# ------------------------------------------------------------------ clamped SwiGLU
def _clamps_exercised(st, limit):
    """the case really clamps: some gates above the limit, some ups beyond it on each side"""
    g, u = st["g"], st["u"]
    assert np.any(g > limit) and np.any(u > limit) and np.any(u < -limit)


@pytest.mark.parametrize("alpha,limit", [(1.0, 10.0), (1.702, 7.0)])
@pytest.mark.parametrize("M", [1, 9])
def test_moe_swiglu_clamp_persistent_kernel(ql, M, alpha, limit):
    E, H, I, topk = 16, 512, 256, 4
    c = synth.moe_case(M, E, H, I, seed=60 + M)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    st = check_moe(c, run_moe(ql, c, wdev, topk, alpha=alpha, limit=limit), I, topk, alpha=alpha, limit=limit)
    _clamps_exercised(st, limit)


@pytest.mark.parametrize("M", [2, 16])
def test_moe_swiglu_clamp_register_kernel(ql, M):
    # I = 128: not a whole 256-K unit, so the MoE runs on the register kernel path
    E, H, I, topk = 16, 256, 128, 4
    c = synth.moe_case(M, E, H, I, seed=70 + M)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    st = check_moe(c, run_moe(ql, c, wdev, topk, alpha=1.0, limit=3.0), I, topk, alpha=1.0, limit=3.0)
    _clamps_exercised(st, 3.0)


def test_moe_swiglu_rejects_bad_parameters(ql):
    E, H, I, topk = 8, 256, 256, 2
    c = synth.moe_case(1, E, H, I, seed=5)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    for alpha, limit in ((float("nan"), 10.0), (1.0, -1.0), (1.0, float("nan")), (float("inf"), 10.0)):
        with pytest.raises(ql.QLError):
            run_moe(ql, c, wdev, topk, alpha=alpha, limit=limit)


@pytest.mark.parametrize("M", [1, 9])
def test_moe_swiglu_clamp_full_size_sampled(ql, moe_full, M):
    E, H, I, topk = 256, 4096, 2048, 8
    w, dev = moe_full
    c = dict(w, **synth.moe_tokens(M, E, H, seed=3))
    got = run_moe(ql, c, dev, topk, alpha=1.0, limit=10.0)
    st = check_moe(c, got, I, topk, cols=sample_rows(I, 48, seed=M), rows=sample_rows(H, 24, seed=M + 1),
                   alpha=1.0, limit=10.0)
    _clamps_exercised(st, 10.0)
