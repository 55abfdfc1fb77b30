"""Grouped MoE for batches of more than 16 tokens (tcgen05 path, x and h quantised per token and
128-K group to E4M3 with UE8M0 scales): CUDA path vs the oracle.  Routing ids bit-exact, weights
to 1e-6 relative; h within the float tolerance carried through the activation; y within the
float bar on the kernel's own h (quantised by the oracle, exactly as the kernel does)."""
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


def run(ql, c, wdev, topk, ids=None, wts=None, alpha=1.0, limit=None):
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
    assert path == "moe_mxfp4_tcgen05"
    return bits_of(y), gi.cpu().numpy(), gw.cpu().numpy(), bits_of(h)


def check(c, got, I, topk, cols=None, rows=None, ids=None, wts=None, alpha=1.0, limit=None):
    y, gi, gw, h = got
    if ids is None:
        ids, wts = Q.route_topk(c["logits"], topk)
        assert np.array_equal(gi, ids), "routing ids differ"
        assert np.allclose(gw, wts, rtol=1e-6, atol=0), "routing weights differ"
    valid = np.asarray(ids) >= 0
    cols = np.arange(I) if cols is None else cols
    pairs = np.flatnonzero(valid.reshape(-1))
    st = Q.moe_gate_up_act_quant(c["x"], np.where(valid, ids, 0), c["w13"], c["s13"], I, pairs=pairs, cols=cols,
                                 alpha=alpha, limit=limit)
    hv = F.bf16_to_f64(h[pairs][:, cols])
    err = np.abs(hv - F.bf16_to_f64(st["h"]))
    tol = h_tolerance(st, alpha, limit)
    assert np.all(err <= tol), f"h: {np.sum(err > tol)} of {err.size} entries outside tolerance"
    # stage 2 on the kernel's own h (pairs that were not dispatched carry weight 0)
    w_eff = np.where(valid, np.asarray(gw, np.float64), 0.0)
    h_used = np.where(valid.reshape(-1, 1), h, 0).astype(np.uint16)
    yb, y64, a = Q.moe_down_combine_act_quant(h_used, np.where(valid, ids, 0), w_eff, c["w2"], c["s2"], rows=rows)
    sl = slice(None) if rows is None else rows
    check_float(y[:, sl], y64, a)
    return st


@pytest.mark.parametrize("M,E,topk", [(17, 16, 4), (40, 16, 4), (100, 32, 8), (64, 4, 2)])
def test_moe_grouped_small(ql, M, E, topk):
    H, I = 256, 256
    c = synth.moe_case(M, E, H, I, seed=80 + M + E)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    check(c, run(ql, c, wdev, topk), I, topk)


def test_moe_grouped_long_k_and_ragged_tiles(ql):
    # H = 1024 (8 groups), I = 384 (3 groups); 8 experts over 50 tokens x top-3 = 150 pairs
    M, E, H, I, topk = 50, 8, 1024, 384, 3
    c = synth.moe_case(M, E, H, I, seed=90)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    check(c, run(ql, c, wdev, topk), I, topk)


def test_moe_grouped_given_ids_with_an_invalid_id(ql):
    M, E, H, I, topk = 20, 8, 256, 128, 2
    c = synth.moe_case(M, E, H, I, seed=91)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    rng = np.random.default_rng(91)
    ids = np.stack([rng.choice(E, size=topk, replace=False) for _ in range(M)]).astype(np.int32)
    ids[3, 1] = E + 5  # out of range: flagged and not dispatched
    wts = rng.uniform(0.1, 1.0, size=(M, topk)).astype(np.float32)
    ws = ql.Workspace()
    x = to_bf16_tensor(c["x"])
    y, gi, gw, h, path = ql.moe_mxfp4_grouped(x, *wdev, topk_ids=torch.from_numpy(ids).cuda(),
                                              topk_weights=torch.from_numpy(wts).cuda(), debug=True, workspace=ws)
    torch.cuda.synchronize()
    assert path == "moe_mxfp4_tcgen05"
    st, flags = ql.read_device_status(ws.buf, clear=True)
    assert flags & 2, "the out-of-range expert id was not flagged"
    gi = gi.cpu().numpy()
    exp_ids = ids.copy()
    exp_ids[3, 1] = -1
    assert np.array_equal(gi, exp_ids)
    check(c, (bits_of(y), gi, gw.cpu().numpy(), bits_of(h)), I, topk, ids=exp_ids, wts=wts)


def test_moe_grouped_swiglu_clamp(ql):
    M, E, H, I, topk = 33, 16, 512, 256, 4
    c = synth.moe_case(M, E, H, I, seed=92)
    wdev = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    st = check(c, run(ql, c, wdev, topk, alpha=1.0, limit=10.0), I, topk, alpha=1.0, limit=10.0)
    assert np.any(st["g"] > 10.0) and np.any(np.abs(st["u"]) > 10.0)


@pytest.fixture(scope="module")
def moe_full():
    E, H, I = 256, 4096, 2048
    w = synth.moe_weights_only(E, H, I, seed=0)
    dev = [torch.from_numpy(w[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    return w, dev


@pytest.mark.parametrize("M", [32, 128])
def test_moe_grouped_full_size_sampled(ql, moe_full, M):
    E, H, I, topk = 256, 4096, 2048, 8
    w, dev = moe_full
    c = dict(w, **synth.moe_tokens(M, E, H, seed=5))
    got = run(ql, c, dev, topk)
    check(c, got, I, topk, cols=sample_rows(I, 16, seed=M), rows=sample_rows(H, 16, seed=M + 1))
