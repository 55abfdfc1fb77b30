"""Softmax top-k routing on the GPU against the oracle's routing: ids bit-exact, weights to 1e-6
relative (renormalised or not).

One warp router serves every MoE launch; its loops are unrolled to E/32 keys per lane (E up to
128, 256, 512 or 1024), so expert counts are taken from each size class and off multiples of 32.
Logits are coarse (multiples of 1/4), so many experts tie and the lower id must win, and carry
signed zeros (-0 and +0 compare equal).  Each launch path routes: the persistent kernel's fused
router (H and I multiples of 256), the routing launch of the register path (H = 128) and the
grouped path's per-token router (more than 16 tokens)."""
import numpy as np
import pytest
import torch

import synth
from _util import gpu_lib, to_bf16_tensor
from oracle import formats as F
from oracle import qlinear_oracle as Q

pytestmark = pytest.mark.gpu

_WEIGHTS = {}


@pytest.fixture(scope="module")
def ql():
    return gpu_lib()


def weights(E, H, I):
    key = (E, H, I)
    if key not in _WEIGHTS:
        w = synth.moe_weights_only(E, H, I, seed=E + H)
        _WEIGHTS.clear()  # one expert set on the device at a time
        _WEIGHTS[key] = [torch.from_numpy(w[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    return _WEIGHTS[key]


def tied_logits(M, E, seed):
    """bf16 bits of N(0,1) logits rounded to multiples of 1/4, with some exact zeros of both signs."""
    r = np.random.default_rng(seed)
    v = np.round(r.standard_normal((M, E)) * 4.0) / 4.0
    bits = F.round_to_bf16(v)
    zero = r.random((M, E)) < 0.1
    neg = r.random((M, E)) < 0.5
    bits[zero & neg] = 0x8000
    bits[zero & ~neg] = 0x0000
    return bits


def route_and_check(ql, M, E, H, I, topk, renorm, path, seed):
    wdev = weights(E, H, I)
    x = to_bf16_tensor(synth.bf16_normal(synth.rng(seed, 1), (M, H)))
    lg = tied_logits(M, E, seed)
    _, gi, gw, _, p = ql.moe_mxfp4_grouped(x, *wdev, router_logits=to_bf16_tensor(lg), topk=topk,
                                           renormalize=renorm, debug=True)
    torch.cuda.synchronize()
    assert p == path
    ids, wts = Q.route_topk(lg, topk, renormalize=renorm)
    assert np.array_equal(gi.cpu().numpy(), ids), "routing ids differ"
    assert np.allclose(gw.cpu().numpy(), wts, rtol=1e-6, atol=0), "routing weights differ"


@pytest.mark.parametrize("E", [100, 300, 1000])
@pytest.mark.parametrize("topk,renorm", [(1, False), (8, True), (16, False)])
def test_routing_fused_in_the_persistent_kernel(ql, E, topk, renorm):
    route_and_check(ql, 5, E, 256, 256, topk, renorm, "moe_mxfp4", seed=E + topk)


@pytest.mark.parametrize("E", [300, 1000])
@pytest.mark.parametrize("topk,renorm", [(8, False), (16, True)])
def test_routing_launch_of_the_register_path(ql, E, topk, renorm):
    route_and_check(ql, 3, E, 128, 128, topk, renorm, "moe_mxfp4", seed=2 * E + topk)


@pytest.mark.parametrize("E", [300, 1000])
@pytest.mark.parametrize("topk,renorm", [(8, True), (16, False)])
def test_routing_of_the_grouped_path(ql, E, topk, renorm):
    route_and_check(ql, 20, E, 256, 256, topk, renorm, "moe_mxfp4_tcgen05", seed=3 * E + topk)
