"""Device-side failure detection without a GPU fault: every wait in the skinny kernel is bounded
(ql_set_wait_limit).  With the limit at 0 the producer gives up on the activation hand-off at its
first poll, flags QL_DEV_TIMEOUT in the workspace status word, still issues its loads (so no
stage is left waiting) and the kernel returns; the host reads the flag, re-initialises the
workspace and the next call is exact again.  No wait here is unbounded and nothing traps."""
import numpy as np
import pytest
import torch

import synth
from _util import gpu_lib, to_bf16_tensor
from oracle import qlinear_oracle as Q

pytestmark = pytest.mark.gpu

DEV_TIMEOUT = 1
DEFAULT_WAIT_LIMIT = 1 << 20


@pytest.fixture(scope="module")
def ql():
    return gpu_lib()


def test_wait_timeout_is_reported_and_recoverable(ql):
    # M * K above the local-activation limit: the call shares one activation image, so its
    # producers wait for the image at the hand-off
    c = synth.int8_case(3, 640, 16384, seed=7)
    x = to_bf16_tensor(c["x"])
    w = torch.from_numpy(c["w"]).cuda()
    s = torch.from_numpy(c["w_s"]).cuda()
    ref = Q.int8_w8a8(c["x"], c["w"], c["w_s"])
    ws = ql.Workspace()

    def call():
        _, acc, _, _, _ = ql.qlinear_int8_w8a8(x, w, s, debug=True, workspace=ws)
        torch.cuda.synchronize()
        return acc.cpu().numpy()

    assert np.array_equal(call(), ref["acc"])
    st, flags = ql.read_device_status(ws.buf)
    assert st == 0 and flags == 0

    ql.set_wait_limit(0)
    try:
        seen = False
        for _ in range(8):  # the first poll finds the image unfinished in practice; retry to be sure
            call()
            st, flags = ql.read_device_status(ws.buf, clear=True)
            if flags & DEV_TIMEOUT:
                seen = True
                break
    finally:
        ql.set_wait_limit(DEFAULT_WAIT_LIMIT)
    assert seen, "a zero wait limit never timed out"
    assert st != 0  # read_device_status reports QL_ERR_TIMEOUT with the flag

    # the context survives: counters may be left mid-count, so re-initialise the workspace
    ws.buf.zero_()
    torch.cuda.synchronize()
    assert np.array_equal(call(), ref["acc"])
    st, flags = ql.read_device_status(ws.buf)
    assert st == 0 and flags == 0


def _timeout_then_exact(ql, call, check):
    """Run `call` (returns host results) with the wait limit at 0 until the status word shows
    QL_DEV_TIMEOUT, then with the default limit on a re-initialised workspace: `check` must
    pass again.  `call(ws)` takes the workspace to use."""
    ws = ql.Workspace()
    check(call(ws))
    st, flags = ql.read_device_status(ws.buf)
    assert st == 0 and flags == 0
    ql.set_wait_limit(0)
    try:
        seen = False
        for _ in range(8):
            call(ws)
            st, flags = ql.read_device_status(ws.buf, clear=True)
            if flags & DEV_TIMEOUT:
                seen = True
                break
    finally:
        ql.set_wait_limit(DEFAULT_WAIT_LIMIT)
    assert seen and st != 0, "a zero wait limit never timed out"
    ws.buf.zero_()
    torch.cuda.synchronize()
    check(call(ws))
    st, flags = ql.read_device_status(ws.buf)
    assert st == 0 and flags == 0


def test_int8_tcgen05_gemm_timeout_is_reported_and_recoverable(ql):
    """M > 16: the tcgen05 INT8 GEMM (producer, widening warps, MMA issuer and drain warps all
    bound their waits; in-flight loads and MMAs are waited for and tensor memory is freed)."""
    c = synth.int8_case(40, 384, 2048, seed=8)
    x, w, s = to_bf16_tensor(c["x"]), torch.from_numpy(c["w"]).cuda(), torch.from_numpy(c["w_s"]).cuda()
    ref = Q.int8_w8a8(c["x"], c["w"], c["w_s"])

    def call(ws):
        _, acc, _, _, path = ql.qlinear_int8_w8a8(x, w, s, debug=True, workspace=ws)
        torch.cuda.synchronize()
        assert path == "int8_tcgen05"
        return acc.cpu().numpy()

    _timeout_then_exact(ql, call, lambda acc: np.testing.assert_array_equal(acc, ref["acc"]))


def test_block_scaled_tcgen05_gemm_timeout_is_reported_and_recoverable(ql):
    """The block-scaled tcgen05 GEMM (FP8 weights, 1x128 E4M3 activations)."""
    from oracle import formats as F
    from _util import bits_of, check_float
    c = synth.fp8_block_case(64, 256, 1024, seed=9)
    x, w, s = to_bf16_tensor(c["x"]), torch.from_numpy(c["w"]).cuda(), torch.from_numpy(c["s"]).cuda()
    ref = Q.fp8_block_act_quant(c["x"], c["w"], c["s"], 1024)

    def call(ws):
        y, _, _, path = ql.qlinear_fp8_block(x, w, s, act_mode=ql.ACT_E4M3_1X128, debug=True, workspace=ws)
        torch.cuda.synchronize()
        assert path == "fp8_tcgen05"
        return bits_of(y)

    _timeout_then_exact(ql, call, lambda y: check_float(y, ref["y_f64"], ref["abs_sum"]))


def test_grouped_moe_timeout_is_reported_and_recoverable(ql):
    """M > 16 MoE: routing, dispatch and the two grouped tcgen05 GEMMs."""
    c = synth.moe_case(20, E=8, H=256, I=256, seed=10)
    wd = [torch.from_numpy(c[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    x, lg = to_bf16_tensor(c["x"]), to_bf16_tensor(c["logits"])
    rid, _ = Q.route_topk(c["logits"], 2)

    def call(ws):
        y, ids, _, _, path = ql.moe_mxfp4_grouped(x, *wd, router_logits=lg, topk=2, debug=True, workspace=ws)
        torch.cuda.synchronize()
        assert path == "moe_mxfp4_tcgen05"
        return ids.cpu().numpy(), y.float().cpu().numpy()

    first = {}

    def check(res):
        ids, y = res
        np.testing.assert_array_equal(ids, rid)
        if "y" in first:  # the same inputs give the same outputs once the workspace is clean
            np.testing.assert_array_equal(y, first["y"])
        else:
            first["y"] = y

    _timeout_then_exact(ql, call, check)
