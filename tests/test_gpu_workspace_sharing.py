"""One workspace shared by every operation, in an interleaved order: each result must be
bit-identical to the same call on a fresh workspace.  The operations carve different regions of
the same buffer (activation images, partial sums, routing lists, per-expert counters), so a
call that relied on state left by another would show here."""
import numpy as np
import pytest
import torch

import synth
from _util import bits_of, gpu_lib, to_bf16_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ql():
    return gpu_lib()


def _calls(ql):
    i8a = synth.int8_case(4, 640, 1024, seed=51)
    i8b = synth.int8_case(40, 384, 1024, seed=52)
    bf = synth.bf16_dense_case(3, 260, 512, seed=53)
    f8 = synth.fp8_channel_case(5, 300, 768, seed=54, w_fmt="e5m2")
    moe_s = synth.moe_case(3, 16, 512, 256, seed=55)
    moe_g = synth.moe_case(24, 16, 512, 256, seed=56)

    def dev(a):
        return torch.from_numpy(a).cuda()

    def int8(c):
        return lambda ws: ql.qlinear_int8_w8a8(to_bf16_tensor(c["x"]), dev(c["w"]), dev(c["w_s"]), workspace=ws)

    def bf16(ws):
        w = torch.from_numpy(bf["w"].view(np.int16)).cuda().view(torch.bfloat16)
        return ql.qlinear_bf16(to_bf16_tensor(bf["x"]), w, workspace=ws)

    def fp8(ws):
        return ql.qlinear_fp8(to_bf16_tensor(f8["x"]), dev(f8["w"]), dev(f8["w_s"]), "e5m2", workspace=ws)

    def moe(c, topk):
        def f(ws):
            wd = [dev(c[k]) for k in ("w13", "s13", "w2", "s2")]
            return ql.moe_mxfp4_grouped(to_bf16_tensor(c["x"]), *wd, router_logits=to_bf16_tensor(c["logits"]),
                                        topk=topk, workspace=ws)
        return f

    return [("int8 skinny", int8(i8a)), ("moe grouped", moe(moe_g, 4)), ("bf16", bf16), ("int8 gemm", int8(i8b)),
            ("moe skinny", moe(moe_s, 4)), ("fp8 e5m2", fp8), ("moe grouped", moe(moe_g, 4)),
            ("int8 skinny", int8(i8a))]


def test_interleaved_calls_on_one_workspace_match_fresh_workspaces(ql):
    calls = _calls(ql)
    fresh = []
    for _, f in calls:
        fresh.append(bits_of(f(ql.Workspace())))
        torch.cuda.synchronize()
    shared = ql.Workspace()
    shared.get(64 << 20)  # sized once up front, so no call gets a freshly zeroed buffer
    for (name, f), want in zip(calls, fresh):
        got = bits_of(f(shared))
        torch.cuda.synchronize()
        assert np.array_equal(got, want), f"{name}: result differs on the shared workspace"
    st, flags = ql.read_device_status(shared.buf)
    assert flags == 0
