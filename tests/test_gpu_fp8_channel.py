"""FP8 weights with per-channel / per-tensor fp32 scales (e4m3fn and e5m2 codes): CUDA path vs
the oracle on identical seeded inputs.  y within 1e-3*|w_s| sum|w x| + 1 bf16 ulp (the float
bar); bias added after the bf16 cast."""
import numpy as np
import pytest
import torch

import synth
from _util import bits_of, check_float, gpu_lib, sample_rows, to_bf16_tensor
from oracle import formats as F
from oracle import qlinear_oracle as Q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ql():
    return gpu_lib()


def run(ql, c, fmt, bias=None):
    x = to_bf16_tensor(c["x"])
    w = torch.from_numpy(c["w"]).cuda()
    s = torch.from_numpy(c["w_s"]).cuda()
    b = None if bias is None else to_bf16_tensor(bias)
    y, path = ql.qlinear_fp8(x, w, s, fmt, b, debug=True)
    torch.cuda.synchronize()
    assert path == "fp8_channel_skinny"
    return bits_of(y)


def compare(c, y, fmt, K, rows=None, bias=None):
    ref, a = Q.fp8_channel(c["x"], c["w"], fmt, c["w_s"], K, rows=rows)
    sl = slice(None) if rows is None else rows
    if bias is None:
        check_float(y[:, sl], ref, a)
    else:
        yb = F.round_to_bf16(F.bf16_to_f64(F.round_to_bf16(ref)) + F.bf16_to_f64(bias)[None, sl])
        check_float(y[:, sl], F.bf16_to_f64(yb), a)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (3, 200, 144), (16, 384, 1024), (9, 1000, 2048),
                                   (5, 77, 16), (2, 130, 17408), (12, 4097, 320)])
def test_fp8_channel_small_and_ragged(ql, fmt, per_channel, M, N, K):
    c = synth.fp8_channel_case(M, N, K, seed=M + N, w_fmt=fmt, per_channel=per_channel)
    compare(c, run(ql, c, fmt), fmt, K)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_channel_padded_rows_nan_padding(ql, fmt):
    # rows padded to K + 48 with 0xFF (NaN in both formats): the kernel must never read past K
    c = synth.fp8_channel_case(4, 300, 784, seed=7, ldw=784 + 48, w_fmt=fmt)
    compare(c, run(ql, c, fmt), fmt, 784)


def test_fp8_channel_bias(ql):
    c = synth.fp8_channel_case(3, 260, 512, seed=8, w_fmt="e5m2")
    bias = synth.bf16_normal(synth.rng(8, 3), (260,))
    compare(c, run(ql, c, "e5m2", bias), "e5m2", 512, bias=bias)


def test_fp8_channel_many_tokens_chunked(ql):
    c = synth.fp8_channel_case(33, 300, 640, seed=9)
    compare(c, run(ql, c, "e4m3"), "e4m3", 640)


def test_fp8_channel_rejects_bad_arguments(ql):
    c = synth.fp8_channel_case(2, 64, 256, seed=1)
    x = to_bf16_tensor(c["x"])
    w = torch.from_numpy(c["w"]).cuda()
    with pytest.raises(ql.QLError):  # scale length neither 1 nor N
        ql.qlinear_fp8(x, w, torch.ones(3, dtype=torch.float32, device="cuda"))
    with pytest.raises(KeyError):
        ql.qlinear_fp8(x, w, torch.ones(1, dtype=torch.float32, device="cuda"), "e3m4")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
@pytest.mark.parametrize("M", [1, 16])
def test_fp8_channel_full_size_sampled(ql, fmt, N, K, M):
    c = synth.fp8_channel_case(M, N, K, seed=0, w_fmt=fmt)
    rows = sample_rows(N, seed=M)
    compare(c, run(ql, c, fmt), fmt, K, rows=rows)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
def test_fp8_channel_full_size_every_row(ql, fmt, N, K):
    # every output row of a 1-token call (local activation images where they fit)
    c = synth.fp8_channel_case(1, N, K, seed=200, w_fmt=fmt)
    compare(c, run(ql, c, fmt), fmt, K)
