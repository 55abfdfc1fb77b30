"""BF16 dense GEMV parity: CUDA path vs the oracle on identical seeded inputs.
y within 1e-3*sum|w x| + 1 bf16 ulp (the float bar); bias added after the bf16 cast."""
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


def run(ql, c, bias=None):
    x = to_bf16_tensor(c["x"])
    w = torch.from_numpy(c["w"].view(np.int16)).cuda().view(torch.bfloat16)
    b = None if bias is None else to_bf16_tensor(bias)
    y, path = ql.qlinear_bf16(x, w, b, debug=True)
    torch.cuda.synchronize()
    assert path == "bf16_skinny"
    return bits_of(y)


def compare(c, y, K, rows=None, bias=None):
    ref, a = Q.bf16_linear(c["x"], c["w"], K, rows=rows)
    sl = slice(None) if rows is None else rows
    if bias is None:
        check_float(y[:, sl], ref, a)
    else:
        # bias after the cast: compare bf16(y_ref) + bias, one more rounding on both sides
        yb = F.round_to_bf16(F.bf16_to_f64(F.round_to_bf16(ref)) + F.bf16_to_f64(bias)[None, sl])
        check_float(y[:, sl], F.bf16_to_f64(yb), a)


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (3, 200, 136), (16, 384, 1024), (9, 1000, 2048),
                                   (5, 77, 8), (2, 130, 17408), (12, 4097, 320)])
def test_bf16_small_and_ragged(ql, M, N, K):
    c = synth.bf16_dense_case(M, N, K, seed=M + N)
    compare(c, run(ql, c), K)


def test_bf16_padded_rows_nan_padding(ql):
    # rows padded to K + 64 with NaN: the kernel must never read past K
    c = synth.bf16_dense_case(4, 300, 768, seed=7, ldw=768 + 64)
    compare(c, run(ql, c), 768)


def test_bf16_bias(ql):
    c = synth.bf16_dense_case(3, 260, 512, seed=8)
    bias = synth.bf16_normal(synth.rng(8, 3), (260,))
    compare(c, run(ql, c, bias), 512, bias=bias)


def test_bf16_many_tokens_chunked(ql):
    c = synth.bf16_dense_case(33, 300, 640, seed=9)
    compare(c, run(ql, c), 640)


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_bf16_full_size_sampled(ql, N, K, M):
    c = synth.bf16_dense_case(M, N, K, seed=0)
    rows = sample_rows(N, seed=M)
    compare(c, run(ql, c), K, rows=rows)


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
def test_bf16_full_size_every_row(ql, N, K):
    c = synth.bf16_dense_case(4, N, K, seed=201)
    compare(c, run(ql, c), K)
