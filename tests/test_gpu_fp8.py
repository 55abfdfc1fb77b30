"""FP8 E4M3 128x128 block-scaled parity (bf16 activations): CUDA path vs the oracle.
y within 1e-3*sum|w x scales| + 1 bf16 ulp."""
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


def run(ql, c, K, bn=128, bk=128):
    x = to_bf16_tensor(c["x"])
    w = torch.from_numpy(c["w"]).cuda()
    s = torch.from_numpy(c["s"]).cuda()
    y, _, _, path = ql.qlinear_fp8_block(x, w, s, K=K, block_n=bn, block_k=bk, debug=True)
    torch.cuda.synchronize()
    assert path == "fp8_skinny"
    return bits_of(y)


def compare(c, y, K, rows=None, bn=128, bk=128):
    ref, a = Q.fp8_block(F.bf16_to_f64(c["x"]), c["w"], c["s"], K, bn, bk, rows=rows)
    sl = slice(None) if rows is None else rows
    check_float(y[:, sl], ref, a)


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (4, 200, 640), (16, 384, 1024), (9, 1000, 2048),
                                   (3, 130, 17408), (2, 64, 128)])
def test_fp8_small(ql, M, N, K):
    c = synth.fp8_block_case(M, N, K, seed=M * 7 + N)
    compare(c, run(ql, c, K), K)


def test_fp8_padded_rows_nan_padding(ql):
    # rows padded to K + 256 with NaN codes: the kernel must never read past K
    c = synth.fp8_block_case(5, 256, 1024, seed=21, ldw=1024 + 256)
    compare(c, run(ql, c, 1024), 1024)


def test_fp8_other_block_sizes_and_tails(ql):
    c = synth.fp8_block_case(6, 100, 448, seed=22, block_n=32, block_k=64)
    compare(c, run(ql, c, 448, 32, 64), 448, bn=32, bk=64)


@pytest.mark.parametrize("M,N,K,bn,bk", [(3, 150, 576, 48, 192), (12, 300, 1120, 128, 320)])
def test_fp8_block_k_not_power_of_two(ql, M, N, K, bn, bk):
    # block sizes the persistent kernel does not index by shift take the register kernel
    c = synth.fp8_block_case(M, N, K, seed=24 + M, block_n=bn, block_k=bk)
    compare(c, run(ql, c, K, bn, bk), K, bn=bn, bk=bk)


def test_fp8_large_activations_no_overflow(ql):
    c = synth.fp8_block_case(2, 128, 256, seed=23)
    c["x"][0] = synth.f32_to_bf16_bits((np.linspace(-1, 1, 256) * 3e6).astype(np.float32))
    c["x"][1] = synth.f32_to_bf16_bits((np.linspace(-1, 1, 256) * 1e-6).astype(np.float32))
    compare(c, run(ql, c, 256), 256)


def test_fp8_many_tokens_chunked(ql):
    c = synth.fp8_block_case(33, 256, 512, seed=24)
    compare(c, run(ql, c, 512), 512)


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_fp8_full_size_sampled(ql, N, K, M):
    c = synth.fp8_block_case(M, N, K, seed=0)
    rows = sample_rows(N, seed=M)
    compare(c, run(ql, c, K), K, rows=rows)


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
@pytest.mark.parametrize("M", [1, 4])
def test_fp8_full_size_every_row(ql, N, K, M):
    # 1 token: local activation images where they fit; 4 tokens: the shared image
    c = synth.fp8_block_case(M, N, K, seed=100 + M)
    compare(c, run(ql, c, K), K)


def test_workspace_reuse_across_shapes(ql):
    """A small-N call with split-K partials, then a large-N call on the same workspace: every
    row of the second call must be right (the split-K tickets must not be disturbed)."""
    c1 = synth.fp8_block_case(4, 1024, 5120, seed=25)
    run(ql, c1, 5120)
    c2 = synth.fp8_block_case(4, 17408, 1024, seed=26)
    compare(c2, run(ql, c2, 1024), 1024)
