"""INT8 W8A8 parity: CUDA path vs the oracle on identical seeded inputs.
Bit-exact: x_q, x_s, int32 accumulators.  y within 1e-3*sum|w x| + 1 bf16 ulp."""
import numpy as np
import pytest
import torch

import synth
from _util import bits_of, check_float, gpu_lib, sample_rows, to_bf16_tensor
from oracle import qlinear_oracle as Q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ql():
    return gpu_lib()


def run(ql, c, bias=None, wsl=None):
    x = to_bf16_tensor(c["x"])
    w = torch.from_numpy(c["w"]).cuda()
    ws = torch.from_numpy(c["w_s"] if wsl is None else c["w_s"][:wsl]).cuda()
    b = None if bias is None else to_bf16_tensor(bias)
    y, acc, xq, xs, path = ql.qlinear_int8_w8a8(x, w, ws, b, debug=True)
    torch.cuda.synchronize()
    # up to 32 tokens: the persistent skinny kernel; more: the tcgen05 GEMM
    assert path == ("int8_skinny" if c["x"].shape[0] <= 32 else "int8_tcgen05")
    return bits_of(y), acc.cpu().numpy(), xq.cpu().numpy(), xs.cpu().numpy()


def compare(c, got, rows=None, bias=None, wsl=None):
    y, acc, xq, xs = got
    K = c["x"].shape[1]
    ref = Q.int8_w8a8(c["x"], c["w"][:, :K], c["w_s"] if wsl is None else c["w_s"][:wsl], bias, rows=rows)
    assert np.array_equal(xq, ref["x_q"]), "x_q differs"
    assert np.array_equal(xs.view(np.uint32), ref["x_s"].view(np.uint32)), "x_s differs"
    sl = slice(None) if rows is None else rows
    assert np.array_equal(acc[:, sl], ref["acc"]), "int32 accumulators differ"
    y_ref = ref["y"]
    from oracle import formats as F
    check_float(y[:, sl], F.bf16_to_f64(y_ref), ref["abs_sum"] + 0.0)


@pytest.mark.parametrize("M,N,K", [(1, 512, 1024), (3, 200, 304), (16, 1000, 2048), (9, 130, 4096),
                                   (5, 77, 16), (8, 64, 17408), (2, 4097, 640)])
def test_int8_small(ql, M, N, K):
    c = synth.int8_case(M, N, K, seed=M + N)
    compare(c, run(ql, c))


@pytest.mark.parametrize("M,N,K", [(2, 3000, 1008), (7, 3000, 1008), (8, 5000, 2192), (4, 9000, 2000)])
def test_int8_local_image_multi_token(ql, M, N, K):
    # M * K <= 18432: every CTA builds its own image of 2..8 tokens in one pass over the rows,
    # K ragged against the 256-K unit (zero tails in the last unit's slots)
    c = synth.int8_case(M, N, K, seed=M * 7 + K)
    compare(c, run(ql, c))


def test_int8_many_tokens_chunked(ql):
    c = synth.int8_case(37, 96, 512, seed=3)
    compare(c, run(ql, c))


def test_int8_bias_per_tensor_scale_padded_rows(ql):
    c = synth.int8_case(4, 150, 256, seed=11, ldw=320)
    bias = synth.bf16_normal(synth.rng(11, 99), (150,))
    compare(c, run(ql, c, bias=bias, wsl=1), bias=bias, wsl=1)


def test_int8_zero_token_and_large_values(ql):
    c = synth.int8_case(3, 128, 256, seed=12)
    c["x"][1] = 0
    c["x"][2] = synth.f32_to_bf16_bits(np.linspace(-3e4, 3e4, 256).astype(np.float32))
    got = run(ql, c)
    assert got[3][1] == 0 and not got[2][1].any() and not got[0][1].any()
    compare(c, got)


def test_int8_repeat_is_deterministic(ql):
    c = synth.int8_case(16, 5120, 17408 // 4, seed=13)
    a = run(ql, c)
    b = run(ql, c)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408), (10240, 5120)])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_int8_full_size_sampled(ql, N, K, M):
    c = synth.int8_case(M, N, K, seed=0)
    rows = sample_rows(N, seed=M)
    compare(c, run(ql, c), rows=rows)


@pytest.mark.parametrize("M,N,K", [(17, 300, 2048), (24, 1000, 4096), (32, 130, 17408), (31, 4097, 640)])
def test_int8_skinny_up_to_32_tokens(ql, M, N, K):
    # 17..32 tokens: the persistent kernel with four 8-token MMA tiles
    c = synth.int8_case(M, N, K, seed=M * 3 + N)
    compare(c, run(ql, c))


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408), (10240, 5120)])
@pytest.mark.parametrize("M", [1, 2, 4, 16, 32])
def test_int8_full_size_every_row(ql, N, K, M):
    # every output row against the oracle, for each way the activations reach the CTAs: local
    # images (1 token, 2 tokens at K = 5120), the shared image with cells (2 tokens at K = 17408,
    # 4 tokens), partial slots (16 tokens) and four MMA tiles (32 tokens); a row block's units
    # may be split between CTAs differently per shape
    c = synth.int8_case(M, N, K, seed=100 + M)
    compare(c, run(ql, c))


def _tie_tokens(K):
    """Three tokens whose quotients x / x_s land exactly on half-integers: x_s = 1 (amax 127),
    2 (amax 254) and 0.5 (amax 63.5), with x = x_s * (k + 1/2) in both signs."""
    rows = []
    for xs, amax in ((1.0, 127.0), (2.0, 254.0), (0.5, 63.5)):
        half = np.arange(K - 1) % 127 + 0.5          # 0.5, 1.5, ..., 126.5
        sign = np.where(np.arange(K - 1) % 2 == 0, 1.0, -1.0)
        rows.append(np.concatenate([[amax], sign * half * xs]))
    return synth.f32_to_bf16_bits(np.array(rows, np.float32))


def test_int8_quantisation_ties_round_half_even(ql):
    # the kernel's reciprocal product is exact here, so every code comes from the IEEE-quotient
    # branch: rint must round each .5 to the even neighbour, as the oracle's does
    K = 512
    c = synth.int8_case(3, 256, K, seed=31)
    c["x"] = _tie_tokens(K)
    got = run(ql, c)
    xq_ref, xs_ref = Q.quant_int8_per_token(c["x"])
    assert xs_ref.tolist() == [1.0, 2.0, 0.5]
    assert np.array_equal(got[2], xq_ref) and np.array_equal(got[3], xs_ref)
    assert np.all(np.abs(xq_ref[:, 1:]) % 2 == 0)  # every tie went to an even code
    compare(c, got)


# ------------------------------------------------------------------ M > 16: the tcgen05 GEMM
@pytest.mark.parametrize("M,N,K", [(17, 128, 256), (33, 200, 320), (64, 256, 1024), (100, 300, 640),
                                   (128, 130, 2048), (129, 64, 512), (200, 384, 1088), (256, 512, 4096)])
def test_int8_gemm_small_and_ragged(ql, M, N, K):
    c = synth.int8_case(M, N, K, seed=M + N + K)
    compare(c, run(ql, c))


def test_int8_gemm_bias_per_tensor_scale_padded_rows(ql):
    c = synth.int8_case(40, 150, 576, seed=21, ldw=640)
    bias = synth.bf16_normal(synth.rng(21, 99), (150,))
    compare(c, run(ql, c, bias=bias, wsl=1), bias=bias, wsl=1)


@pytest.mark.parametrize("sign", ["same", "mixed"])
def test_int8_gemm_drain_exactness_at_the_limit(ql, sign):
    # every code and weight at +-127: each 512-K group sums to 512 * 127^2 = 8,258,048 (just below
    # 2^23) and the whole K to 16384 * 127^2 = 264,257,536, exact only through the int32 drain
    M, N, K = 24, 130, 16384
    c = synth.int8_case(M, N, K, seed=22)
    c["x"][:] = synth.f32_to_bf16_bits(np.full((M, K), 2.0, np.float32))
    c["w"][:] = 127
    if sign == "mixed":
        c["x"][1::2, ::3] = synth.f32_to_bf16_bits(np.float32(-2.0))
        c["w"][::2, 1::2] = -127
    got = run(ql, c)
    assert got[1].max() == K * 127 * 127 or sign == "mixed"
    compare(c, got)


def test_int8_gemm_zero_token_and_large_values(ql):
    c = synth.int8_case(20, 128, 256, seed=23)
    c["x"][1] = 0
    c["x"][19] = synth.f32_to_bf16_bits(np.linspace(-3e4, 3e4, 256).astype(np.float32))
    got = run(ql, c)
    assert got[3][1] == 0 and not got[2][1].any() and not got[0][1].any()
    compare(c, got)


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408), (10240, 5120)])
@pytest.mark.parametrize("M", [32, 64, 256])
def test_int8_gemm_full_size_sampled(ql, N, K, M):
    c = synth.int8_case(M, N, K, seed=1)
    rows = sample_rows(N, seed=M)
    compare(c, run(ql, c), rows=rows)


@pytest.mark.parametrize("M,N,offset", [(64, 9736, 0), (100, 9736, 0), (64, 9736, 1), (64, 9732, 0), (64, 300, 0)])
def test_int8_gemm_output_pitch_and_alignment(ql, M, N, offset):
    # as the block-scaled GEMM: with 77 row blocks K is not split, so a padded-pitch aligned view
    # with N a multiple of 8 takes the TMA-store epilogue (ragged N and M clipped); an unaligned
    # view, an N ending inside a 16-byte chunk, or a split K (N = 300) the element stores; all
    # equal the dense output, nothing outside the view is written
    K = 640
    c = synth.int8_case(M, N, K, seed=78)
    x, w, s = to_bf16_tensor(c["x"]), torch.from_numpy(c["w"]).cuda(), torch.from_numpy(c["w_s"]).cuda()
    ref = ql.qlinear_int8_w8a8(x, w, s)
    big = torch.full((M + 3, N + 44), -7.0, dtype=torch.bfloat16, device="cuda")  # pitch 688 B
    out = big[:M, offset:offset + N]
    ql.qlinear_int8_w8a8(x, w, s, out=out)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(out.contiguous()), bits_of(ref))
    rest = big.clone()
    rest[:M, offset:offset + N] = -7.0
    bad = (rest != -7.0).nonzero().cpu().numpy()
    assert len(bad) == 0, f"the store wrote outside the output view: {len(bad)} elements, first {bad[:4].tolist()}"
