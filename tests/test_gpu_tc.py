"""tcgen05 block-scaled GEMM parity (1x128 E4M3 activations, FP8 128x128-block or MXFP4
weights): the activation codes and scales bit-exact, y within 1e-3*sum|a w scales| + 1 ulp."""
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


def run_fp8(ql, c, K):
    y, aq, as_, path = ql.qlinear_fp8_block(to_bf16_tensor(c["x"]), torch.from_numpy(c["w"]).cuda(),
                                            torch.from_numpy(c["s"]).cuda(), K=K, act_mode=ql.ACT_E4M3_1X128,
                                            debug=True)
    torch.cuda.synchronize()
    assert path == "fp8_tcgen05"
    return bits_of(y), aq.cpu().numpy(), as_.cpu().numpy()


def run_fp4(ql, c):
    y, aq, as_, path = ql.qlinear_mxfp4(to_bf16_tensor(c["x"]), torch.from_numpy(c["w"]).cuda(),
                                        torch.from_numpy(c["s"]).cuda(), act_mode=ql.ACT_E4M3_1X128, debug=True)
    torch.cuda.synchronize()
    assert path == "mxfp4_tcgen05"
    return bits_of(y), aq.cpu().numpy(), as_.cpu().numpy()


def pad_scales(c, K, mult=16):
    lds = -(-(K // 32) // mult) * mult
    sp = np.full((c["s"].shape[0], lds), 255, np.uint8)
    sp[:, : K // 32] = c["s"]
    return dict(c, s=sp), c["s"]


@pytest.mark.parametrize("M,N,K", [(64, 256, 512), (17, 128, 256), (100, 300, 640), (256, 384, 1024),
                                   (300, 256, 512), (128, 17408 // 16, 5120)])
def test_tc_fp8_small(ql, M, N, K):
    c = synth.fp8_block_case(M, N, K, seed=M + N)
    y, aq, as_ = run_fp8(ql, c, K)
    r = Q.fp8_block_act_quant(c["x"], c["w"], c["s"], K)
    assert np.array_equal(aq, r["q"]), "activation codes differ"
    assert np.array_equal(as_, r["s"]), "activation scales differ"
    check_float(y, r["y_f64"], r["abs_sum"])


@pytest.mark.parametrize("M,N,K", [(64, 256, 512), (17, 128, 256), (100, 300, 640), (256, 384, 1024),
                                   (300, 256, 512)])
def test_tc_mxfp4_small(ql, M, N, K):
    c0 = synth.mxfp4_dense_case(M, N, K, seed=M + N)
    c, s_raw = pad_scales(c0, K)
    y, aq, as_ = run_fp4(ql, c)
    r = Q.mxfp4_act_quant(c0["x"], c0["w"], s_raw)
    assert np.array_equal(aq, r["q"]) and np.array_equal(as_, r["s"])
    check_float(y, r["y_f64"], r["abs_sum"])


@pytest.mark.parametrize("M", [64, 128, 256])
def test_tc_fp8_full_size_sampled(ql, M):
    N, K = 17408, 5120
    c = synth.fp8_block_case(M, N, K, seed=0)
    y, aq, as_ = run_fp8(ql, c, K)
    rows = sample_rows(N, 32, seed=M)
    r = Q.fp8_block_act_quant(c["x"], c["w"], c["s"], K, rows=rows)
    assert np.array_equal(aq, r["q"]) and np.array_equal(as_, r["s"])
    check_float(y[:, rows], r["y_f64"], r["abs_sum"])


@pytest.mark.parametrize("M", [64, 128, 256])
def test_tc_mxfp4_full_size_sampled(ql, M):
    N, K = 17408, 5120
    c = synth.mxfp4_dense_case(M, N, K, seed=0)
    y, aq, as_ = run_fp4(ql, c)
    rows = sample_rows(N, 32, seed=M)
    r = Q.mxfp4_act_quant(c["x"], c["w"], c["s"], rows=rows)
    assert np.array_equal(aq, r["q"]) and np.array_equal(as_, r["s"])
    check_float(y[:, rows], r["y_f64"], r["abs_sum"])


# Long K: the scales of (256, 256, 32768) and of both MXFP4 cases do not fit the 48 KB
# shared-memory staging area, so the kernel reads them from global memory stage by stage;
# (64, 130, 40960) still stages them (320 stages of scales)
@pytest.mark.parametrize("M,N,K", [(256, 256, 32768), (64, 130, 40960)])
def test_tc_fp8_long_k(ql, M, N, K):
    c = synth.fp8_block_case(M, N, K, seed=7)
    y, aq, as_ = run_fp8(ql, c, K)
    r = Q.fp8_block_act_quant(c["x"], c["w"], c["s"], K)
    assert np.array_equal(aq, r["q"]) and np.array_equal(as_, r["s"])
    check_float(y, r["y_f64"], r["abs_sum"])


@pytest.mark.parametrize("M,N,K", [(64, 256, 32768), (200, 128, 16384)])
def test_tc_mxfp4_long_k(ql, M, N, K):
    c0 = synth.mxfp4_dense_case(M, N, K, seed=8)
    c, s_raw = pad_scales(c0, K)
    y, aq, as_ = run_fp4(ql, c)
    r = Q.mxfp4_act_quant(c0["x"], c0["w"], s_raw)
    assert np.array_equal(aq, r["q"]) and np.array_equal(as_, r["s"])
    check_float(y, r["y_f64"], r["abs_sum"])


@pytest.mark.parametrize("M,N,offset", [(64, 304, 0), (100, 304, 0), (100, 304, 1), (100, 300, 0)])
def test_tc_fp8_output_pitch_and_alignment(ql, M, N, offset):
    # y written into a wider buffer: a 16-byte aligned view with a padded row pitch and N a
    # multiple of 8 takes the TMA-store epilogue (ragged N and M clipped by the store), a view
    # one element off alignment or an N ending inside a 16-byte chunk the element stores; all
    # equal the dense output bit for bit and write nothing outside the view
    K = 640
    c = synth.fp8_block_case(M, N, K, seed=77)
    x, w, s = to_bf16_tensor(c["x"]), torch.from_numpy(c["w"]).cuda(), torch.from_numpy(c["s"]).cuda()
    ref = ql.qlinear_fp8_block(x, w, s, K=K, act_mode=ql.ACT_E4M3_1X128)
    big = torch.full((M + 3, N + 44), -7.0, dtype=torch.bfloat16, device="cuda")  # pitch 688 B
    out = big[:M, offset:offset + N]
    ql.qlinear_fp8_block(x, w, s, K=K, act_mode=ql.ACT_E4M3_1X128, out=out)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(out.contiguous()), bits_of(ref))
    rest = big.clone()
    rest[:M, offset:offset + N] = -7.0
    bad = (rest != -7.0).nonzero().cpu().numpy()
    assert len(bad) == 0, f"the store wrote outside the output view: {len(bad)} elements, first {bad[:4].tolist()}"
