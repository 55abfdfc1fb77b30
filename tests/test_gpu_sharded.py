"""Sharded layers through the library on one GPU: both shards of a split run one after the
other and the collective step is done in the test (max / sum over the two shards' results).
Column-parallel outputs and row-parallel INT8 outputs must equal the unsharded call's bit for
bit (INT8 accumulators also the oracle's); row-parallel FP8 block and MXFP4 outputs must meet
the float bar against the oracle."""
import numpy as np
import pytest
import torch

import synth
from _util import bits_of, check_float, gpu_lib, sample_rows, to_bf16_tensor
from oracle import formats as F
from oracle import qlinear_oracle as Q

pytestmark = pytest.mark.gpu
WORLD = 2


@pytest.fixture(scope="module")
def ql():
    return gpu_lib()


@pytest.mark.parametrize("M,N,K", [(1, 1000, 4096), (4, 640, 1040), (9, 300, 2048), (40, 512, 2048),
                                   (4, 17408, 5120)])
def test_int8_row_parallel_is_bit_exact(ql, M, N, K):
    from skinny_gemm_dequant_gb300 import sharded as S
    c = synth.int8_case(M, N, K, seed=70 + M)
    xf = F.bf16_to_f32(c["x"]).copy()
    xf[0, K - 5] = 13.0  # token 0's amax in the last shard
    c["x"] = synth.f32_to_bf16_bits(xf)
    bias = synth.bf16_normal(synth.rng(70, M), (N,))
    x, w = to_bf16_tensor(c["x"]), torch.from_numpy(c["w"]).cuda()
    ws, b = torch.from_numpy(c["w_s"]).cuda(), to_bf16_tensor(bias)
    shards = [S.int8_row_shard(x, w, WORLD, r) for r in range(WORLD)]
    amax = torch.stack([ql.token_amax(xs) for xs, _ in shards]).amax(0)          # all-reduce MAX
    parts = [ql.qlinear_int8_w8a8_partial(xs, wsh, amax, debug=True) for xs, wsh in shards]
    acc = sum(p[0] for p in parts)                                                 # all-reduce SUM
    y = ql.qlinear_int8_epilogue(acc, amax, ws, b)
    y1, acc1, xq1, _, _ = ql.qlinear_int8_w8a8(x, w, ws, b, debug=True)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([p[1] for p in parts], dim=1), xq1)              # the unsharded codes
    assert torch.equal(acc, acc1) and torch.equal(y.view(torch.int16), y1.view(torch.int16))
    rows = sample_rows(N, seed=M) if N > 4096 else None
    ref = Q.int8_w8a8(c["x"], c["w"], c["w_s"], bias, rows=rows)
    sl = slice(None) if rows is None else rows
    assert np.array_equal(acc.cpu().numpy()[:, sl], ref["acc"])


@pytest.mark.parametrize("M,N,K", [(1, 384, 1024), (4, 256, 640), (16, 17408, 5120)])
def test_fp8_block_row_parallel(ql, M, N, K):
    from skinny_gemm_dequant_gb300 import sharded as S
    c = synth.fp8_block_case(M, N, K, seed=80 + M)
    x, w, s = to_bf16_tensor(c["x"]), torch.from_numpy(c["w"]).cuda(), torch.from_numpy(c["s"]).cuda()
    y32 = sum(ql.qlinear_fp8_block_partial(*S.fp8_block_row_shard(x, w, s, WORLD, r)) for r in range(WORLD))
    y = bits_of(ql.finish_f32(y32))
    rows = sample_rows(N, seed=M) if N > 4096 else None
    ref, a = Q.fp8_block(F.bf16_to_f64(c["x"]), c["w"], c["s"], K, rows=rows)
    check_float(y if rows is None else y[:, rows], ref, a)


@pytest.mark.parametrize("M,N,K", [(1, 96, 1024), (5, 300, 2048)])
def test_mxfp4_row_parallel(ql, M, N, K):
    from skinny_gemm_dequant_gb300 import sharded as S
    c = synth.mxfp4_dense_case(M, N, K, seed=90 + M)
    x, w, s = to_bf16_tensor(c["x"]), torch.from_numpy(c["w"]).cuda(), torch.from_numpy(c["s"]).cuda()
    bias = synth.bf16_normal(synth.rng(90, M), (N,))
    y32 = sum(ql.qlinear_mxfp4_partial(*S.mxfp4_row_shard(x, w, s, WORLD, r)) for r in range(WORLD))
    y = bits_of(ql.finish_f32(y32, to_bf16_tensor(bias)))
    wd = Q.mxfp4_dequant(c["w"], c["s"])
    xv = F.bf16_to_f64(c["x"])
    ref = F.bf16_to_f64(F.round_to_bf16(F.bf16_to_f64(F.round_to_bf16(xv @ wd.T)) + F.bf16_to_f64(bias)[None, :]))
    check_float(y, ref, np.abs(xv) @ np.abs(wd).T + 2 * F.bf16_ulp(ref) / 1e-3)


def test_column_parallel_concatenation_is_bit_exact(ql):
    from skinny_gemm_dequant_gb300 import sharded as S
    c = synth.int8_case(4, 1000, 2048, seed=95)
    x, w, ws = to_bf16_tensor(c["x"]), torch.from_numpy(c["w"]).cuda(), torch.from_numpy(c["w_s"]).cuda()
    parts = []
    for r in range(WORLD):
        n0, n1 = S.column_shard(1000, WORLD, r, "int8")
        parts.append(ql.qlinear_int8_w8a8(x, w[n0:n1], ws[n0:n1]))
    assert torch.equal(torch.cat(parts, 1).view(torch.int16), ql.qlinear_int8_w8a8(x, w, ws).view(torch.int16))
    f = synth.fp8_block_case(4, 640, 1024, seed=96)
    x, w, s = to_bf16_tensor(f["x"]), torch.from_numpy(f["w"]).cuda(), torch.from_numpy(f["s"]).cuda()
    parts = []
    for r in range(WORLD):
        n0, n1 = S.column_shard(640, WORLD, r, "fp8_block")
        parts.append(ql.qlinear_fp8_block(x, w[n0:n1], s[n0 // 128:-(-n1 // 128)]))
    assert torch.equal(torch.cat(parts, 1).view(torch.int16), ql.qlinear_fp8_block(x, w, s).view(torch.int16))


def test_partial_entry_points_reject_unsupported_shapes(ql):
    x = torch.zeros(1, 384, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(64, 192, dtype=torch.uint8, device="cuda")
    s = torch.zeros(64, 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ql.QLError):  # MXFP4 partial sums need whole 256-K units
        ql.qlinear_mxfp4_partial(x, w, s)
    w8 = torch.zeros(64, 384, dtype=torch.uint8, device="cuda")
    s8 = torch.zeros(1, 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(ql.QLError):  # block_k must be a power of two for the partial path
        ql.qlinear_fp8_block_partial(x, w8, s8, block_k=192)
