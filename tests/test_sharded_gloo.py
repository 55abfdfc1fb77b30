"""Sharded (tensor-parallel) linear layers on two gloo ranks on CPU.

Each rank's compute step is the oracle (no GPU here); the split, the boundaries and the
collectives are the library's own host logic (skinny_gemm_dequant_gb300.sharded) running over
real torch.distributed gloo collectives:
  * column-parallel: the gathered outputs equal the unsharded oracle's, bit for bit;
  * row-parallel INT8: the all-reduced amax gives every shard the unsharded codes, the int32
    sums add exactly, and y equals the unsharded oracle's bit for bit;
  * row-parallel FP8 block and MXFP4: fp64 partial sums added over the ranks, one rounding,
    within the float bar of the unsharded oracle."""
import os
import socket

import numpy as np
import pytest
import torch

import synth
from _util import ensure_built
from oracle import formats as F
from oracle import qlinear_oracle as Q

WORLD = 2


def _bits_t(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


def _np_bits(t):
    return t.numpy().view(np.uint16)


class OracleOps:
    """The sharded layer's steps on one CPU rank: compute by the oracle, collectives by gloo."""

    def __init__(self, group=None):
        self.group = group

    def all_reduce(self, t, op):
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM, group=self.group)
        return t

    def all_gather_cols(self, y_bits):
        from skinny_gemm_dequant_gb300.sharded import LibraryOps
        return _np_bits(LibraryOps(self.group).all_gather_cols(_bits_t(y_bits)))

    def int8(self, x, w, w_s, bias=None):
        return Q.int8_w8a8(x, w, w_s, bias)["y"]

    def token_amax(self, x):
        return torch.from_numpy(np.max(np.abs(F.bf16_to_f32(x)), axis=1).astype(np.float32))

    def int8_partial(self, x, w, amax):
        xq, _ = Q.quant_int8_per_token(x, amax.numpy())
        self.last_codes = xq
        return torch.from_numpy(Q.int8_accumulate(xq, w))

    def int8_epilogue(self, acc, amax, w_s, bias=None):
        xs = (amax.numpy().astype(np.float32) / np.float32(127.0)).astype(np.float32)
        return Q.int8_epilogue(acc.numpy(), xs, w_s, bias)

    def fp8_block(self, x, w, s, bias=None, block_n=128, block_k=128):
        y, _ = Q.fp8_block(F.bf16_to_f64(x), w, s, x.shape[1], block_n, block_k)
        return self.finish_f32(torch.from_numpy(y), bias)

    def fp8_block_partial(self, x, w, s, block_n=128, block_k=128):
        y, _ = Q.fp8_block(F.bf16_to_f64(x), w, s, x.shape[1], block_n, block_k)
        return torch.from_numpy(y)

    def mxfp4(self, x, w, s, bias=None):
        return self.finish_f32(self.mxfp4_partial(x, w, s), bias)

    def mxfp4_partial(self, x, w, s):
        return torch.from_numpy(F.bf16_to_f64(x) @ Q.mxfp4_dequant(w, s).T)

    def finish_f32(self, y, bias=None):
        yb = F.round_to_bf16(y.numpy())
        if bias is not None:
            yb = F.round_to_bf16(F.bf16_to_f64(yb) + F.bf16_to_f64(bias)[None, :])
        return yb


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port):
    import torch.distributed as dist
    from skinny_gemm_dequant_gb300 import sharded as S
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ops = OracleOps()
        # INT8 column-parallel: N = 300 split 150 / 150 (any row boundary), with bias
        c = synth.int8_case(3, 300, 512, seed=61)
        bias = synth.bf16_normal(synth.rng(61, 9), (300,))
        n0, n1 = S.column_shard(300, world, rank, "int8")
        y = S.int8_column_parallel(c["x"], c["w"][n0:n1], c["w_s"][n0:n1], bias[n0:n1], ops=ops)
        assert np.array_equal(y, Q.int8_w8a8(c["x"], c["w"], c["w_s"], bias)["y"])

        # INT8 row-parallel: K = 1040 split 512 / 528; token 1's amax lies in rank 1's range and
        # token 2's in rank 0's, so a shard's own amax would give other codes
        c = synth.int8_case(3, 200, 1040, seed=62)
        xf = F.bf16_to_f32(c["x"]).copy()
        xf[1, 1000] = 9.0
        xf[2, 3] = -7.5
        c["x"] = synth.f32_to_bf16_bits(xf)
        bias = synth.bf16_normal(synth.rng(62, 9), (200,))
        xs_, ws_ = S.int8_row_shard(c["x"], c["w"], world, rank)
        y = S.int8_row_parallel(xs_, ws_, c["w_s"], bias, ops=ops)
        ref = Q.int8_w8a8(c["x"], c["w"], c["w_s"], bias)
        k0, k1 = S.shard_range(1040, world, rank, S.K_ALIGN["int8"])
        assert (k0, k1) == ((0, 512), (512, 1040))[rank]
        assert np.array_equal(ops.last_codes, ref["x_q"][:, k0:k1])
        assert np.array_equal(y, ref["y"])

        # FP8 block: row-parallel over K = 640 (5 blocks: 384 / 256) and column-parallel over
        # N = 384 (3 blocks: 256 / 128), with bias
        c = synth.fp8_block_case(2, 384, 640, seed=63)
        bias = synth.bf16_normal(synth.rng(63, 9), (384,))
        ref, a = Q.fp8_block(F.bf16_to_f64(c["x"]), c["w"], c["s"], 640)
        yref = F.bf16_to_f64(F.round_to_bf16(F.bf16_to_f64(F.round_to_bf16(ref)) + F.bf16_to_f64(bias)[None, :]))
        xs_, ws_, ss_ = S.fp8_block_row_shard(c["x"], c["w"], c["s"], world, rank)
        y = S.fp8_block_row_parallel(xs_, ws_, ss_, bias, ops=ops)
        tol = 1e-3 * a + 2 * F.bf16_ulp(yref) + 1e-300
        assert np.all(np.abs(F.bf16_to_f64(y) - yref) <= tol)
        n0, n1 = S.column_shard(384, world, rank, "fp8_block")
        assert n0 % 128 == 0 and (n1 % 128 == 0 or n1 == 384)
        y = S.fp8_block_column_parallel(c["x"], c["w"][n0:n1], c["s"][n0 // 128:-(-n1 // 128)], bias[n0:n1],
                                        ops=ops)
        y1 = ops.fp8_block(c["x"], c["w"], c["s"], bias)
        assert np.array_equal(y, y1)

        # MXFP4 row-parallel: K = 1024 (four 256-K units: 512 / 512)
        c = synth.mxfp4_dense_case(2, 96, 1024, seed=64)
        xs_, ws_, ss_ = S.mxfp4_row_shard(c["x"], c["w"], c["s"], world, rank)
        y = S.mxfp4_row_parallel(xs_, ws_, ss_, ops=ops)
        wd = Q.mxfp4_dequant(c["w"], c["s"])
        xv = F.bf16_to_f64(c["x"])
        ref, a = xv @ wd.T, np.abs(xv) @ np.abs(wd).T
        assert np.all(np.abs(F.bf16_to_f64(y) - ref) <= 1e-3 * a + F.bf16_ulp(ref))
    finally:
        dist.destroy_process_group()


def test_shard_ranges_cover_and_align():
    ensure_built()
    from skinny_gemm_dequant_gb300 import sharded as S
    for n, world, align in [(1040, 2, 16), (640, 2, 128), (640, 3, 128), (5120, 8, 256), (7, 4, 1), (0, 2, 16)]:
        ranges = [S.shard_range(n, world, r, align) for r in range(world)]
        assert ranges[0][0] == 0 and ranges[-1][1] == n
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
        assert all(lo % align == 0 and (hi % align == 0 or hi == n) for lo, hi in ranges)


def test_sharded_layers_on_two_gloo_ranks():
    ensure_built()
    import torch.multiprocessing as mp
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    mp.spawn(_rank_main, args=(WORLD, _free_port()), nprocs=WORLD, join=True)


def test_planted_local_amax_breaks_row_parallel_int8():
    """Negative control: quantising a K shard with its own amax (no all-reduce) gives codes
    that differ from the unsharded layer's, so the exactness check above has teeth."""
    c = synth.int8_case(2, 64, 1024, seed=65)
    xf = F.bf16_to_f32(c["x"]).copy()
    xf[0, 900] = 11.0
    c["x"] = synth.f32_to_bf16_bits(xf)
    ref = Q.int8_w8a8(c["x"], c["w"], c["w_s"])
    local, _ = Q.quant_int8_per_token(c["x"][:, :512])
    assert not np.array_equal(local, ref["x_q"][:, :512])
