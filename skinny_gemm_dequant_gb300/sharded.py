"""Tensor-parallel (sharded) forms of the quantized linear layers.

The pages run these layers split over 2, 4 or 8 GPUs ([Z100] chapter 一 §5, communication and
parallelism under TP = 2/4/8; [DSV4] §0, TP = 4/8).  Two splits, one process per GPU:

* column-parallel (split N): each rank holds a block of output rows of W (with their scales and
  bias) and the whole x; every rank's output columns are exactly the unsharded layer's, and an
  all-gather concatenates them.  FP8 block scales are per block_n rows, so shard boundaries fall
  on whole blocks; INT8, FP8-channel, BF16 and MXFP4 scales are per row, any boundary works.
* row-parallel (split K): each rank holds a K range of W and of x.
    - INT8: the per-token activation scale is max|x| / 127 over the WHOLE row, so the ranks
      first all-reduce (MAX) their K range's amax; quantised with that amax, each rank's codes
      are exactly the unsharded codes.  Each rank's int32 sums are exact, an all-reduce (SUM)
      adds them exactly, and one epilogue kernel applies (acc * x_s) * w_s (+ bias): the result
      equals the unsharded layer's, bit for bit.
    - FP8 block (bf16 activations) and MXFP4: each rank's fp32 partial sums (no rounding, no
      bias), an all-reduce (SUM), then one bf16 rounding and the bias.  Boundaries: whole
      block_k ranges (FP8), whole 256-K units (MXFP4: the persistent kernel's unit, which also
      keeps the per-32 scale rows whole).

The compute steps go through the library's kernels (``LibraryOps``) and the collectives
through ``torch.distributed``; an ``ops`` object with the same methods can stand in for both
(the CPU tests use the oracle and gloo ranks).
"""
from __future__ import annotations

import torch


def shard_range(n: int, world: int, rank: int, align: int = 1):
    """[lo, hi) of rank's share of range(n): contiguous, in rank order, covering range(n), every
    boundary a multiple of ``align`` (the last share takes the ragged end)."""
    if world < 1 or not 0 <= rank < world or align < 1:
        raise ValueError("shard_range: need world >= 1, 0 <= rank < world, align >= 1")
    units = -(-n // align)
    lo = min(n, align * (units * rank // world))
    hi = min(n, align * (units * (rank + 1) // world))
    return lo, hi


# alignment of the K boundaries of a row-parallel shard, per format
K_ALIGN = {"int8": 16, "fp8_block": 128, "mxfp4": 256}
# alignment of the N boundaries of a column-parallel shard, per format
N_ALIGN = {"int8": 1, "fp8_block": 128, "mxfp4": 1, "fp8": 1, "bf16": 1}


class LibraryOps:
    """Compute steps through libqlinear's kernels, collectives through torch.distributed on
    ``group`` (None: the default group; a single process without a group reduces nothing)."""

    def __init__(self, group=None):
        self.group = group

    # ---------------------------------------------------------------- collectives
    def _dist(self):
        import torch.distributed as dist
        return dist if dist.is_available() and dist.is_initialized() else None

    def all_reduce(self, t, op):
        dist = self._dist()
        if dist is None:
            return t
        dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM, group=self.group)
        return t

    def all_gather_cols(self, y):
        """Concatenate every rank's [M, n_r] block along the columns (shares may differ)."""
        dist = self._dist()
        if dist is None:
            return y
        world = dist.get_world_size(self.group)
        widths = [torch.zeros(1, dtype=torch.int64, device=y.device) for _ in range(world)]
        dist.all_gather(widths, torch.tensor([y.shape[1]], dtype=torch.int64, device=y.device), group=self.group)
        wmax = int(max(int(w.item()) for w in widths))
        pad = torch.zeros(y.shape[0], wmax, dtype=y.dtype, device=y.device)
        pad[:, : y.shape[1]] = y
        raw = pad.view(torch.uint8)  # bytes: every backend moves them (gloo has no 16-bit types)
        parts = [torch.empty_like(raw) for _ in range(world)]
        dist.all_gather(parts, raw, group=self.group)
        return torch.cat([p.view(y.dtype)[:, : int(w.item())] for p, w in zip(parts, widths)], dim=1)

    # ---------------------------------------------------------------- compute
    @staticmethod
    def _ql():
        import skinny_gemm_dequant_gb300 as ql
        return ql

    def int8(self, x, w, w_scale, bias=None):
        return self._ql().qlinear_int8_w8a8(x, w, w_scale, bias)

    def fp8_block(self, x, w, w_scale, bias=None, block_n=128, block_k=128):
        return self._ql().qlinear_fp8_block(x, w, w_scale, block_n=block_n, block_k=block_k, bias=bias)

    def mxfp4(self, x, w, w_scale, bias=None):
        return self._ql().qlinear_mxfp4(x, w, w_scale, bias=bias)

    def token_amax(self, x):
        return self._ql().token_amax(x)

    def int8_partial(self, x, w, amax):
        return self._ql().qlinear_int8_w8a8_partial(x, w, amax)

    def int8_epilogue(self, acc, amax, w_scale, bias=None):
        return self._ql().qlinear_int8_epilogue(acc, amax, w_scale, bias)

    def fp8_block_partial(self, x, w, w_scale, block_n=128, block_k=128):
        return self._ql().qlinear_fp8_block_partial(x, w, w_scale, block_n=block_n, block_k=block_k)

    def mxfp4_partial(self, x, w, w_scale):
        return self._ql().qlinear_mxfp4_partial(x, w, w_scale)

    def finish_f32(self, y32, bias=None):
        return self._ql().finish_f32(y32, bias)


# -------------------------------------------------------------------- column-parallel
def int8_column_parallel(x, w_shard, w_scale_shard, bias_shard=None, *, ops=None, gather=True):
    """This rank's output rows of an INT8 layer (whole x), gathered into [M, N] if asked."""
    ops = ops or LibraryOps()
    y = ops.int8(x, w_shard, w_scale_shard, bias_shard)
    return ops.all_gather_cols(y) if gather else y


def fp8_block_column_parallel(x, w_shard, s_shard, bias_shard=None, *, block_n=128, block_k=128, ops=None,
                              gather=True):
    """This rank's output rows of an FP8-block layer; shard boundaries on whole block_n rows."""
    ops = ops or LibraryOps()
    y = ops.fp8_block(x, w_shard, s_shard, bias_shard, block_n, block_k)
    return ops.all_gather_cols(y) if gather else y


def mxfp4_column_parallel(x, w_shard, s_shard, bias_shard=None, *, ops=None, gather=True):
    ops = ops or LibraryOps()
    y = ops.mxfp4(x, w_shard, s_shard, bias_shard)
    return ops.all_gather_cols(y) if gather else y


# -------------------------------------------------------------------- row-parallel
def int8_row_parallel(x_shard, w_shard, w_scale, bias=None, *, ops=None):
    """An INT8 layer whose K is split over the ranks: amax all-reduce (MAX), exact int32 partial
    sums, all-reduce (SUM), one epilogue.  Returns the whole y [M, N] on every rank."""
    ops = ops or LibraryOps()
    amax = ops.all_reduce(ops.token_amax(x_shard), "max")
    acc = ops.all_reduce(ops.int8_partial(x_shard, w_shard, amax), "sum")
    return ops.int8_epilogue(acc, amax, w_scale, bias)


def fp8_block_row_parallel(x_shard, w_shard, s_shard, bias=None, *, block_n=128, block_k=128, ops=None):
    """An FP8-block layer whose K is split over the ranks (whole block_k ranges): fp32 partial
    sums, all-reduce (SUM), one bf16 rounding, then the bias."""
    ops = ops or LibraryOps()
    y32 = ops.all_reduce(ops.fp8_block_partial(x_shard, w_shard, s_shard, block_n, block_k), "sum")
    return ops.finish_f32(y32, bias)


def mxfp4_row_parallel(x_shard, w_shard, s_shard, bias=None, *, ops=None):
    """An MXFP4 layer whose K is split over the ranks (whole 256-K units)."""
    ops = ops or LibraryOps()
    y32 = ops.all_reduce(ops.mxfp4_partial(x_shard, w_shard, s_shard), "sum")
    return ops.finish_f32(y32, bias)


# -------------------------------------------------------------------- shard preparation
def int8_row_shard(x, w, world, rank):
    """(x[:, k0:k1], w[:, k0:k1]) views of rank's K range (16-aligned)."""
    k0, k1 = shard_range(x.shape[1], world, rank, K_ALIGN["int8"])
    return x[:, k0:k1], w[:, k0:k1]


def fp8_block_row_shard(x, w, s, world, rank, block_k=128):
    """x and w views of rank's K range (whole block_k ranges) and its block-scale columns, made
    contiguous (the library reads the scale grid row-major with ceil(K/block_k) columns)."""
    k0, k1 = shard_range(x.shape[1], world, rank, block_k)
    sk = s[:, k0 // block_k:-(-k1 // block_k)]
    return x[:, k0:k1], w[:, k0:k1], (sk.contiguous() if hasattr(sk, "contiguous") else sk.copy())


def mxfp4_row_shard(x, w, s, world, rank):
    """x, packed w (two codes per byte) and per-32 scale views of rank's K range (whole 256-K
    units: 128 weight bytes and 8 scale bytes per row per unit)."""
    k0, k1 = shard_range(x.shape[1], world, rank, K_ALIGN["mxfp4"])
    return x[:, k0:k1], w[:, k0 // 2:k1 // 2], s[:, k0 // 32:k1 // 32]


def column_shard(n, world, rank, fmt="int8", block_n=128):
    """[n0, n1) of rank's output rows (FP8 block: whole block_n rows)."""
    return shard_range(n, world, rank, block_n if fmt == "fp8_block" else N_ALIGN.get(fmt, 1))
