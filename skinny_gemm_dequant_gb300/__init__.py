"""Python binding of libqlinear.so, the GB300 quantized decode linear layer.

Argument marshalling only: every function passes device pointers, sizes and the current CUDA
stream to the C ABI declared in ``include/qlinear.h``; all computation runs in the library's
CUDA kernels.  PyTorch is used for device memory (outputs, workspace) and streams.

The library must have been built (``python -m skinny_gemm_dequant_gb300._build`` or
``__graft_entry__.build()``); importing this package without it raises ``ImportError`` -
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB as _LIB_PATH

__all__ = [
    "lib", "QLError", "qlinear_int8_w8a8", "qlinear_fp8_block", "qlinear_mxfp4", "moe_mxfp4_grouped",
    "workspace_bytes", "Workspace", "read_device_status", "set_wait_limit",
    "OP_INT8_W8A8", "OP_FP8_BLOCK", "OP_MXFP4", "OP_MOE_MXFP4", "OP_BF16", "OP_FP8_CHANNEL", "qlinear_bf16",
    "qlinear_fp8", "FP8_E4M3", "FP8_E5M2", "ACT_BF16", "ACT_E4M3_1X128", "PATHS",
    "token_amax", "qlinear_int8_w8a8_partial", "qlinear_int8_epilogue", "qlinear_fp8_block_partial",
    "qlinear_mxfp4_partial", "finish_f32",
]

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libqlinear.so is not built ({_LIB_PATH}); run skinny_gemm_dequant_gb300._build.build()")

lib = ctypes.CDLL(_LIB_PATH)

_vp, _i64, _int, _u32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_size_t
_ip = ctypes.POINTER(ctypes.c_int)

lib.ql_status_string.restype = ctypes.c_char_p
lib.ql_status_string.argtypes = [_int]
lib.ql_version.restype = _int
lib.ql_workspace_bytes.restype = _sz
lib.ql_workspace_bytes.argtypes = [_int, _i64, _i64, _i64, _int, _int]
lib.ql_workspace_init.restype = _int
lib.ql_workspace_init.argtypes = [_vp, _sz, _vp]
lib.ql_read_device_status.restype = _int
lib.ql_read_device_status.argtypes = [_vp, _vp, _int, ctypes.POINTER(_u32)]
lib.ql_set_wait_limit.restype = None
lib.ql_set_wait_limit.argtypes = [_u32]
lib.qlinear_int8_w8a8.restype = _int
lib.qlinear_int8_w8a8.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _vp, _i64,
                                  _vp, _vp, _vp, _vp, _sz, _vp, _ip]
lib.qlinear_fp8_block.restype = _int
lib.qlinear_fp8_block.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _int, _int, _int, _vp, _vp,
                                  _i64, _vp, _vp, _vp, _sz, _vp, _ip]
lib.qlinear_bf16.restype = _int
lib.qlinear_bf16.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _sz, _vp,
                             ctypes.POINTER(_int)]
lib.qlinear_fp8.restype = _int
lib.qlinear_fp8.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _int, _vp, _i64, _vp, _vp, _i64, _vp, _sz,
                            _vp, _ip]
lib.qlinear_mxfp4.restype = _int
lib.qlinear_mxfp4.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _int, _vp, _vp, _i64,
                              _vp, _vp, _vp, _sz, _vp, _ip]
lib.moe_mxfp4_grouped.restype = _int
lib.moe_mxfp4_grouped.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp, _int, _int, _int, _vp, _vp, _vp, _vp, _i64,
                                  ctypes.c_float, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _ip]

lib.ql_token_amax.restype = _int
lib.ql_token_amax.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp]
lib.qlinear_int8_w8a8_partial.restype = _int
lib.qlinear_int8_w8a8_partial.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp, _ip]
lib.qlinear_int8_epilogue.restype = _int
lib.qlinear_int8_epilogue.argtypes = [_vp, _i64, _i64, _vp, _vp, _i64, _vp, _vp, _i64, _vp]
lib.qlinear_fp8_block_partial.restype = _int
lib.qlinear_fp8_block_partial.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _int, _int, _vp, _i64, _vp,
                                          _sz, _vp, _ip]
lib.qlinear_mxfp4_partial.restype = _int
lib.qlinear_mxfp4_partial.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _sz, _vp,
                                      _ip]
lib.ql_finish_f32.restype = _int
lib.ql_finish_f32.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _vp]

OP_INT8_W8A8, OP_FP8_BLOCK, OP_MXFP4, OP_MOE_MXFP4, OP_BF16, OP_FP8_CHANNEL = 1, 2, 3, 4, 5, 6
FP8_E4M3, FP8_E5M2 = 0, 1
ACT_BF16, ACT_E4M3_1X128 = 0, 1
PATHS = {0: "none", 1: "int8_skinny", 2: "fp8_skinny", 3: "fp8_tcgen05", 4: "mxfp4_skinny",
         5: "mxfp4_tcgen05", 6: "moe_mxfp4", 7: "bf16_skinny", 8: "fp8_channel_skinny",
         9: "int8_tcgen05", 10: "moe_mxfp4_tcgen05"}


class QLError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.ql_status_string(status).decode()} (status {status})")


def _check(status: int, where: str):
    if status != 0:
        raise QLError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def workspace_bytes(op: int, M: int, N: int, K: int, E: int = 0, topk: int = 0) -> int:
    return int(lib.ql_workspace_bytes(op, M, N, K, E, topk))


class Workspace:
    """Device scratch for the library calls; zeroed once when (re)allocated, as the C ABI
    requires.  Calls sharing one Workspace must be ordered (same stream)."""

    def __init__(self, device=None):
        self.device = torch.device(device if device is not None else "cuda")
        self.buf = None

    def get(self, nbytes: int, stream=None) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            _check(lib.ql_workspace_init(_ptr(self.buf), self.buf.numel(), _stream(stream)), "ql_workspace_init")
        return self.buf


_default_ws: dict = {}


def _ws(device, nbytes, stream, workspace):
    if workspace is None:
        # keyed by the stream's handle: a Python object's id can be reused once it is collected
        key = (torch.device(device).index, None if stream is None else int(stream.cuda_stream))
        workspace = _default_ws.setdefault(key, Workspace(device))
    return workspace.get(nbytes, stream)


def read_device_status(ws: torch.Tensor, clear: bool = True, stream=None):
    flags = _u32(0)
    st = lib.ql_read_device_status(_ptr(ws), _stream(stream), int(clear), ctypes.byref(flags))
    return st, int(flags.value)


def set_wait_limit(polls: int):
    lib.ql_set_wait_limit(int(polls))


def _bf16(t, name):
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
    return t


def qlinear_int8_w8a8(x, w, w_scale, bias=None, *, debug=False, out=None, workspace=None, stream=None):
    """y = bf16((acc * x_s) * w_s) (+ bias) with per-token dynamic INT8 activations.
    x: bf16 [M, K]; w: int8 [N, K] (row stride w.stride(0)); w_scale: fp32 [N] or [1].
    With debug=True returns (y, acc int32 [M,N], x_q int8 [M,K], x_s fp32 [M], path)."""
    _bf16(x, "x")
    M, K = x.shape
    N = w.shape[0]
    if w.dtype != torch.int8 or w.stride(1) != 1 or x.stride(1) != 1:
        raise TypeError("w must be int8 with unit inner stride; x must have unit inner stride")
    y = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    acc = xq = xs = None
    if debug:
        acc = torch.empty(M, N, dtype=torch.int32, device=x.device)
        xq = torch.empty(M, K, dtype=torch.int8, device=x.device)
        xs = torch.empty(M, dtype=torch.float32, device=x.device)
    nbytes = workspace_bytes(OP_INT8_W8A8, M, N, K)
    ws = _ws(x.device, nbytes, stream, workspace)
    path = ctypes.c_int(0)
    _check(lib.qlinear_int8_w8a8(_ptr(x), M, K, x.stride(0), _ptr(w), N, w.stride(0), _ptr(w_scale),
                                 w_scale.numel(), _ptr(bias), _ptr(y), y.stride(0), _ptr(acc), _ptr(xq), _ptr(xs),
                                 _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(path)), "qlinear_int8_w8a8")
    if debug:
        return y, acc, xq, xs, PATHS[path.value]
    return y


def qlinear_fp8_block(x, w, w_scale, *, K=None, block_n=128, block_k=128, act_mode=ACT_BF16, bias=None,
                      debug=False, out=None, workspace=None, stream=None):
    """Block-scaled FP8 linear.  w: uint8 E4M3 codes [N, ldw] (first K columns used);
    w_scale: uint8 UE8M0 [ceil(N/block_n), ceil(K/block_k)].  debug=True returns
    (y, aq, as, path) where aq/as are the 1x128 activation codes/scales (act_mode 1)."""
    _bf16(x, "x")
    M, Kx = x.shape
    K = Kx if K is None else K
    N = w.shape[0]
    y = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    aq = as_ = None
    if debug and act_mode == ACT_E4M3_1X128:
        aq = torch.empty(M, K, dtype=torch.uint8, device=x.device)
        as_ = torch.empty(M, K // 128, dtype=torch.uint8, device=x.device)
    ws = _ws(x.device, workspace_bytes(OP_FP8_BLOCK, M, N, K), stream, workspace)
    path = ctypes.c_int(0)
    _check(lib.qlinear_fp8_block(_ptr(x), M, K, x.stride(0), _ptr(w), N, w.stride(0), _ptr(w_scale), block_n,
                                 block_k, act_mode, _ptr(bias), _ptr(y), y.stride(0), _ptr(aq), _ptr(as_), _ptr(ws),
                                 ws.numel(), _stream(stream), ctypes.byref(path)), "qlinear_fp8_block")
    if debug:
        return y, aq, as_, PATHS[path.value]
    return y


def qlinear_mxfp4(x, w, w_scale, *, act_mode=ACT_BF16, bias=None, debug=False, out=None, workspace=None,
                  stream=None):
    """MXFP4 linear.  w: packed E2M1 uint8 [N, >=K/2]; w_scale: UE8M0 uint8 [N, >=K/32]."""
    _bf16(x, "x")
    M, K = x.shape
    N = w.shape[0]
    y = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    aq = as_ = None
    if debug and act_mode == ACT_E4M3_1X128:
        aq = torch.empty(M, K, dtype=torch.uint8, device=x.device)
        as_ = torch.empty(M, K // 128, dtype=torch.uint8, device=x.device)
    ws = _ws(x.device, workspace_bytes(OP_MXFP4, M, N, K), stream, workspace)
    path = ctypes.c_int(0)
    _check(lib.qlinear_mxfp4(_ptr(x), M, K, x.stride(0), _ptr(w), N, w.stride(0), _ptr(w_scale), w_scale.stride(0),
                             act_mode, _ptr(bias), _ptr(y), y.stride(0), _ptr(aq), _ptr(as_), _ptr(ws), ws.numel(),
                             _stream(stream), ctypes.byref(path)), "qlinear_mxfp4")
    if debug:
        return y, aq, as_, PATHS[path.value]
    return y


def qlinear_bf16(x, w, bias=None, *, debug=False, out=None, workspace=None, stream=None):
    """BF16 linear on unquantised weights.  x: bf16 [M, K]; w: bf16 [N, >=K] (row stride
    w.stride(0)).  With debug=True returns (y, path)."""
    _bf16(x, "x")
    M, K = x.shape
    N = w.shape[0]
    if w.dtype != torch.bfloat16 or w.stride(1) != 1 or x.stride(1) != 1:
        raise TypeError("w must be bfloat16 with unit inner stride; x must have unit inner stride")
    y = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    ws = _ws(x.device, workspace_bytes(OP_BF16, M, N, K), stream, workspace)
    path = ctypes.c_int(0)
    _check(lib.qlinear_bf16(_ptr(x), M, K, x.stride(0), _ptr(w), N, w.stride(0), _ptr(bias), _ptr(y), y.stride(0),
                            _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(path)), "qlinear_bf16")
    if debug:
        return y, PATHS[path.value]
    return y


def qlinear_fp8(x, w, w_scale, w_fmt="e4m3", bias=None, *, debug=False, out=None, workspace=None, stream=None):
    """y = bf16(w_scale[n or 0] * sum_k x w) (+ bias) on FP8 weight codes.  x: bf16 [M, K];
    w: uint8 FP8 codes [N, >=K] (row stride w.stride(0)); w_fmt: "e4m3" or "e5m2"; w_scale:
    fp32 [N] (per channel) or [1] (per tensor).  With debug=True returns (y, path)."""
    _bf16(x, "x")
    M, K = x.shape
    N = w.shape[0]
    if w.dtype != torch.uint8 or w.stride(1) != 1 or x.stride(1) != 1:
        raise TypeError("w must be uint8 FP8 codes with unit inner stride; x must have unit inner stride")
    if w_scale.dtype != torch.float32:
        raise TypeError("w_scale must be float32")
    fmt = {"e4m3": FP8_E4M3, "e5m2": FP8_E5M2}[w_fmt]
    y = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    ws = _ws(x.device, workspace_bytes(OP_FP8_CHANNEL, M, N, K), stream, workspace)
    path = ctypes.c_int(0)
    _check(lib.qlinear_fp8(_ptr(x), M, K, x.stride(0), _ptr(w), N, w.stride(0), fmt, _ptr(w_scale), w_scale.numel(),
                           _ptr(bias), _ptr(y), y.stride(0), _ptr(ws), ws.numel(), _stream(stream),
                           ctypes.byref(path)), "qlinear_fp8")
    if debug:
        return y, PATHS[path.value]
    return y


def moe_mxfp4_grouped(x, w13, s13, w2, s2, *, router_logits=None, topk_ids=None, topk_weights=None, topk=8,
                      renormalize=False, swiglu_alpha=1.0, swiglu_limit=None, debug=False, out=None, workspace=None,
                      stream=None):
    """MXFP4 MoE decode layer.  x: bf16 [M, H]; w13 [E, 2I, H/2], s13 [E, 2I, H/32],
    w2 [E, H, I/2], s2 [E, H, I/32] (uint8).  Either router_logits (bf16 [M, E]) or
    topk_ids/topk_weights.  Expert activation silu(alpha * min(g, limit)) * clamp(u, +-limit)
    (swiglu_limit None: plain silu(g) * u).  debug=True returns (y, ids, weights, h, path)."""
    _bf16(x, "x")
    M, H = x.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    if topk_ids is not None:
        topk = topk_ids.shape[1]
    y = out if out is not None else torch.empty(M, H, dtype=torch.bfloat16, device=x.device)
    ids = wts = h = None
    if debug:
        ids = torch.empty(M, topk, dtype=torch.int32, device=x.device)
        wts = torch.empty(M, topk, dtype=torch.float32, device=x.device)
        h = torch.empty(M * topk, I, dtype=torch.bfloat16, device=x.device)
    ws = _ws(x.device, workspace_bytes(OP_MOE_MXFP4, M, H, I, E, topk), stream, workspace)
    path = ctypes.c_int(0)
    _check(lib.moe_mxfp4_grouped(_ptr(x), M, H, _ptr(router_logits), _ptr(topk_ids), _ptr(topk_weights), E, topk,
                                 int(renormalize), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), I, float(swiglu_alpha),
                                 float("inf") if swiglu_limit is None else float(swiglu_limit), _ptr(ids), _ptr(wts),
                                 _ptr(h), _ptr(y), _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(path)),
           "moe_mxfp4_grouped")
    if debug:
        return y, ids, wts, h, PATHS[path.value]
    return y


_u32 = ctypes.c_uint32


# ------------------------------------------------------------------ sharded layers
def token_amax(x, *, out=None, stream=None):
    """Per-token max |x| of a K shard (fp32 [M]): the row-parallel INT8 layer's all-reduce MAX
    input."""
    _bf16(x, "x")
    M, K = x.shape
    amax = out if out is not None else torch.empty(M, dtype=torch.float32, device=x.device)
    _check(lib.ql_token_amax(_ptr(x), M, K, x.stride(0), _ptr(amax), _stream(stream)), "ql_token_amax")
    return amax


def qlinear_int8_w8a8_partial(x, w, amax, *, debug=False, out=None, workspace=None, stream=None):
    """A K shard of a row-parallel INT8 layer: exact int32 sums [M, N] over this shard's K, with
    x_s = amax / 127 (amax: the tokens' amax over the whole row).  debug=True also returns the
    codes and the path: (acc, x_q, path)."""
    _bf16(x, "x")
    M, K = x.shape
    N = w.shape[0]
    if w.dtype != torch.int8 or w.stride(1) != 1 or x.stride(1) != 1:
        raise TypeError("w must be int8 with unit inner stride; x must have unit inner stride")
    acc = out if out is not None else torch.empty(M, N, dtype=torch.int32, device=x.device)
    xq = torch.empty(M, K, dtype=torch.int8, device=x.device) if debug else None
    ws = _ws(x.device, workspace_bytes(OP_INT8_W8A8, M, N, K), stream, workspace)
    path = ctypes.c_int(0)
    _check(lib.qlinear_int8_w8a8_partial(_ptr(x), M, K, x.stride(0), _ptr(w), N, w.stride(0), _ptr(amax), _ptr(acc),
                                         _ptr(xq), _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(path)),
           "qlinear_int8_w8a8_partial")
    if debug:
        return acc, xq, PATHS[path.value]
    return acc


def qlinear_int8_epilogue(acc, amax, w_scale, bias=None, *, out=None, stream=None):
    """y = bf16((acc * amax/127) * w_scale) (+ bias) on int32 sums added over the shards."""
    M, N = acc.shape
    y = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=acc.device)
    _check(lib.qlinear_int8_epilogue(_ptr(acc), M, N, _ptr(amax), _ptr(w_scale), w_scale.numel(), _ptr(bias), _ptr(y),
                                     y.stride(0), _stream(stream)), "qlinear_int8_epilogue")
    return y


def qlinear_fp8_block_partial(x, w, w_scale, *, K=None, block_n=128, block_k=128, out=None, workspace=None,
                              stream=None):
    """A K shard of a row-parallel FP8-block layer: fp32 partial sums [M, N] (no bias)."""
    _bf16(x, "x")
    M, Kx = x.shape
    K = Kx if K is None else K
    N = w.shape[0]
    y32 = out if out is not None else torch.empty(M, N, dtype=torch.float32, device=x.device)
    ws = _ws(x.device, workspace_bytes(OP_FP8_BLOCK, M, N, K), stream, workspace)
    path = ctypes.c_int(0)
    _check(lib.qlinear_fp8_block_partial(_ptr(x), M, K, x.stride(0), _ptr(w), N, w.stride(0), _ptr(w_scale), block_n,
                                         block_k, _ptr(y32), y32.stride(0), _ptr(ws), ws.numel(), _stream(stream),
                                         ctypes.byref(path)), "qlinear_fp8_block_partial")
    return y32


def qlinear_mxfp4_partial(x, w, w_scale, *, out=None, workspace=None, stream=None):
    """A K shard of a row-parallel MXFP4 layer: fp32 partial sums [M, N] (no bias)."""
    _bf16(x, "x")
    M, K = x.shape
    N = w.shape[0]
    y32 = out if out is not None else torch.empty(M, N, dtype=torch.float32, device=x.device)
    ws = _ws(x.device, workspace_bytes(OP_MXFP4, M, N, K), stream, workspace)
    path = ctypes.c_int(0)
    _check(lib.qlinear_mxfp4_partial(_ptr(x), M, K, x.stride(0), _ptr(w), N, w.stride(0), _ptr(w_scale),
                                     w_scale.stride(0), _ptr(y32), y32.stride(0), _ptr(ws), ws.numel(), _stream(stream),
                                     ctypes.byref(path)), "qlinear_mxfp4_partial")
    return y32


def finish_f32(y32, bias=None, *, out=None, stream=None):
    """bf16(y32) (+ bias after the cast): the one rounding of fp32 sums added over the shards."""
    M, N = y32.shape
    y = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=y32.device)
    _check(lib.ql_finish_f32(_ptr(y32), M, N, y32.stride(0), _ptr(bias), _ptr(y), y.stride(0), _stream(stream)),
           "ql_finish_f32")
    return y
