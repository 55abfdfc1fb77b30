"""The C-ABI library loads and exports every entry point of include/qlinear.h; host-side
argument validation rejects bad calls before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

from _util import ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "qlinear.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:QL_API\s+)?(?:const\s+)?[a-z_0-9]+\**\s+\**([a-z_0-9]+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    return ctypes.CDLL(ensure_built())


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("qlinear_int8_w8a8", "qlinear_fp8_block", "qlinear_mxfp4", "moe_mxfp4_grouped",
              "ql_workspace_bytes", "ql_status_string", "ql_read_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    lib.ql_status_string.restype = ctypes.c_char_p
    assert lib.ql_status_string(0) == b"ok"
    assert b"workspace" in lib.ql_status_string(4)


def test_workspace_query(lib):
    f = lib.ql_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    assert f(1, 1, 512, 1024, 0, 0) >= 256 + 1024
    assert f(4, 9, 4096, 2048, 256, 8) >= 72 * 2048 * 2 + 72 * 4096 * 4
    assert f(99, 1, 1, 1, 0, 0) == 0
    assert f(1, -1, 1, 1, 0, 0) == 0


def test_int8_gemm_workspace_holds_split_k_partials_only_when_k_is_split(lib):
    """M > 16 INT8 GEMM: one CTA per 128 weight rows and token tile.  When those tiles fill fewer
    than half of the 152 SMs, K is split (up to 8 ranges, one split per 512-K group at most) and
    the workspace holds an int32 slot [ks][M][N] per split on top of the f16 activation image."""
    f = lib.ql_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    op = 1  # QL_OP_INT8_W8A8
    image = lambda M, K: M * (-(-K // 64) * 64) * 2
    # 5120 rows, 128 tokens: 40 tiles -> 3 splits (120 CTAs)
    assert f(op, 128, 5120, 17408, 0, 0) >= image(128, 17408) + 3 * 128 * 5120 * 4
    # 17408 rows: 136 tiles fill the SMs -> no split (two slots alone would exceed the bound)
    big = f(op, 128, 17408, 5120, 0, 0)
    assert big >= image(128, 5120) and big < image(128, 5120) + 2 * 128 * 17408 * 4


def _int8_call(lib, **kw):
    a = dict(x=16, M=1, K=64, ldx=64, w=16, N=64, ldw=64, ws=16, wsl=64, bias=None, y=16, ldy=64,
             acc=None, xq=None, xs=None, work=16, wbytes=1 << 20)
    a.update(kw)
    f = lib.qlinear_int8_w8a8
    f.restype = ctypes.c_int
    v, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [v, i64, i64, i64, v, i64, i64, v, i64, v, v, i64, v, v, v, v, ctypes.c_size_t, v,
                  ctypes.POINTER(ctypes.c_int)]
    path = ctypes.c_int(-1)
    st = f(a["x"], a["M"], a["K"], a["ldx"], a["w"], a["N"], a["ldw"], a["ws"], a["wsl"], a["bias"], a["y"],
           a["ldy"], a["acc"], a["xq"], a["xs"], a["work"], a["wbytes"], None, ctypes.byref(path))
    return st, path.value


def test_validation_rejects_before_launch(lib):
    # fake device addresses are never dereferenced: validation fails first
    assert _int8_call(lib, x=None) == (1, 0)
    assert _int8_call(lib, M=0)[0] == 1
    assert _int8_call(lib, ldx=32)[0] == 1            # ldx < K
    assert _int8_call(lib, wsl=3)[0] == 1             # scale length neither N nor 1
    assert _int8_call(lib, K=40, ldx=40, ldw=48)[0] == 2   # K % 16
    assert _int8_call(lib, x=17)[0] == 3              # misaligned activations
    assert _int8_call(lib, ldw=72)[0] == 3            # row stride not a multiple of 16 bytes
    assert _int8_call(lib, work=None)[0] == 4
    assert _int8_call(lib, wbytes=16)[0] == 4


def test_moe_validation(lib):
    f = lib.moe_mxfp4_grouped
    f.restype = ctypes.c_int
    v, i64, c = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fl = ctypes.c_float
    f.argtypes = [v, i64, i64, v, v, v, c, c, c, v, v, v, v, i64, fl, fl, v, v, v, v, v, ctypes.c_size_t, v,
                  ctypes.POINTER(c)]
    path = c(0)
    inf = float("inf")
    base = [16, 1, 256, 16, None, None, 16, 4, 0, 16, 16, 16, 16, 128, 1.0, inf, None, None, None, 16, 16, 1 << 30,
            None]
    args = list(base); args[3] = None                  # neither logits nor ids
    assert f(*args, ctypes.byref(path)) == 1
    args = list(base); args[1] = 65536                 # M > 65535
    assert f(*args, ctypes.byref(path)) == 2
    args = list(base); args[7] = 17                    # topk > E
    assert f(*args, ctypes.byref(path)) == 2
    args = list(base); args[13] = 100                  # I % 128
    assert f(*args, ctypes.byref(path)) == 2
    for alpha, limit in ((float("nan"), 10.0), (inf, 10.0), (1.0, -1.0), (1.0, float("nan"))):
        args = list(base); args[14], args[15] = alpha, limit   # SwiGLU alpha not finite / limit < 0 or NaN
        assert f(*args, ctypes.byref(path)) == 1
