"""The no-allocation INT8 entry point (qlinear_int8_w8a8_noalloc) against the workspace entry
point (qlinear_int8_w8a8), both called through the C ABI, on two calls in a row.

Callers that cannot allocate device memory (no allocator of their own, or a framework that
owns all GPU memory and forbids cudaMalloc) use the no-allocation entry point, whose scratch
is a 16 MiB array inside the library.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _util import bits_of, check_float, gpu_lib, to_bf16_tensor
from oracle import qlinear_oracle as Q

pytestmark = pytest.mark.gpu

_v, _i64 = ctypes.c_void_p, ctypes.c_int64


def _noalloc(ql):
    f = ql.lib.qlinear_int8_w8a8_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [_v, _i64, _i64, _i64, _v, _i64, _i64, _v, _i64, _v, _v, _i64, _v, _v, _v, _v,
                  ctypes.POINTER(ctypes.c_int)]
    return f


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _run_both(ql, c, path_code=1):
    M, K = c["x"].shape
    N = c["w"].shape[0]
    x = to_bf16_tensor(c["x"])
    w = torch.from_numpy(c["w"]).cuda()
    ws = torch.from_numpy(c["w_s"]).cuda()
    y_new = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    acc_new = torch.empty(M, N, dtype=torch.int32, device="cuda")
    path = ctypes.c_int(-1)
    st = _noalloc(ql)(_p(x), M, K, x.stride(0), _p(w), N, w.stride(0), _p(ws), N, None, _p(y_new), N,
                      _p(acc_new), None, None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                      ctypes.byref(path))
    assert st == 0, ql.lib.ql_status_string(st)
    assert path.value == path_code
    y_old, acc_old, _, _, _ = ql.qlinear_int8_w8a8(x, w, ws, debug=True)  # workspace entry point
    torch.cuda.synchronize()
    return bits_of(y_new), acc_new.cpu().numpy(), bits_of(y_old), acc_old.cpu().numpy()


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    ql = gpu_lib()
    from oracle import formats as F
    for (M, N, K, seed) in [(9, 1000, 4096, 41), (4, 17408, 1024, 42)]:
        c = synth.int8_case(M, N, K, seed=seed)
        y_new, acc_new, y_old, acc_old = _run_both(ql, c)
        assert np.array_equal(acc_new, acc_old)
        ref = Q.int8_w8a8(c["x"], c["w"], c["w_s"])
        check_float(y_new, F.bf16_to_f64(y_old), ref["abs_sum"])


def test_noalloc_more_than_16_tokens_takes_the_gemm_path():
    # 40 tokens: the tcgen05 GEMM (path 9); its activation image fits the scratch
    ql = gpu_lib()
    c = synth.int8_case(40, 640, 2048, seed=43)
    y_new, acc_new, y_old, acc_old = _run_both(ql, c, path_code=9)
    ref = Q.int8_w8a8(c["x"], c["w"], c["w_s"])
    assert np.array_equal(acc_new, ref["acc"]) and np.array_equal(acc_old, ref["acc"])
    assert np.array_equal(y_new, y_old)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    ql = gpu_lib()
    f = _noalloc(ql)
    # 16 tokens of K = 262144 need more than the 16 MiB scratch (the activation image alone is
    # 16 MiB, the partial sums come on top): the call is rejected before any launch, so the
    # placeholder addresses are never touched
    M, N, K = 16, 1024, 262144
    assert ql.workspace_bytes(ql.OP_INT8_W8A8, M, N, K) > 16 << 20
    st = f(ctypes.c_void_p(16), M, K, K, ctypes.c_void_p(16), N, K, ctypes.c_void_p(16), N, None,
           ctypes.c_void_p(16), N, None, None, None, None, ctypes.byref(ctypes.c_int()))
    assert st == 4
