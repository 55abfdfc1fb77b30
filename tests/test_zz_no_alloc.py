"""The no-allocation INT8 entry point (qlinear_int8_w8a8_noalloc), called through the C ABI.

Callers that cannot allocate device memory (no allocator of their own, or a framework that
owns all GPU memory and forbids cudaMalloc) use the no-allocation entry point, whose scratch
is a 16 MiB array inside the library.  Its results are checked against the oracle (int32
accumulators bit-exact, y within the float bar) and against the workspace entry point
(qlinear_int8_w8a8), on two calls in a row.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _util import bits_of, check_float, gpu_lib, sample_rows, to_bf16_tensor
from oracle import formats as F
from oracle import qlinear_oracle as Q

pytestmark = pytest.mark.gpu

_v, _i64 = ctypes.c_void_p, ctypes.c_int64
DEFAULT_WAIT_LIMIT = 1 << 20


def _noalloc(ql):
    f = ql.lib.qlinear_int8_w8a8_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [_v, _i64, _i64, _i64, _v, _i64, _i64, _v, _i64, _v, _v, _i64, _v, _v, _v, _v,
                  ctypes.POINTER(ctypes.c_int)]
    return f


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_noalloc(ql, x, w, ws, path_code=None):
    M, K = x.shape
    N = w.shape[0]
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(M, N, dtype=torch.int32, device="cuda")
    path = ctypes.c_int(-1)
    st = _noalloc(ql)(_p(x), M, K, x.stride(0), _p(w), N, w.stride(0), _p(ws), ws.numel(), None, _p(y), N,
                      _p(acc), None, None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                      ctypes.byref(path))
    assert st == 0, ql.lib.ql_status_string(st)
    if path_code is not None:
        assert path.value == path_code
    return y, acc


def _run_both(ql, c, path_code=1):
    x = to_bf16_tensor(c["x"])
    w = torch.from_numpy(c["w"]).cuda()
    ws = torch.from_numpy(c["w_s"]).cuda()
    y_new, acc_new = _call_noalloc(ql, x, w, ws, path_code)
    y_old, acc_old, _, _, _ = ql.qlinear_int8_w8a8(x, w, ws, debug=True)  # workspace entry point
    torch.cuda.synchronize()
    return bits_of(y_new), acc_new.cpu().numpy(), bits_of(y_old), acc_old.cpu().numpy()


def _check_vs_oracle(c, y, acc, rows=None):
    ref = Q.int8_w8a8(c["x"], c["w"], c["w_s"], rows=rows)
    sl = slice(None) if rows is None else rows
    assert np.array_equal(acc[:, sl], ref["acc"]), "int32 accumulators differ from the oracle"
    check_float(y[:, sl], F.bf16_to_f64(ref["y"]), ref["abs_sum"])
    return ref


def test_noalloc_matches_oracle_and_workspace_entry_on_two_calls_in_a_row():
    ql = gpu_lib()
    for (M, N, K, seed) in [(9, 1000, 4096, 41), (4, 17408, 1024, 42)]:
        c = synth.int8_case(M, N, K, seed=seed)
        y_new, acc_new, y_old, acc_old = _run_both(ql, c)
        ref = _check_vs_oracle(c, y_new, acc_new)
        assert np.array_equal(acc_new, acc_old)
        check_float(y_new, F.bf16_to_f64(y_old), ref["abs_sum"])


def test_noalloc_more_than_16_tokens_takes_the_gemm_path():
    # 40 tokens: the tcgen05 GEMM (path 9); its activation image fits the scratch
    ql = gpu_lib()
    c = synth.int8_case(40, 640, 2048, seed=43)
    y_new, acc_new, y_old, acc_old = _run_both(ql, c, path_code=9)
    _check_vs_oracle(c, y_new, acc_new)
    assert np.array_equal(acc_old, acc_new) and np.array_equal(y_new, y_old)


def test_noalloc_after_a_timed_out_call_split_k_and_largest_shape():
    """A call cut short by a zero wait limit leaves counters mid-count in the scratch; the
    next calls clear them and are exact again: the GEMM path with several token tiles and a
    K split (M = 384, N = 2048: 48 output tiles, so K is split), and the 27B-class shape
    M = 128, N = 5120, K = 17408 (about 12 MiB of scratch)."""
    ql = gpu_lib()
    c0 = synth.int8_case(4, 4096, 2048, seed=44)
    x0, w0, s0 = to_bf16_tensor(c0["x"]), torch.from_numpy(c0["w"]).cuda(), torch.from_numpy(c0["w_s"]).cuda()
    ql.set_wait_limit(0)
    try:
        for _ in range(4):
            _call_noalloc(ql, x0, w0, s0)
        torch.cuda.synchronize()
    finally:
        ql.set_wait_limit(DEFAULT_WAIT_LIMIT)
    y, acc = _call_noalloc(ql, x0, w0, s0, path_code=1)
    torch.cuda.synchronize()
    _check_vs_oracle(c0, bits_of(y), acc.cpu().numpy())

    c1 = synth.int8_case(384, 2048, 4096, seed=45)
    assert ql.workspace_bytes(ql.OP_INT8_W8A8, 384, 2048, 4096) <= 16 << 20
    y, acc = _call_noalloc(ql, to_bf16_tensor(c1["x"]), torch.from_numpy(c1["w"]).cuda(),
                           torch.from_numpy(c1["w_s"]).cuda(), path_code=9)
    torch.cuda.synchronize()
    _check_vs_oracle(c1, bits_of(y), acc.cpu().numpy())

    c2 = synth.int8_case(128, 5120, 17408, seed=46)
    assert ql.workspace_bytes(ql.OP_INT8_W8A8, 128, 5120, 17408) <= 16 << 20
    for _ in range(2):
        y, acc = _call_noalloc(ql, to_bf16_tensor(c2["x"]), torch.from_numpy(c2["w"]).cuda(),
                               torch.from_numpy(c2["w_s"]).cuda(), path_code=9)
        torch.cuda.synchronize()
        _check_vs_oracle(c2, bits_of(y), acc.cpu().numpy(), rows=sample_rows(5120, n=400, seed=46))


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
