"""Shared helpers of the parity tests: building/loading the library, tolerance checks."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import formats as F  # noqa: E402


def load_build_module():
    """The build script, loaded by path (importing the package would load the library)."""
    import importlib.util
    path = os.path.join(ROOT, "skinny_gemm_dequant_gb300", "_build.py")
    spec = importlib.util.spec_from_file_location("_ql_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def ensure_built():
    b = load_build_module()
    if not os.path.exists(b.LIB):
        b.build()
    return b.LIB


def bits_of(t):
    """bf16 torch tensor -> numpy uint16 bit patterns."""
    import torch
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def to_bf16_tensor(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def check_float(y_bits, y_ref, abs_sum, rtol=1e-3, what="y"):
    """|y - y_ref| <= rtol * sum_k |w x| + 1 bf16 ulp(y_ref): the float parity bar."""
    y = F.bf16_to_f64(y_bits)
    err = np.abs(y - y_ref)
    tol = rtol * abs_sum + F.bf16_ulp(y_ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = ", ".join(f"{tuple(i)}: got {y[tuple(i)]!r} want {y_ref[tuple(i)]!r} tol {tol[tuple(i)]:.3g}" for i in idx)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; {msg}")
    return float(np.max(err / np.maximum(tol, 1e-300)))


def gpu_lib():
    """Build if needed and import the binding (the GPU tests' entry to the C ABI)."""
    ensure_built()
    import skinny_gemm_dequant_gb300 as ql
    return ql


def sample_rows(N, n=48, seed=0):
    g = np.random.default_rng(seed)
    r = np.unique(np.concatenate([[0, N - 1, N // 2], g.integers(0, N, n)]))
    return r


def h_tolerance(st, alpha=1.0, limit=None):
    """|dh| <= 1e-3 (1.1 alpha |u_c| G + |silu(alpha g_c)| U) + 1.1e-6 alpha G U + 2^-20 |h|
    + ulp(h): the float bar on g and u (1e-3 * sum|w x|) carried through
    h = silu(alpha g_c) * u_c, where g_c = min(g, limit) and u_c = clip(u, +-limit) are
    1-Lipschitz in g and u and |d silu(alpha g)/dg| <= 1.1 alpha, plus fp32 evaluation of
    the activation and the final bf16 rounding."""
    from oracle import qlinear_oracle as Q
    g, u, G, U = st["g"], st["u"], st["G"], st["U"]
    if limit is not None:
        g, u = np.minimum(g, limit), np.clip(u, -limit, limit)
    s = Q.silu(alpha * g)
    return 1e-3 * (1.1 * abs(alpha) * np.abs(u) * G + np.abs(s) * U) + 1.1e-6 * abs(alpha) * G * U \
        + 2.0 ** -20 * np.abs(s * u) + F.bf16_ulp(st["h_f64"])
