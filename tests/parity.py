"""Acceptance checks shared by the GPU parity tests.

The bound is the one the FP32 path must meet for random inputs: per element
|C_gpu - C_ref| <= 4 K 2^-24 sum_k |A[m, k] B[k, n]|, where C_ref is the
oracle's float64 value.  It covers any summation order with at most K
roundings of unit 2^-24 (the classical gamma_K bound for recursive, blocked
or split summation), the final rounding to FP32, and margin.  Integer-valued
inputs whose partial sums stay below 2^24 must match exactly.
"""
from __future__ import annotations

import numpy as np

U24 = 2.0 ** -24

# The pages' own acceptance gate for a kernel's output: finite values and
# max |err| / max |ref| below 1e-4 ("Beyond Kernel 7: Closing the Gap to cuBLAS
# on an H100 FP32 GEMM", section "What the result establishes").
PAGES_GATE = 1e-4

# (check, max relative error, max |err| / max |ref|) of every check_within_bound
# call in this process; printed at the end of the pytest run (conftest.py).
REPORT: list[tuple[str, float, float]] = []


def bound(K: int, E: np.ndarray) -> np.ndarray:
    return 4.0 * K * U24 * E


def check_within_bound(C_gpu, C_ref, E, K, what=""):
    """Assert the elementwise bound; return (max relative error, max |err| / max |ref|)."""
    C_gpu = np.asarray(C_gpu, dtype=np.float64)
    assert C_gpu.shape == C_ref.shape, (C_gpu.shape, C_ref.shape)
    assert np.all(np.isfinite(C_gpu)), f"{what}: non-finite output"
    err = np.abs(C_gpu - C_ref)
    lim = bound(K, E)
    bad = err > lim
    if np.any(bad):
        idx = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements outside 4K2^-24 sum|ab|; first at {tuple(idx)}: "
            f"gpu {C_gpu[tuple(idx)]!r} ref {C_ref[tuple(idx)]!r} err {err[tuple(idx)]:.3e} "
            f"bound {lim[tuple(idx)]:.3e}")
    nz = np.abs(C_ref) > 0
    max_rel = float((err[nz] / np.abs(C_ref[nz])).max()) if np.any(nz) else 0.0
    ref_max = float(np.abs(C_ref).max()) if C_ref.size else 0.0
    norm = float(err.max()) / ref_max if ref_max > 0 else 0.0
    assert norm < PAGES_GATE, f"{what}: max|err|/max|ref| = {norm:.3e}, the pages' gate is 1e-4"
    REPORT.append((what, max_rel, norm))
    return max_rel, norm


def check_exact(C_gpu, C_ref, what=""):
    C_gpu = np.asarray(C_gpu, dtype=np.float64)
    assert C_gpu.shape == C_ref.shape
    if not np.array_equal(C_gpu, C_ref):
        idx = np.argwhere(C_gpu != C_ref)[0]
        raise AssertionError(f"{what}: not bit-exact at {tuple(idx)}: gpu {C_gpu[tuple(idx)]!r} "
                             f"ref {C_ref[tuple(idx)]!r}")
