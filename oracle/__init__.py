"""CPU oracle for FP32 GEMM -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does, and this
package imports nothing from the product package: the two share no code.

What it computes is the plain definition from "Beyond Kernel 7: Closing the
Gap to cuBLAS on an H100 FP32 GEMM", section "The operation: GEMM and the
precision of the comparison": ``C[m, n] = sum_k A[m, k] * B[k, n]`` for
row-major A (M x K) and B (K x N), alpha = 1, beta = 0.  The arithmetic is a
C triple loop in ``ref_sgemm.c`` that widens every FP32 input to float64
(products exact, sums rounded in k order).  Next to C it returns
``E[m, n] = sum_k |A[m, k] * B[k, n]|``, which scales the acceptance bound.

Pins (``tests/test_oracle_pins.py``): identity and permutation matrices,
the rank-1 closed form, brute force against exact rational arithmetic on all
shapes 1..8, an independent float64 library product, K-split additivity and
the transpose identity.  The scaled forms: ``sgemm_ex_f64`` (alpha, beta,
row- or column-major storage) and ``sgemm_op_f64`` (the same with a
transposition flag per operand, op(A) = A or A^T, op(B) = B or B^T), pinned
by integer products of explicit transposes, bit-identity with the plain
definition on explicitly transposed operands, and the transpose identity.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_sgemm.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libref_sgemm.so")
_CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC"]

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``ref_sgemm.c`` with gcc into ``oracle/_build/`` and return the path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, fp, dp = ctypes.c_int64, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_int64)
            lib.ref_sgemm_f64.argtypes = [i64, i64, i64, fp, i64, fp, i64, dp, i64, dp, i64]
            lib.ref_sgemm_f64.restype = ctypes.c_int
            lib.ref_sgemm_entries_f64.argtypes = [i64, i64, i64, fp, i64, fp, i64, i64, lp, lp, dp, dp]
            lib.ref_sgemm_entries_f64.restype = ctypes.c_int
            lib.ref_sgemm_ex_f64.argtypes = [ctypes.c_int, i64, i64, i64, ctypes.c_double, fp, i64, fp,
                                             i64, ctypes.c_double, fp, i64, dp, i64]
            lib.ref_sgemm_ex_f64.restype = ctypes.c_int
            lib.ref_sgemm_op_f64.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, i64, i64,
                                             ctypes.c_double, fp, i64, fp, i64, ctypes.c_double, fp,
                                             i64, dp, i64]
            lib.ref_sgemm_op_f64.restype = ctypes.c_int
            lib.ref_set_threads.argtypes = [ctypes.c_int]
            lib.ref_set_threads.restype = None
            lib.ref_max_threads.argtypes = []
            lib.ref_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_f32_rows(x, name):
    """Accept a 2-D float32 array (numpy or CPU torch tensor) with unit column stride."""
    if hasattr(x, "detach"):  # a CPU torch tensor; no torch import needed here
        if x.device.type != "cpu":
            raise ValueError(f"{name}: the oracle takes host arrays only")
        x = x.detach().numpy()
    x = np.asarray(x)
    if x.dtype != np.float32 or x.ndim != 2:
        raise ValueError(f"{name}: expected a 2-D float32 array, got {x.dtype} {x.shape}")
    if x.strides[1] != 4 or (x.shape[0] > 1 and x.strides[0] % 4):
        x = np.ascontiguousarray(x)
    ld = x.strides[0] // 4 if x.shape[0] > 1 else max(x.shape[1], 1)
    return x, ld


def _fptr(x):
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def sgemm_f64(A, B, with_abs: bool = True):
    """Return ``(C, E)``: C = A.B and E = |A|.|B| elementwise sums, both float64 (M x N).

    ``A`` is M x K and ``B`` is K x N, float32, row-major with any row stride.
    ``E`` is None when ``with_abs`` is False.
    """
    A, lda = _as_f32_rows(A, "A")
    B, ldb = _as_f32_rows(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {A.shape} x {B.shape}")
    C = np.zeros((M, N), dtype=np.float64)
    E = np.zeros((M, N), dtype=np.float64) if with_abs else None
    dp = ctypes.POINTER(ctypes.c_double)
    st = _load().ref_sgemm_f64(
        M, N, K, _fptr(A), lda, _fptr(B), ldb,
        C.ctypes.data_as(dp), max(N, 1),
        E.ctypes.data_as(dp) if E is not None else None, max(N, 1))
    if st != 0:
        raise ValueError(f"ref_sgemm_f64 rejected its arguments (status {st})")
    return C, E


def sgemm_entries_f64(A, B, rows, cols):
    """Return ``(c, e)`` float64 vectors: C and E at the given (row, col) pairs only."""
    A, lda = _as_f32_rows(A, "A")
    B, ldb = _as_f32_rows(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {A.shape} x {B.shape}")
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    c = np.zeros(rows.shape[0], dtype=np.float64)
    e = np.zeros(rows.shape[0], dtype=np.float64)
    lp, dp = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)
    st = _load().ref_sgemm_entries_f64(
        M, N, K, _fptr(A), lda, _fptr(B), ldb, rows.shape[0],
        rows.ctypes.data_as(lp), cols.ctypes.data_as(lp),
        c.ctypes.data_as(dp), e.ctypes.data_as(dp))
    if st != 0:
        raise ValueError(f"ref_sgemm_entries_f64 rejected its arguments (status {st})")
    return c, e


def sgemm_ex_f64(A, B, alpha=1.0, beta=0.0, C0=None, col_major=False):
    """alpha * (A . B) + beta * C0 in float64 (M x N, row-major result).

    With ``col_major`` the float32 arrays are column-major: pass them as numpy
    arrays in Fortran order (A: M x K, B: K x N, C0: M x N).  beta == 0 never
    reads C0.
    """
    def prep(x, name):
        if hasattr(x, "detach"):
            x = x.detach().numpy()
        x = np.asarray(x)
        if x.dtype != np.float32 or x.ndim != 2:
            raise ValueError(f"{name}: expected a 2-D float32 array")
        if col_major:
            x = np.asfortranarray(x)
            return x, max(x.shape[0], 1)
        x = np.ascontiguousarray(x)
        return x, max(x.shape[1], 1)
    A, lda = prep(A, "A")
    B, ldb = prep(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {A.shape} x {B.shape}")
    if beta != 0.0:
        C0, ldc = prep(C0, "C0")
        if C0.shape != (M, N):
            raise ValueError("C0 has the wrong shape")
        c0p = _fptr(C0)
    else:
        ldc, c0p = max(M if col_major else N, 1), None
    out = np.zeros((M, N), dtype=np.float64)
    st = _load().ref_sgemm_ex_f64(int(bool(col_major)), M, N, K, float(alpha), _fptr(A), lda,
                                  _fptr(B), ldb, float(beta), c0p, ldc,
                                  out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), max(N, 1))
    if st != 0:
        raise ValueError(f"ref_sgemm_ex_f64 rejected its arguments (status {st})")
    return out


def sgemm_op_f64(A, B, trans_a=False, trans_b=False, alpha=1.0, beta=0.0, C0=None,
                 col_major=False):
    """alpha * (op(A) . op(B)) + beta * C0 in float64 (M x N, row-major result).

    ``A`` and ``B`` are the STORED float32 arrays: A is M x K, or K x M when
    ``trans_a`` (op(A) = A^T); B is K x N, or N x K when ``trans_b``.  With
    ``col_major`` they (and C0) are taken in Fortran order, as for
    ``sgemm_ex_f64``.  beta == 0 never reads C0.
    """
    def prep(x, name):
        if hasattr(x, "detach"):
            x = x.detach().numpy()
        x = np.asarray(x)
        if x.dtype != np.float32 or x.ndim != 2:
            raise ValueError(f"{name}: expected a 2-D float32 array")
        if col_major:
            x = np.asfortranarray(x)
            return x, max(x.shape[0], 1)
        x = np.ascontiguousarray(x)
        return x, max(x.shape[1], 1)
    A, lda = prep(A, "A")
    B, ldb = prep(B, "B")
    M, K = (A.shape[1], A.shape[0]) if trans_a else A.shape
    K2, N = (B.shape[1], B.shape[0]) if trans_b else B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: op(A) {M}x{K}, op(B) {K2}x{N}")
    if beta != 0.0:
        C0, ldc = prep(C0, "C0")
        if C0.shape != (M, N):
            raise ValueError("C0 has the wrong shape")
        c0p = _fptr(C0)
    else:
        ldc, c0p = max(M if col_major else N, 1), None
    out = np.zeros((M, N), dtype=np.float64)
    st = _load().ref_sgemm_op_f64(int(bool(col_major)), int(bool(trans_a)), int(bool(trans_b)),
                                  M, N, K, float(alpha), _fptr(A), lda, _fptr(B), ldb, float(beta),
                                  c0p, ldc, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                  max(N, 1))
    if st != 0:
        raise ValueError(f"ref_sgemm_op_f64 rejected its arguments (status {st})")
    return out


def set_threads(n: int) -> None:
    """Set the OpenMP thread count the oracle uses (n <= 0 keeps the default)."""
    _load().ref_set_threads(int(n))


def max_threads() -> int:
    """Threads the oracle's OpenMP loops use at most."""
    return int(_load().ref_max_threads())
