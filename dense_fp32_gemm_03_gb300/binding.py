"""Thin Python binding of the C ABI in ``include/sgemm.h`` (ctypes).

Argument marshalling only: every FLOP runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  There is no CPU
fallback: if ``libsgemm.so`` is missing or cannot load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

# sgemm_status_t
OK, ERR_INVALID_VALUE, ERR_LAUNCH, ERR_TIMEOUT, ERR_UNSUPPORTED, ERR_ALLOC = range(6)
# sgemm_variant_t
AUTO, GUARDED, TILED, STREAMK, TILED_SMALL, STREAMK_SMALL, STAGED, SPECIALIZED, SMALL = (
    -1, 0, 1, 2, 3, 4, 5, 6, 7)
VARIANTS = {"guarded": GUARDED, "tiled": TILED, "streamk": STREAMK,
            "tiled_small": TILED_SMALL, "streamk_small": STREAMK_SMALL, "staged": STAGED,
            "specialized": SPECIALIZED, "small": SMALL}

# Every entry point include/sgemm.h declares.
EXPORTS = ("sgemm", "sgemm_variant", "sgemm_select_variant", "sgemm_workspace_size",
           "sgemm_query_device_status", "sgemm_release_workspaces", "sgemm_status_string",
           "sgemm_variant_name", "sgemm_debug_expire_wait", "sgemm_debug_owner_publishes",
           "sgemm_streamk_static",
           "sgemm_tf32", "sgemm_ex", "sgemm_ex2", "sgemm_host")


class SgemmError(RuntimeError):
    """A nonzero sgemm_status_t."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load ``libsgemm.so`` (raises if it is absent: build it first)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run __graft_entry__.build() (the CUDA library "
                               "is required; there is no fallback)")
        lib = ctypes.CDLL(path)
        i64, vp, st = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        gemm_args = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp]
        lib.sgemm.argtypes = gemm_args
        lib.sgemm.restype = st
        lib.sgemm_variant.argtypes = [ctypes.c_int, *gemm_args]
        lib.sgemm_variant.restype = st
        lib.sgemm_select_variant.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64]
        lib.sgemm_select_variant.restype = ctypes.c_int
        lib.sgemm_workspace_size.argtypes = [ctypes.c_int, i64, i64, i64]
        lib.sgemm_workspace_size.restype = ctypes.c_size_t
        lib.sgemm_query_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.sgemm_query_device_status.restype = st
        lib.sgemm_release_workspaces.argtypes = []
        lib.sgemm_release_workspaces.restype = None
        lib.sgemm_status_string.argtypes = [ctypes.c_int]
        lib.sgemm_status_string.restype = ctypes.c_char_p
        lib.sgemm_variant_name.argtypes = [ctypes.c_int]
        lib.sgemm_variant_name.restype = ctypes.c_char_p
        lib.sgemm_debug_expire_wait.argtypes = [ctypes.c_uint64, vp]
        lib.sgemm_debug_expire_wait.restype = st
        lib.sgemm_debug_owner_publishes.argtypes = [ctypes.c_int]
        lib.sgemm_debug_owner_publishes.restype = None
        lib.sgemm_streamk_static.argtypes = gemm_args
        lib.sgemm_streamk_static.restype = st
        lib.sgemm_tf32.argtypes = gemm_args
        lib.sgemm_tf32.restype = st
        f32 = ctypes.c_float
        lib.sgemm_ex.argtypes = [ctypes.c_int, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        lib.sgemm_ex.restype = st
        lib.sgemm_ex2.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, i64, i64, f32, vp,
                                  i64, vp, i64, f32, vp, i64, vp]
        lib.sgemm_ex2.restype = st
        lib.sgemm_host.argtypes = gemm_args
        lib.sgemm_host.restype = st
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().sgemm_status_string(int(status)).decode()


def variant_name(variant: int) -> str:
    return load().sgemm_variant_name(int(variant)).decode()


# ------------------------------------------------------------ raw pointer calls
def sgemm_raw(M, N, K, A, lda, B, ldb, C, ldc, stream=0, variant=AUTO) -> int:
    """Call the C ABI with integer device addresses; returns the status code."""
    lib = load()
    if variant == AUTO:
        return lib.sgemm(M, N, K, A, lda, B, ldb, C, ldc, stream)
    return lib.sgemm_variant(variant, M, N, K, A, lda, B, ldb, C, ldc, stream)


# ------------------------------------------------------------- tensor interface
def _check_operand(t, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda" or t.dtype != torch.float32 or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D float32 CUDA tensor, got {t.dtype} {tuple(t.shape)} on {t.device}")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major (unit column stride)")
    # Row stride in elements; for a single row it only has to cover the row.
    return max(t.stride(0), t.shape[1], 1)


def _stream_handle(device, stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def sgemm(A, B, out=None, variant: int = AUTO, stream=None):
    """C = A @ B for 2-D float32 CUDA tensors (row-major, any row stride).

    Runs on ``stream`` (default: the current stream of A's device).  ``out``
    (M x N, float32, row-major) receives the result if given.
    """
    import torch
    lda = _check_operand(A, "A")
    ldb = _check_operand(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {tuple(A.shape)} @ {tuple(B.shape)}")
    if B.device != A.device:
        raise ValueError("A and B must be on the same device")
    if out is None:
        out = torch.empty((M, N), device=A.device, dtype=torch.float32)
    else:
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out has shape {tuple(out.shape)}, expected {(M, N)}")
    ldc = _check_operand(out, "out")
    with torch.cuda.device(A.device):
        st = sgemm_raw(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc,
                       _stream_handle(A.device, stream), variant)
    if st != OK:
        raise SgemmError(st, "sgemm")
    return out


ROW_MAJOR, COL_MAJOR = 0, 1


def sgemm_ex(A, B, C, alpha=1.0, beta=0.0, layout=ROW_MAJOR, stream=None):
    """C = alpha * A @ B + beta * C in place, for 2-D float32 CUDA tensors.

    ``layout`` ROW_MAJOR: tensors with unit column stride; COL_MAJOR: tensors
    with unit row stride (e.g. ``x.t().contiguous().t()``), as BLAS expects.
    """
    import torch

    def ld(t, name):
        if t.device.type != "cuda" or t.dtype != torch.float32 or t.dim() != 2:
            raise ValueError(f"{name} must be a 2-D float32 CUDA tensor")
        if layout == ROW_MAJOR:
            if t.shape[1] > 1 and t.stride(1) != 1:
                raise ValueError(f"{name} must have unit column stride")
            return max(t.stride(0), t.shape[1], 1)
        if t.shape[0] > 1 and t.stride(0) != 1:
            raise ValueError(f"{name} must have unit row stride")
        return max(t.stride(1), t.shape[0], 1)
    lda, ldb, ldc = ld(A, "A"), ld(B, "B"), ld(C, "C")
    M, K = A.shape
    K2, N = B.shape
    if K != K2 or tuple(C.shape) != (M, N):
        raise ValueError(f"shapes do not match: {tuple(A.shape)} @ {tuple(B.shape)} -> {tuple(C.shape)}")
    with torch.cuda.device(A.device):
        st = load().sgemm_ex(int(layout), M, N, K, float(alpha), A.data_ptr(), lda,
                             B.data_ptr(), ldb, float(beta), C.data_ptr(), ldc,
                             _stream_handle(A.device, stream))
    if st != OK:
        raise SgemmError(st, "sgemm_ex")
    return C


OP_N, OP_T = 0, 1


def sgemm_ex2(A, B, C, alpha=1.0, beta=0.0, trans_a=False, trans_b=False, layout=ROW_MAJOR,
              stream=None):
    """C = alpha * op(A) @ op(B) + beta * C in place; op(X) = X.T when trans_x.

    ``A`` and ``B`` are the stored matrices: A is M x K (K x M when
    ``trans_a``), B is K x N (N x K when ``trans_b``); C is M x N.  Storage
    order as for :func:`sgemm_ex` (``layout``).
    """
    import torch

    def ld(t, name):
        if t.device.type != "cuda" or t.dtype != torch.float32 or t.dim() != 2:
            raise ValueError(f"{name} must be a 2-D float32 CUDA tensor")
        if layout == ROW_MAJOR:
            if t.shape[1] > 1 and t.stride(1) != 1:
                raise ValueError(f"{name} must have unit column stride")
            return max(t.stride(0), t.shape[1], 1)
        if t.shape[0] > 1 and t.stride(0) != 1:
            raise ValueError(f"{name} must have unit row stride")
        return max(t.stride(1), t.shape[0], 1)
    lda, ldb, ldc = ld(A, "A"), ld(B, "B"), ld(C, "C")
    M, K = (A.shape[1], A.shape[0]) if trans_a else tuple(A.shape)
    K2, N = (B.shape[1], B.shape[0]) if trans_b else tuple(B.shape)
    if K != K2 or tuple(C.shape) != (M, N):
        raise ValueError(f"shapes do not match: op(A) {M}x{K}, op(B) {K2}x{N}, C {tuple(C.shape)}")
    with torch.cuda.device(A.device):
        st = load().sgemm_ex2(int(layout), OP_T if trans_a else OP_N, OP_T if trans_b else OP_N,
                              M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb,
                              float(beta), C.data_ptr(), ldc, _stream_handle(A.device, stream))
    if st != OK:
        raise SgemmError(st, "sgemm_ex2")
    return C


def sgemm_host(A, B, out=None, stream=None, wait: bool = True):
    """C = A @ B for 2-D float32 CPU tensors, computed on the current CUDA device.

    The library copies A and B to the device, multiplies and copies C back
    (``sgemm_host`` in include/sgemm.h), on ``stream`` (default: the current
    stream of the current device).  Pinned tensors (``pin_memory()``) give
    asynchronous, overlapped copies.  ``out`` (M x N float32 CPU tensor, unit
    column stride) receives C; by default a pinned tensor is allocated.  With
    ``wait`` the call returns after the stream has finished; without it C is
    complete only once the stream has.
    """
    import torch

    def ld(t, name):
        if t.device.type != "cpu" or t.dtype != torch.float32 or t.dim() != 2:
            raise ValueError(f"{name} must be a 2-D float32 CPU tensor")
        if t.shape[1] > 1 and t.stride(1) != 1:
            raise ValueError(f"{name} must have unit column stride")
        return max(t.stride(0), t.shape[1], 1)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"shapes do not match: A {tuple(A.shape)}, B {tuple(B.shape)}")
    lda, ldb = ld(A, "A"), ld(B, "B")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    if tuple(out.shape) != (M, N):
        raise ValueError(f"out must be {M} x {N}")
    ldc = ld(out, "out")
    device = torch.cuda.current_device()
    handle = _stream_handle(device, stream)
    st = load().sgemm_host(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc, handle)
    if st != OK:
        raise SgemmError(st, "sgemm_host")
    if wait:
        (stream if stream is not None else torch.cuda.current_stream(device)).synchronize()
    return out


def sgemm_tf32(A, B, out=None, stream=None):
    """Opt-in TF32 tensor-core mode (not FP32 arithmetic): C = A @ B with TF32 products."""
    import torch
    lda = _check_operand(A, "A")
    ldb = _check_operand(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {tuple(A.shape)} @ {tuple(B.shape)}")
    if out is None:
        out = torch.empty((M, N), device=A.device, dtype=torch.float32)
    ldc = _check_operand(out, "out")
    with torch.cuda.device(A.device):
        st = load().sgemm_tf32(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc,
                               _stream_handle(A.device, stream))
    if st != OK:
        raise SgemmError(st, "sgemm_tf32")
    return out


def select_variant(A, B, out) -> int:
    lda, ldb, ldc = _check_operand(A, "A"), _check_operand(B, "B"), _check_operand(out, "out")
    import torch
    with torch.cuda.device(A.device):
        return load().sgemm_select_variant(A.shape[0], B.shape[1], A.shape[1], A.data_ptr(), lda,
                                           B.data_ptr(), ldb, out.data_ptr(), ldc)


def workspace_size(M: int, N: int, K: int, variant: int = AUTO) -> int:
    return int(load().sgemm_workspace_size(variant, M, N, K))


def query_device_status(stream=None) -> tuple[int, int]:
    """(status, wait site) of the current device; reading clears it."""
    import torch
    detail = ctypes.c_uint32(0)
    st = load().sgemm_query_device_status(_stream_handle(torch.cuda.current_device(), stream),
                                          ctypes.byref(detail))
    return st, int(detail.value)


def debug_expire_wait(limit_ns: int, stream=None) -> int:
    import torch
    return load().sgemm_debug_expire_wait(int(limit_ns),
                                          _stream_handle(torch.cuda.current_device(), stream))


def debug_owner_publishes(on: bool) -> None:
    """Test switch: split tiles are always summed from the workspace (see include/sgemm.h)."""
    load().sgemm_debug_owner_publishes(1 if on else 0)


def sgemm_streamk_static_raw(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """The allocation-free Stream-K entry point, with integer device addresses."""
    return load().sgemm_streamk_static(M, N, K, A, lda, B, ldb, C, ldc, stream)


def release_workspaces() -> None:
    load().sgemm_release_workspaces()
