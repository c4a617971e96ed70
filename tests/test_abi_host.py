"""Host-side checks of the C ABI (no GPU needed).

* the library builds, loads and exports every function ``include/sgemm.h``
  declares;
* argument validation rejects bad calls before touching the device: these
  paths return their status without any CUDA call, so they run on CPU.
"""
import ctypes
import os
import re

import pytest

from dense_fp32_gemm_03_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(sgemm\w*)\s*\(", text))
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert {"sgemm", "sgemm_variant", "sgemm_select_variant", "sgemm_query_device_status",
            "sgemm_status_string"} <= names
    assert names == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libsgemm.so does not export {name}"
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_and_variant_names(lib):
    assert binding.status_string(binding.OK) == "ok"
    assert "invalid" in binding.status_string(binding.ERR_INVALID_VALUE)
    assert "time" in binding.status_string(binding.ERR_TIMEOUT)
    assert binding.status_string(99) == "unknown status"
    for name, v in binding.VARIANTS.items():
        assert binding.variant_name(v) == name
    assert binding.variant_name(42) == "unknown"


# Fake device addresses: validation fails before any of them is dereferenced.
P_A, P_B, P_C = 0x10000000, 0x20000000, 0x30000000


@pytest.mark.parametrize("args", [
    (-1, 4, 4, P_A, 4, P_B, 4, P_C, 4),      # negative M
    (4, -1, 4, P_A, 4, P_B, 4, P_C, 4),      # negative N
    (4, 4, -1, P_A, 4, P_B, 4, P_C, 4),      # negative K
    (4, 4, 8, P_A, 7, P_B, 4, P_C, 4),       # lda < K
    (4, 8, 4, P_A, 4, P_B, 7, P_C, 8),       # ldb < N
    (4, 8, 4, P_A, 4, P_B, 8, P_C, 7),       # ldc < N
    (4, 4, 4, 0, 4, P_B, 4, P_C, 4),         # null A
    (4, 4, 4, P_A, 4, 0, 4, P_C, 4),         # null B
    (4, 4, 4, P_A, 4, P_B, 4, 0, 4),         # null C
    (4, 4, 4, P_A, 4, P_B, 4, P_A + 16, 4),  # C overlaps A
    (4, 4, 4, P_A, 4, P_B, 4, P_B + 60, 4),  # C overlaps B's last element
])
def test_invalid_arguments_rejected(lib, args):
    assert binding.sgemm_raw(*args) == binding.ERR_INVALID_VALUE
    assert lib.sgemm_select_variant(*args) == -1


def _header_constant(name):
    text = open(os.path.join(ROOT, "include", "sgemm.h")).read()
    return int(re.search(rf"\b{name}\s*=\s*(-?\d+)", text).group(1))


# One past the last variant id, as the header declares it.
VARIANT_COUNT = _header_constant("SGEMM_VARIANT_COUNT")


def test_variant_ids_cover_the_header_enum():
    assert sorted(binding.VARIANTS.values()) == list(range(VARIANT_COUNT))


@pytest.mark.parametrize("variant", [VARIANT_COUNT, -2, 1000])
def test_unknown_variant_rejected(lib, variant):
    """The range check runs before any device is touched, so the status is exact here."""
    assert binding.sgemm_raw(4, 4, 4, P_A, 4, P_B, 4, P_C, 4, variant=variant) == \
        binding.ERR_INVALID_VALUE


def test_oversized_dimension_unsupported(lib):
    big = 2 ** 31
    assert binding.sgemm_raw(big, 4, 4, P_A, 4, P_B, 4, P_C, 4) == binding.ERR_UNSUPPORTED


def test_null_pointers_allowed_for_empty_extents(lib):
    """M == 0 or N == 0 is a no-op; K == 0 needs only C.  Validation accepts them
    (they then need a device, so only the validator is exercised here)."""
    assert lib.sgemm_workspace_size(binding.STREAMK, 0, 4, 4) == 0


@pytest.mark.parametrize("args", [
    (0, 2, 0, 4, 4, 4),       # trans_a neither N nor T
    (0, 0, -1, 4, 4, 4),      # trans_b neither N nor T
    (5, 0, 0, 4, 4, 4),       # unknown layout
])
def test_ex2_rejects_bad_flags(lib, args):
    layout, ta, tb, M, N, K = args
    assert lib.sgemm_ex2(layout, ta, tb, M, N, K, 1.0, P_A, 8, P_B, 8, 0.0, P_C, 8, None) == \
        binding.ERR_INVALID_VALUE


@pytest.mark.parametrize("args", [
    # (trans_a, trans_b, M, N, K, lda, ldb, ldc): leading dimensions of the stored matrices
    (1, 0, 8, 4, 3, 7, 4, 4),     # A stored K x M needs lda >= M = 8
    (0, 1, 4, 8, 3, 3, 2, 8),     # B stored N x K needs ldb >= K = 3
    (1, 1, 5, 6, 9, 5, 8, 6),     # both transposed: ldb >= K = 9 fails
])
def test_ex2_checks_stored_leading_dimensions(lib, args):
    ta, tb, M, N, K, lda, ldb, ldc = args
    assert lib.sgemm_ex2(0, ta, tb, M, N, K, 1.0, P_A, lda, P_B, ldb, 0.0, P_C, ldc, None) == \
        binding.ERR_INVALID_VALUE
    # The same leading dimensions are fine once they cover the stored rows.  (Only
    # without a GPU: with one, the fake addresses would reach a kernel.)
    import torch
    if torch.cuda.is_available():
        return
    st = lib.sgemm_ex2(0, ta, tb, M, N, K, 1.0, P_A, max(lda, M if ta else K), P_B,
                       max(ldb, K if tb else N), 0.0, P_C, ldc, None)
    assert st != binding.ERR_INVALID_VALUE   # no device here: UNSUPPORTED


# sgemm_host takes host addresses; its checks also run before any memory is touched.
@pytest.mark.parametrize("args", [
    (-1, 4, 4, P_A, 4, P_B, 4, P_C, 4),      # negative M
    (4, 4, -1, P_A, 4, P_B, 4, P_C, 4),      # negative K
    (4, 4, 8, P_A, 7, P_B, 4, P_C, 4),       # lda < K
    (4, 8, 4, P_A, 4, P_B, 7, P_C, 8),       # ldb < N
    (4, 8, 4, P_A, 4, P_B, 8, P_C, 7),       # ldc < N
    (4, 4, 4, 0, 4, P_B, 4, P_C, 4),         # null A
    (4, 4, 4, P_A, 4, P_B, 4, 0, 4),         # null C
    (4, 4, 4, P_A, 4, P_B, 4, P_A + 16, 4),  # C overlaps A
    (4, 4, 4, P_A, 4, P_B, 4, P_B + 60, 4),  # C overlaps B's last element
])
def test_host_entry_rejects_invalid_arguments(lib, args):
    assert lib.sgemm_host(*args, None) == binding.ERR_INVALID_VALUE


def test_host_entry_empty_and_oversized(lib):
    assert lib.sgemm_host(0, 4, 4, 0, 4, 0, 4, 0, 4, None) == binding.OK    # M == 0: no-op
    assert lib.sgemm_host(4, 0, 4, 0, 4, 0, 4, 0, 4, None) == binding.OK    # N == 0: no-op
    assert lib.sgemm_host(2 ** 31, 4, 4, P_A, 4, P_B, 4, P_C, 4, None) == binding.ERR_UNSUPPORTED
    # Valid arguments reach the device query: without a GPU, UNSUPPORTED.  (With a
    # GPU the fake addresses would be copied from, so the call is not made there.)
    import torch
    if not torch.cuda.is_available():
        assert lib.sgemm_host(4, 4, 4, P_A, 4, P_B, 4, P_C, 4, None) == binding.ERR_UNSUPPORTED
