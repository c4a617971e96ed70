"""The product and the oracle stay apart, and the product has no fallback (CPU).

* No product source (the package's Python modules, its CUDA sources, the
  public header) imports, includes or links the oracle.
* The oracle includes nothing from the product: no product header, no
  package import.  The only module both sides use is the seeded input
  generator (``workloads.py``), which holds none of the arithmetic.
* Without its CUDA library the binding raises instead of computing
  anything elsewhere.
* The benchmark reports a profile's DRAM traffic only for the exact kernel
  source the profile was taken from.
"""
from __future__ import annotations

import glob
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "dense_fp32_gemm_03_gb300")


def _product_sources():
    files = glob.glob(os.path.join(PKG, "*.py"))
    files += glob.glob(os.path.join(PKG, "csrc", "*"))
    files += glob.glob(os.path.join(ROOT, "include", "*.h"))
    return [f for f in files if os.path.isfile(f)]


def test_product_never_uses_the_oracle():
    pattern = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[<\"].*ref_sgemm)|"
                         r"ref_sgemm_\w+\s*\(|libref_sgemm", re.M)
    for path in _product_sources():
        text = open(path, errors="replace").read()
        assert not pattern.search(text), f"{path} refers to the oracle"


def test_oracle_uses_nothing_from_the_product():
    pattern = re.compile(r"dense_fp32_gemm_03_gb300|#\s*include\s*\"|sgemm_\w+\.(h|cuh)|csrc")
    for path in glob.glob(os.path.join(ROOT, "oracle", "*")):
        if os.path.isfile(path):
            text = open(path, errors="replace").read()
            assert not pattern.search(text), f"{path} refers to the product"


def test_missing_library_raises():
    code = ("from dense_fp32_gemm_03_gb300 import binding\n"
            "try:\n"
            "    binding.load('/nonexistent/libsgemm.so')\n"
            "except RuntimeError as e:\n"
            "    print('raised:', e)\n")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT,
                         check=True, timeout=120).stdout
    assert out.startswith("raised:") and "no fallback" in out, out


def test_profile_traffic_applies_to_its_kernel_source_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    traffic = bench.measured_traffic("square_4096_uniform")
    assert traffic is None or traffic > 0
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "0" * 64)
    assert bench.measured_traffic("square_4096_uniform") is None
    assert bench.measured_traffic("no_such_workload") is None


def test_host_tensors_are_refused():
    """The tensor API computes on the GPU only: host tensors raise, nothing is computed."""
    import pytest
    import torch
    import dense_fp32_gemm_03_gb300 as sg
    A = torch.ones(4, 4)
    for call in (lambda: sg.sgemm(A, A), lambda: sg.sgemm_tf32(A, A),
                 lambda: sg.sgemm_ex(A, A, torch.zeros(4, 4))):
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
