"""Builds ``libsgemm.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` file compiles to an object in parallel, then the objects
link into ``dense_fp32_gemm_03_gb300/_build/libsgemm.so``.  The build is
skipped when the library is newer than every source and header.

``build_trace()`` builds a separate instrumented copy,
``_build/trace/libsgemm_trace.so``, with the tile kernel's phase trace
compiled in (``-DSGEMM_PHASE_TRACE``, see ``csrc/sgemm_trace.h``).  It is a
diagnostic build only: the product library never contains the trace, and
nothing but ``phase_trace.py`` loads the traced one.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libsgemm.so")
TRACE_BUILD = os.path.join(BUILD, "trace")
TRACE_LIB = os.path.join(TRACE_BUILD, "libsgemm_trace.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsgemm.so")
    return path


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _compile(src: str, out_dir: str = BUILD, extra: tuple = ()) -> tuple[str, str]:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr  # ptxas -v writes register / spill reports to stderr


def _build_lib(lib: str, out_dir: str, extra: tuple, force: bool, verbose: bool) -> str:
    os.makedirs(out_dir, exist_ok=True)
    if not force and os.path.exists(lib):
        newest = max(os.path.getmtime(p) for p in _inputs())
        if os.path.getmtime(lib) >= newest:
            return lib
    with cf.ThreadPoolExecutor(max_workers=len(sources())) as ex:
        results = list(ex.map(lambda src: _compile(src, out_dir, extra), sources()))
    report = "\n".join(r[1] for r in results)
    with open(os.path.join(out_dir, "ptxas_report.txt"), "w") as f:
        f.write(report)
    if verbose:
        print(report)
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if it is missing or stale; return its path."""
    return _build_lib(LIB, BUILD, (), force, verbose)


def build_trace(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the phase-traced diagnostic copy; return its path."""
    return _build_lib(TRACE_LIB, TRACE_BUILD, ("-DSGEMM_PHASE_TRACE",), force, verbose)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
