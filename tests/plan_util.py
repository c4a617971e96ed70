"""The tile kernel's work decomposition, read from the library's own header.

``plan_launch`` (csrc/sgemm_plan.h) is a constexpr function that the host API
and the size-specialized kernels evaluate.  ``tests/plan_probe.cpp`` prints its
plans; this module compiles that probe once per process (g++ and the CUDA
headers) and gives the tests the plans and the tile raster, so that GPU tests
can pick output blocks that hold split (Stream-K) tiles by the schedule, not by
guess.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_fp32_gemm_03_gb300", "csrc")
FIELDS = ("ok", "tiles_m", "tiles_n", "ipt", "dp_tiles", "sk_tiles", "sk_ctas", "sk_base",
          "sk_extra", "grid", "slots", "group_m", "spec")

_exe = None


def available() -> bool:
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    return shutil.which("g++") is not None and os.path.exists(os.path.join(cuda_inc, "cuda.h"))


def _probe() -> str:
    global _exe
    if _exe is None:
        cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
        exe = os.path.join(tempfile.mkdtemp(prefix="plan_probe"), "plan_probe")
        subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, "-I", cuda_inc,
                        os.path.join(ROOT, "tests", "plan_probe.cpp"), "-o", exe], check=True)
        _exe = exe
    return _exe


def plans(cases):
    """plan_launch for each (M, N, K, bm, bn, bk, resident, streamk) case, as dicts."""
    text = "".join(f"{M} {N} {K} {bm} {bn} {bk} {res} {int(sk)}\n"
                   for M, N, K, bm, bn, bk, res, sk in cases)
    out = subprocess.run([_probe()], input=text, capture_output=True, text=True, check=True).stdout
    return [dict(zip(FIELDS, map(int, line.split()))) for line in out.splitlines()]


def plan(M, N, K, bm, bn, bk, resident, streamk=True):
    return plans([(M, N, K, bm, bn, bk, resident, streamk)])[0]


def tile_coords(p, tile):
    """(tile row, tile column) of linear tile index `tile` in the grouped raster."""
    per_group = p["group_m"] * p["tiles_n"]
    g = tile // per_group
    first = g * p["group_m"]
    rows = min(p["tiles_m"] - first, p["group_m"])
    r = tile - g * per_group
    return first + r % rows, r // rows


def split_tiles(p):
    """Linear indices of the tiles whose K range is shared by several CTAs."""
    return range(p["dp_tiles"], p["dp_tiles"] + p["sk_tiles"])
