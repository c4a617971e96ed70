"""The benchmark's reference arm on the host: its one JSON line keeps the contract.

``bench.py --impl reference`` times the CPU oracle on the benchmark's metric and
workload; it needs no GPU, so its output line is checked here: one JSON object
with the metric, value, unit, step counts, the oracle description
(``cpu_baseline``) and an end-to-end figure with no host/device copies.  The
small 256^3 workload keeps the run to a few seconds.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
         "square_256_uniform", "--steps", "2", "--warmup", "1"],
        capture_output=True, text=True, check=True, timeout=300, cwd=ROOT).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == "FP32 SGEMM TFLOPS (and % of GB300 FFMA peak) at n=1024/4096"
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert (line["steps"], line["warmup"], line["n_gpus"]) == (2, 1, 1)
    assert line["config"]["workload"] == "square_256_uniform"
    assert (line["config"]["M"], line["config"]["N"], line["config"]["K"]) == (256, 256, 256)
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"]
    assert cpu["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_sweep_resumes_by_skipping_workloads_already_written(tmp_path):
    bench = _bench()
    from dense_fp32_gemm_03_gb300 import workloads
    out = tmp_path / "sweep.jsonl"
    everything = [w.name for w in bench.sweep_plan(workloads.ALL, str(out))]   # file absent
    assert "square_256_uniform" in everything and "square_256_int" not in everything
    out.write_text(json.dumps({"workload": "square_256_uniform", "tflops": 1.0}) + "\n"
                   + json.dumps({"workload": "square_512_normal", "tflops": 2.0}) + "\n"
                   + '{"workload": "square_768_nor')          # a line cut off by an interrupted run
    left = [w.name for w in bench.sweep_plan(workloads.ALL, str(out))]
    assert "square_256_uniform" not in left and "square_512_normal" not in left
    assert "square_768_normal" in left
    assert left == [n for n in everything if n not in ("square_256_uniform", "square_512_normal")]
    assert bench.done_workloads(str(out)) == {"square_256_uniform", "square_512_normal"}


def test_sweep_check_flags_results_outside_the_bound():
    import numpy as np
    bench = _bench()
    import oracle
    from dense_fp32_gemm_03_gb300 import workloads
    A = workloads.matrix(24, 256, "normal", 5, 0)
    B = workloads.matrix(256, 40, "normal", 5, 1)
    ref, _ = oracle.sgemm_f64(A, B)
    good = ref.astype(np.float32)                       # the correctly rounded product
    r = bench.check_rows(good, A, B, 256)
    assert r["bound_ok"] and r["rows_checked"] == 24 and r["max_err_over_max_ref"] < 1e-7
    bad = good.copy()
    bad[3, 7] += 1e-3 * np.abs(ref).max()               # one element off by 1e-3 of the scale
    r = bench.check_rows(bad, A, B, 256)
    assert not r["bound_ok"] and r["max_err_over_max_ref"] > 5e-4
    nan = good.copy()
    nan[0, 0] = np.nan
    assert not bench.check_rows(nan, A, B, 256)["bound_ok"]
