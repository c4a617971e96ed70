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
