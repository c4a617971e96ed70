"""Shared pytest configuration: the ``gpu`` marker and the repo root on sys.path."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled extension")


def pytest_terminal_summary(terminalreporter):
    """Report the maximum relative error of every FP32 parity check that ran.

    The relative error max |C_gpu - C_ref| / |C_ref| (over elements with
    C_ref != 0) is reported, not bounded: near-cancelling sums make it large
    while the per-element bound holds.  Beside it, the pages' metric
    max |err| / max |ref|, which every check asserts below 1e-4.
    """
    parity = sys.modules.get("parity")
    report = getattr(parity, "REPORT", None)
    if not report:
        return
    tr = terminalreporter
    tr.section("FP32 parity: maximum relative error per check")
    for what, rel, norm in report:
        tr.write_line(f"{what[:70]:<70} max rel {rel:9.3e}   max|err|/max|ref| {norm:9.3e}")
    worst = max(report, key=lambda r: r[2])
    tr.write_line(f"{len(report)} checks; largest max|err|/max|ref| {worst[2]:.3e} ({worst[0]})")
