"""Host-side checks of the measurement arithmetic (CPU only).

The throughput formula and the reuse models the kernels are sized with are
pinned to numbers the pages print (tests/golden/*.txt, each line cited there).
The multi-replica timing aggregation of bench.py runs as two gloo processes.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from dense_fp32_gemm_03_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [x.strip() for x in line.split("|")]


def _seconds(text):
    value, unit = text.split()
    return float(value) * {"us": 1e-6, "ms": 1e-3, "s": 1.0}[unit]


@pytest.mark.parametrize("row", list(_rows("throughput_accounting.txt")), ids=lambda r: f"{r[0]}-{r[1]}")
def test_throughput_formula_matches_printed_figures(row):
    _, n, t, printed = row
    n = int(n)
    w = workloads.Workload("square", n, n, n, "uniform", 0)
    tflops = w.flops / _seconds(t) / 1e12
    # The pages round their figures to one or two decimals.
    assert abs(tflops - float(printed)) < 0.06


def _ai(bm, bn, bk):
    return 2.0 * bm * bn * bk / (4.0 * (bm * bk + bk * bn))


@pytest.mark.parametrize("row", list(_rows("tile_models.txt")), ids=lambda r: f"{r[0]}-{r[1]}")
def test_reuse_models(row):
    kind, arg, expect = row
    if kind == "square_tile_ai":
        b = int(arg)
        assert _ai(b, b, 8) == pytest.approx(float(expect))
        assert _ai(b, b, 16) == pytest.approx(float(expect))  # independent of the k depth
    else:
        tm, tn = map(int, arg.split("x"))
        assert (tm + tn) / (tm * tn) == pytest.approx(float(expect))


def test_compulsory_bytes_and_peak_formula():
    w = workloads.SQUARE_4096
    assert w.flops == 2 * 4096 ** 3
    assert w.compulsory_bytes == 4 * 3 * 4096 ** 2
    # SMs x 128 FFMA per clock x 2 FLOP x clock
    assert bench.ffma_peak_tflops(152, 2070.0) == pytest.approx(80.54784)
    assert bench.aggregate(1e12, 2.0, 4) == pytest.approx(2.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    slowest = bench.max_over_ranks(times[rank], world)
    bench.barrier(world)
    out[rank] = bench.aggregate(10.0e12, slowest, world)
    dist.destroy_process_group()


def test_replica_timing_takes_the_slowest_rank_gloo():
    world, port = 2, _free_port()
    times = [1.0, 4.0]
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_replica, args=(world, port, times, out), nprocs=world, join=True,
                       start_method="spawn")
    # 2 replicas x 10 TFLOP over the slowest replica's 4 s
    assert out[0] == pytest.approx(5.0) and out[1] == pytest.approx(5.0)
