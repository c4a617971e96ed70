"""Benchmark of the FP32 GEMM C ABI on GB300: one JSON line per run.

A step is one call of the C-ABI ``sgemm`` (the whole hot path: variant
selection, the TMA/FFMA tile kernel and, where the schedule splits tiles, the
in-kernel Stream-K fix-up) on the square 4096 x 4096 x 4096 FP32 problem
with i.i.d. uniform[-1, 1] inputs, already resident in HBM.  L2 is flushed
before every timed step by writing a buffer twice the L2 size, and every step
is timed with CUDA events on the launching stream (the flush is outside the
events), as in "Beyond Kernel 7", section "The confirmed result".
Throughput counts 2*M*N*K operations per call (an FFMA counts as two).
At 1024^3 and 4096^3 (and the sweep's 768^3) the selector
takes a size-specialized kernel instance (shape and schedule compiled in); the
best generic variant is timed on the same protocol and reported beside it
under ``generic``.

Also reported: the same metric end to end through the C-ABI call with host
buffers, ``sgemm_host`` (pinned A, B and C; the host-to-device copies of A and
B and the device-to-host copy of C happen inside each timed call, overlapped
with the multiply in row panels), the 1024^3 problem as a secondary figure, the
roofline position of the tile kernel against the FP32 FFMA peak
(SMs x 128 FFMA/clk x 2 FLOP x clock), and the CPU oracle timed on a bounded
row sample of the same problem on the host cores.

``--impl reference`` times only the oracle (a plain float64 triple loop on the
host cores) on the same workload and metric.  ``--gpus N`` under torchrun
runs N independent replicas (the product does not shard across GPUs).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP32 SGEMM TFLOPS (and % of GB300 FFMA peak) at n=1024/4096"
UNIT = "TFLOP/s"
FFMA_PER_CLK_PER_SM = 128  # FP32 lanes per SM: one FFMA each per clock


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="square_4096_uniform")
    p.add_argument("--variant", default="auto",
                   help="kernel variant of the timed device steps (the end-to-end figure goes "
                        "through sgemm_host, which always lets the selector choose)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target host time of the oracle sample")
    p.add_argument("--sweep", action="store_true",
                   help="one JSON line per workload of the configuration list (not the default line)")
    p.add_argument("--sweep-cpu-seconds", type=float, default=2.0,
                   help="host time of each oracle sample in --sweep (0: no oracle timing)")
    p.add_argument("--out", default=None,
                   help="--sweep: append each line to this file and skip workloads it already holds")
    return p.parse_args(argv)


# ------------------------------------------------------------------ distribution
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of ``x`` over all ranks (timing: the slowest replica decides)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_flops: float, max_seconds: float, world: int) -> float:
    """Whole-job throughput: the work of all replicas over the slowest replica's time."""
    return per_rank_flops * world / max_seconds / 1e12


# ------------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# -------------------------------------------------------------------- GPU timing
def time_steps(fn, steps, warmup, flush=None, stream=None):
    """Per-step device times (ms) of ``fn`` with CUDA events on ``stream``; ``flush`` runs
    before each step outside the events."""
    import torch
    stream = stream or torch.cuda.current_stream()
    for _ in range(warmup):
        if flush:
            flush()
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        if flush:
            flush()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def ffma_peak_tflops(sms: int, mhz: float) -> float:
    return sms * FFMA_PER_CLK_PER_SM * 2 * mhz * 1e6 / 1e12


# The files the tile kernel is compiled from, in a fixed order.
KERNEL_SOURCES = ("sgemm_tile.cu", "sgemm_sched.cuh", "sgemm_device.cuh", "sgemm_plan.h")


def kernel_source_digest() -> str:
    """SHA-256 over the tile kernel's sources: profile counters apply only to this exact kernel."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "dense_fp32_gemm_03_gb300", "csrc", name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def measured_traffic(workload: str):
    """DRAM bytes per launch of the tile kernel on ``workload`` from the committed ncu
    summary, or None when there is none or the kernel source changed since it was taken."""
    import re
    path = os.path.join(ROOT, "profiles", f"tile_kernel_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    digest = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    traffic = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not digest or not traffic or digest.group(1) != kernel_source_digest():
        return None
    return float(traffic.group(1))


# ------------------------------------------------------------ sweep checking
U24 = 2.0 ** -24
PAGES_GATE = 1e-4  # max|err| / max|ref| ("Beyond Kernel 7", "What the result establishes")


def check_rows(C_rows, A_rows, B, K):
    """The sweep's correctness figures for a block of rows of C against the oracle:
    max relative error (over C_ref != 0), max|err| / max|ref| and whether every element
    is within 4 K 2^-24 sum_k |a b| and the pages' gate holds."""
    import numpy as np
    import oracle
    ref, E = oracle.sgemm_f64(A_rows, B)
    got = np.asarray(C_rows, dtype=np.float64)
    err = np.abs(got - ref)
    nz = np.abs(ref) > 0
    max_rel = float((err[nz] / np.abs(ref[nz])).max()) if np.any(nz) else 0.0
    ref_max = float(np.abs(ref).max()) if ref.size else 0.0
    norm = float(err.max()) / ref_max if ref_max > 0 else 0.0
    ok = bool(np.all(np.isfinite(got)) and np.all(err <= 4.0 * K * U24 * E) and norm < PAGES_GATE)
    return {"max_rel_err": max_rel, "max_err_over_max_ref": norm, "bound_ok": ok,
            "rows_checked": int(got.shape[0])}


def done_workloads(path):
    """Workload names already in a sweep output file (missing file: none)."""
    done = set()
    try:
        with open(path) as f:
            for line in f:
                try:
                    rec = json.loads(line)
                except ValueError:
                    continue  # a line cut short by an interrupted run
                if isinstance(rec, dict) and "workload" in rec:
                    done.add(rec["workload"])
    except OSError:
        pass
    return done


def sweep_plan(workloads_all, out_path):
    """The sweep's workloads that still need a line (resume: skip those in out_path)."""
    done = done_workloads(out_path) if out_path else set()
    return [w for w in workloads_all if w.dist != "int8range" and w.name not in done]


def cpu_baseline(w, A, B, seconds: float, threads: int = 0):
    """Time the oracle (as it stands) on a bounded row sample of the workload, on all
    the host cores it may use (threads <= 0) or on `threads` of them."""
    import oracle
    all_cores = oracle.max_threads()
    if threads > 0:
        oracle.set_threads(threads)
    try:
        return _cpu_sample(w, A, B, seconds, oracle)
    finally:
        oracle.set_threads(all_cores)


def _cpu_sample(w, A, B, seconds, oracle):
    cores = oracle.max_threads()
    rows = max(1, min(w.M, cores))
    t0 = time.perf_counter()
    oracle.sgemm_f64(A[:rows], B, with_abs=False)
    dt = time.perf_counter() - t0
    rows2 = int(min(w.M, max(rows, rows * seconds / max(dt, 1e-6))))
    rows2 = max(rows, (rows2 // cores) * cores) if rows2 >= cores else rows2
    # A product small enough to finish well inside the budget is repeated.
    reps = max(1, int(seconds / max(dt * rows2 / rows, 1e-6))) if rows2 == w.M else 1
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.sgemm_f64(A[:rows2], B, with_abs=False)
    total = time.perf_counter() - t0
    dt2 = total / reps
    flops = 2.0 * rows2 * w.N * w.K
    rep_note = f", {reps} repetitions" if reps > 1 else ""
    return {"value": flops / dt2 / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"rows 0..{rows2 - 1} of the {w.M}x{w.N}x{w.K} product ({rows2}x{w.N} outputs, "
                      f"float64 triple loop{rep_note}, {total:.1f} s)",
            "seconds": total, "rows": rows2}


# ------------------------------------------------------------------------- arms
def run_reference(args):
    """The oracle alone, on the host cores, on the same workload and metric."""
    from dense_fp32_gemm_03_gb300 import workloads
    import oracle
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = workloads.BY_NAME[args.workload]
    A, B = workloads.operands(w)
    cores = oracle.max_threads()
    # Rows per step sized so that warm-up plus all steps take a few minutes at most.
    rows = cores
    t0 = time.perf_counter()
    oracle.sgemm_f64(A[:rows], B, with_abs=False)
    one = time.perf_counter() - t0
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(w.M, rows * budget / max(one, 1e-6))))
    times = []
    for i in range(args.warmup + args.steps):
        r0 = (i * rows) % max(1, w.M - rows + 1)
        t0 = time.perf_counter()
        oracle.sgemm_f64(A[r0:r0 + rows], B, with_abs=False)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    per_step = sum(times) / len(times)
    value = 2.0 * rows * w.N * w.K / per_step / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded uniform[-1,1])",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
                   "step": f"{rows} rows of C ({rows}x{w.N} outputs) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows} rows of the {w.M}x{w.N}x{w.K} product per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_workload(w, args, sg, device, flush, variant):
    import torch
    from dense_fp32_gemm_03_gb300 import workloads
    A_h, B_h = workloads.operands(w)
    A = A_h.to(device)
    B = B_h.to(device)
    C = torch.empty((w.M, w.N), device=device)
    stream = torch.cuda.current_stream(device)
    lda, ldb, ldc = w.K, w.N, w.N

    def step():
        st = sg.sgemm_raw(w.M, w.N, w.K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc,
                          stream.cuda_stream, variant)
        if st != 0:
            raise RuntimeError(f"sgemm failed: {sg.status_string(st)}")

    times = time_steps(step, args.steps, args.warmup, flush, stream)
    chosen = sg.select_variant(A, B, C) if variant == sg.AUTO else variant
    return A_h, B_h, A, B, C, times, chosen


def generic_figure(w, args, sg, device, flush, chosen):
    """When the selector took the size-specialized instance, the best of the generic
    pipelined variants on the same workload and protocol, reported beside it."""
    if chosen != sg.SPECIALIZED:
        return None
    import argparse
    sub = argparse.Namespace(**vars(args))
    sub.steps, sub.warmup = max(3, min(args.steps, 50)), 3
    best = None
    for v in (sg.STREAMK, sg.STREAMK_SMALL, sg.TILED, sg.TILED_SMALL):
        *_, times, _ = bench_workload(w, sub, sg, device, flush, v)
        us = statistics.median(times) * 1e3
        if best is None or us < best[1]:
            best = (v, us)
    return {"variant": sg.variant_name(best[0]), "value": w.flops / (best[1] * 1e-6) / 1e12,
            "unit": UNIT, "us_median": best[1], "steps": sub.steps}


def _host_call(sg, w, A_pin, B_pin, C_pin, stream):
    """One C-ABI sgemm_host call: A, B and C in (pinned) host memory, copies inside."""
    st = sg.load().sgemm_host(w.M, w.N, w.K, A_pin.data_ptr(), w.K, B_pin.data_ptr(), w.N,
                              C_pin.data_ptr(), w.N, stream.cuda_stream)
    if st != 0:
        raise RuntimeError(f"sgemm_host failed: {sg.status_string(st)}")


def e2e_pipelined(w, sg, device, A_h, B_h, steps, warmup, streams=3):
    """Seconds for ``steps`` end-to-end steps, each one C-ABI ``sgemm_host`` call on pinned
    host buffers (the library copies A and B in, multiplies and copies C out, overlapping
    the copies with the multiply inside the call).  Calls go round-robin over ``streams``
    streams, each with its own device staging, so one call's copies also overlap another
    call's multiply."""
    import torch
    A_pin, B_pin = A_h.pin_memory(), B_h.pin_memory()
    C_pin = [torch.empty((w.M, w.N), dtype=torch.float32).pin_memory() for _ in range(streams)]
    ss = [torch.cuda.Stream(device) for _ in range(streams)]
    for i in range(max(warmup, streams)):       # every stream's staging allocated untimed
        _host_call(sg, w, A_pin, B_pin, C_pin[i % streams], ss[i % streams])
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(ss[0])
    for s in ss[1:]:
        s.wait_event(start)
    for i in range(steps):
        _host_call(sg, w, A_pin, B_pin, C_pin[i % streams], ss[i % streams])
    for s in ss[1:]:
        ss[0].wait_stream(s)
    end.record(ss[0])
    torch.cuda.synchronize(device)
    return start.elapsed_time(end) / 1e3


def e2e_per_call(w, sg, device, A_h, B_h, calls, warmup):
    """Per-call latency (microseconds) of one C-ABI ``sgemm_host`` call at a time on one
    stream (pinned host A, B and C; the copies in and out happen inside the call),
    bracketed by CUDA events on that stream."""
    import torch
    A_pin, B_pin = A_h.pin_memory(), B_h.pin_memory()
    C_pin = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()
    s = torch.cuda.Stream(device)
    times = []
    for i in range(warmup + calls):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        _host_call(sg, w, A_pin, B_pin, C_pin, s)
        e1.record(s)
        s.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1) * 1e3)
    return times


def cublas_context(w, device, flush, steps=20):
    """torch.matmul with TF32 disabled (FP32 arithmetic) on the same inputs and protocol:
    a same-run context figure, as the pages compare against cuBLAS."""
    import torch
    from dense_fp32_gemm_03_gb300 import workloads
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        A_h, B_h = workloads.operands(w)
        A, B = A_h.to(device), B_h.to(device)
        C = torch.empty((w.M, w.N), device=device)
        times = time_steps(lambda: torch.matmul(A, B, out=C), steps, 3, flush)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return w.flops / (statistics.median(times) * 1e-3) / 1e12


def measured_peaks():
    """MEASURED_PEAKS.json (driver-written on the GPU pool), or {} when absent."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def tf32_mode(w, sg, device, flush, steps=30):
    """The opt-in TF32 tensor-core mode on the same workload, reported apart from FP32.

    Its roofline is the tensor pipe: peak = measured dense bf16 (burst) x the nominal
    TF32/bf16 ratio 1.1/2.25 PFLOP/s, or 1.9 PFLOP/s x that ratio when no measurement exists.
    """
    import torch
    from dense_fp32_gemm_03_gb300 import workloads
    A_h, B_h = workloads.operands(w)
    A, B = A_h.to(device), B_h.to(device)
    C = torch.empty((w.M, w.N), device=device)
    times = time_steps(lambda: sg.sgemm_tf32(A, B, out=C), steps, 3, flush)
    value = w.flops / (statistics.mean(times) * 1e-3) / 1e12
    bf16 = measured_peaks().get("bf16_tflops")
    peak = (bf16 if bf16 else 1900.0) * (1.1 / 2.25)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        ctx = time_steps(lambda: torch.matmul(A, B, out=C), steps, 3, flush)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return {"workload": w.name, "value": value, "unit": UNIT,
            "us_median": statistics.median(times) * 1e3,
            "roofline": {"bound": "tensor", "achieved": value, "peak": peak, "unit": UNIT,
                         "frac": value / peak,
                         "peak_basis": ("measured bf16 burst" if bf16 else "fallback 1.9 PFLOP/s bf16")
                         + " x 1.1/2.25 (nominal TF32/bf16)"},
            "tolerance": "(2^-8 + 4K 2^-24) sum|ab| per element (TF32 inputs)",
            "context_cublas_tf32_tflops": w.flops / (statistics.median(ctx) * 1e-3) / 1e12,
            "note": "separate mode with TF32 numerics; not part of the FP32 value"}


def run_ours(args):
    import torch
    import dense_fp32_gemm_03_gb300 as sg
    from dense_fp32_gemm_03_gb300 import workloads

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    from dense_fp32_gemm_03_gb300 import _build
    _build.build()
    sg.load()
    variant = sg.AUTO if args.variant == "auto" else sg.VARIANTS[args.variant]

    props = torch.cuda.get_device_properties(device)
    sms = props.multi_processor_count
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush_buf = torch.empty(2 * l2 // 4, dtype=torch.float32, device=device)

    def flush():
        flush_buf.fill_(1.0)

    if args.sweep:
        for w in sweep_plan(workloads.ALL, args.out):
            with ClockSampler(local) as clocks:
                A_h, B_h, _, _, C, times, chosen = bench_workload(w, args, sg, device, flush, variant)
            clock = clocks.summary()
            ms = statistics.median(times)
            line = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
                    "variant": sg.variant_name(chosen), "us_median": ms * 1e3,
                    "us_p10": sorted(times)[len(times) // 10] * 1e3,
                    "us_p90": sorted(times)[(9 * len(times)) // 10] * 1e3,
                    "tflops": w.flops / (ms * 1e-3) / 1e12,
                    "clocks": {"sm_mhz": clock["sm_mhz"], "sm_max_mhz": clock["sm_max_mhz"],
                               "reasons": clock["reasons"], "samples": clock["samples"]}}
            if args.sweep_cpu_seconds > 0 and rank == 0:
                # The oracle on the host cores, a reported baseline only: all cores for
                # every workload, one core as well up to 1024^3.
                cpu = {"all_cores": cpu_baseline(w, A_h, B_h, args.sweep_cpu_seconds)}
                if max(w.M, w.N, w.K) <= 1024:
                    cpu["one_core"] = cpu_baseline(w, A_h, B_h, args.sweep_cpu_seconds, threads=1)
                line["cpu_oracle"] = {k: {"tflops": v["value"], "cores": v["cores"], "sample": v["sample"],
                                          "rows": v["rows"]}
                                      for k, v in cpu.items()}
            if rank == 0:
                # The result of the last timed call, checked against the oracle on the
                # last rows of C (the grouped raster puts the Stream-K split tiles
                # last): as many rows as the oracle's timing sample took, or about
                # 2 GFLOP of oracle work when it did not run; at least 8.
                rows = line.get("cpu_oracle", {}).get("all_cores", {}).get("rows") or 0
                rows = max(8, min(w.M, rows or int(2e9 / (2.0 * w.N * w.K))))
                C_h = C[w.M - rows:].cpu().numpy()
                line.update(check_rows(C_h, A_h[w.M - rows:], B_h, w.K))
            text = json.dumps(line)
            print(text, flush=True)
            if args.out and rank == 0:
                with open(args.out, "a") as f:
                    f.write(text + "\n")
        return 0

    w = workloads.BY_NAME[args.workload]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        A_h, B_h, A, B, C, times, chosen = bench_workload(w, args, sg, device, flush, variant)
    barrier(world)
    torch.cuda.synchronize()
    total_s = sum(times) / 1e3
    max_total = max_over_ranks(total_s, world, device)
    mean_ms = max_total / args.steps * 1e3
    value = aggregate(w.flops * args.steps, max_total, world)
    clock = clocks.summary()

    # Roofline of the tile kernel: one launch per step, so the event time is its duration.
    kernel_tflops = w.flops / (statistics.mean(times) * 1e-3) / 1e12
    peak_max = ffma_peak_tflops(sms, clock["sm_max_mhz"] or 2070.0)
    peak_run = ffma_peak_tflops(sms, clock["sm_mhz"]) if clock["sm_mhz"] else None
    traffic = measured_traffic(w.name)

    # End to end through the C-ABI call with host buffers (sgemm_host): every step
    # copies its inputs in, multiplies and copies C out, inside the call.  Steps go
    # round-robin over three streams, so one step's copies also overlap another's
    # multiply.
    e2e_steps = max(3, min(args.steps, 40))
    e2e_total = e2e_pipelined(w, sg, device, A_h, B_h, e2e_steps, warmup=3)
    e2e_total = max_over_ranks(e2e_total, world, device)
    e2e_value = aggregate(w.flops * e2e_steps, e2e_total, world)
    # The same call one at a time on one stream (its own copies still overlap its
    # multiply, panel by panel).
    lat = e2e_per_call(w, sg, device, A_h, B_h, calls=max(3, min(args.steps, 20)), warmup=2)
    lat_us = max_over_ranks(statistics.median(lat), world, device)

    # Secondary size (n = 1024) on the same device.
    w2 = workloads.SQUARE_1024
    *_, times2, chosen2 = bench_workload(w2, args, sg, device, flush, variant)
    t2 = max_over_ranks(sum(times2) / 1e3, world, device)
    value2 = aggregate(w2.flops * args.steps, t2, world)

    # The size-specialized instances are reported apart from the generic kernel.
    generic = generic_figure(w, args, sg, device, flush, chosen)
    generic2 = generic_figure(w2, args, sg, device, flush, chosen2)

    context = {"cublas_fp32_tflops": {w.name: cublas_context(w, device, flush),
                                      w2.name: cublas_context(w2, device, flush)},
               "note": "torch.matmul, TF32 disabled, same flush protocol; context only"}

    tf32 = tf32_mode(w, sg, device, flush)

    status, site = sg.query_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} at wait site {site}")

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded uniform[-1,1], generated on the host)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "layout": "row-major",
                   "variant": sg.variant_name(chosen), "l2": "flushed before each step (2x L2 write)",
                   "us_median": statistics.median(times) * 1e3,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "generic": generic,
        "pct_ffma_peak": {"at_max_clock": 100 * kernel_tflops / peak_max,
                          "at_measured_clock": (100 * kernel_tflops / peak_run) if peak_run else None},
        "roofline": {"bound": "alu", "achieved": kernel_tflops, "peak": peak_max, "unit": UNIT,
                     "frac": kernel_tflops / peak_max, "traffic": traffic,
                     "peak_basis": f"{sms} SMs x {FFMA_PER_CLK_PER_SM} FFMA/clk x 2 x "
                                   f"{clock['sm_max_mhz'] or 2070.0:.0f} MHz (max SM clock)",
                     "peak_at_measured_clock": peak_run},
        "secondary": {"workload": w2.name, "value": value2, "unit": UNIT,
                      "variant": sg.variant_name(chosen2),
                      "us_median": statistics.median(times2) * 1e3, "generic": generic2},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 4 * (w.M * w.K + w.K * w.N),
                "d2h_bytes_per_step": 4 * w.M * w.N,
                "api": "sgemm_host (C ABI, pinned host A, B, C; copies inside the call)",
                "pipelining": "row panels inside each call; calls round-robin over 3 streams",
                "per_call": {"us_median": lat_us, "value": w.flops / (lat_us * 1e-6) / 1e12,
                             "unit": UNIT, "calls": len(lat),
                             "what": "one sgemm_host call at a time on one stream: H2D of B, "
                                     "then A and the multiply and the D2H of C in row panels"}},
        "context": context,
        "tf32_mode": tf32,
        "gpu_launches": args.steps,
        "clocks": {"sm_mhz": clock["sm_mhz"], "sm_max_mhz": clock["sm_max_mhz"],
                   "reasons": clock["reasons"], "samples": clock["samples"]},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = {k: v for k, v in cpu_baseline(w, A_h, B_h, args.cpu_seconds).items()
                                if k not in ("seconds", "rows")}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
