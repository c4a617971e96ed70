"""Phase traces of the tile kernel: where a launch's time goes, CTA by CTA.

The diagnostic library ``libsgemm_trace.so`` (``_build.build_trace()``) is the
product library with ``-DSGEMM_PHASE_TRACE``: every CTA of the tile kernel
writes %globaltimer stamps of its phases into a device buffer (record layout
in ``csrc/sgemm_trace.h``).  This module decodes such a buffer and reduces it
to the figures that explain a launch's duration:

* start latency: kernel entry to the first ring stage landing in shared memory;
* k-loop: time per k-tile of each unit of work, and the FFMA efficiency it
  implies at a given SM clock;
* epilogue: whole-tile stores, split-tile publishes, split-tile reductions;
* skew: spread of the CTAs' entry and exit times, and the time from the first
  entry to the last exit.

``python -m dense_fp32_gemm_03_gb300.phase_trace --m 1024 --n 1024 --k 1024``
runs one traced call on the current GPU (L2 flushed first, as the benchmark
does) and prints the breakdown.  Only this module loads the traced library;
the product never contains the trace.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import statistics
from dataclasses import dataclass, field

import numpy as np

# Record kinds (TraceKind in csrc/sgemm_trace.h).
(ENTRY, FIRST_STAGE, KLOOP_END, STORE_END, PUBLISH_END, REDUCE_END, EXIT, PRODUCER_ISSUED,
 OWNER_WAIT, PRODUCER_START, FIRST_A_LANDED, BARRIERS_READY, CTA_SYNCED) = range(1, 14)
SLOTS = 64            # records per CTA (kTraceSlots)
PRODUCER_SLOT0 = 56   # producer records start here (kTraceProducerSlot0)
FFMA_PER_CLK_PER_SM = 128


@dataclass
class Event:
    t: int      # global time, ns
    kind: int
    a: int
    b: int


@dataclass
class Unit:
    tile: int
    ktiles: int
    kloop_ns: int        # from the previous phase's end to the unit's last k-tile
    epilogue: str        # how the unit ended: "store", "publish" or "reduce"
    epilogue_ns: int     # from the last k-tile to the unit's end
    partials_read: int = 0
    wait_ns: int = 0     # the owner's wait for the other sharers (0: none)
    waited: bool | None = None   # True: they all arrived in time
    prefetched: bool = False     # their partials were prefetched into shared memory
    publish_ns: int = 0  # publishing this CTA's partial (0: not published)


@dataclass
class CtaTrace:
    cta: int
    sm: int
    entry: int
    first_stage: int | None
    exit: int | None
    producer_issued: int | None
    units: list[Unit] = field(default_factory=list)
    producer_start: int | None = None
    first_a_landed: int | None = None
    barriers_ready: int | None = None
    cta_synced: int | None = None


def decode(words: np.ndarray, ctas: int) -> list[list[Event]]:
    """Records of each CTA, in the order written (consumer records, then producer ones)."""
    w = np.asarray(words, dtype=np.uint64).reshape(-1)
    if w.size < ctas * SLOTS * 2:
        raise ValueError(f"buffer holds {w.size} words, {ctas} CTAs need {ctas * SLOTS * 2}")
    w = w[:ctas * SLOTS * 2].reshape(ctas, SLOTS, 2)
    out = []
    for c in range(ctas):
        ev = []
        for i in range(SLOTS):
            t, info = int(w[c, i, 0]), int(w[c, i, 1])
            kind = info >> 56
            if kind == 0:
                continue
            ev.append(Event(t, kind, (info >> 32) & 0xFFFFFF, info & 0xFFFFFFFF))
        out.append(ev)
    return out


def per_cta(events: list[list[Event]]) -> list[CtaTrace]:
    """Each CTA's phases: entry, first stage, units of work with their epilogues, exit."""
    traces = []
    for c, ev in enumerate(events):
        entry = next((e for e in ev if e.kind == ENTRY), None)
        if entry is None:
            continue
        first = next((e.t for e in ev if e.kind == FIRST_STAGE), None)
        prod = next((e.t for e in ev if e.kind == PRODUCER_ISSUED), None)
        ct = CtaTrace(c, entry.a, entry.t, first, None, prod,
                      producer_start=next((e.t for e in ev if e.kind == PRODUCER_START), None),
                      first_a_landed=next((e.t for e in ev if e.kind == FIRST_A_LANDED), None),
                      barriers_ready=next((e.t for e in ev if e.kind == BARRIERS_READY), None),
                      cta_synced=next((e.t for e in ev if e.kind == CTA_SYNCED), None))
        prev = first if first is not None else entry.t
        unit, mark = None, 0     # the unit in its epilogue, and the end of its last phase
        for e in ev:
            if e.kind == KLOOP_END:
                unit = Unit(e.a, e.b, e.t - prev, "", 0)
                mark = kend = e.t
            elif unit is None:
                if e.kind == EXIT:
                    ct.exit = e.t
                continue
            elif e.kind == OWNER_WAIT:
                unit.wait_ns, unit.waited, mark = unit.wait_ns + e.t - mark, bool(e.b), e.t
                unit.prefetched = unit.prefetched or e.b == 2
            elif e.kind == PUBLISH_END:
                unit.publish_ns, mark = e.t - mark, e.t
                if not e.b:      # not the last to arrive: the unit ends here
                    unit.epilogue, unit.epilogue_ns = "publish", e.t - kend
            elif e.kind in (STORE_END, REDUCE_END):
                unit.epilogue = "store" if e.kind == STORE_END else "reduce"
                unit.epilogue_ns = e.t - kend
                unit.partials_read = e.b if e.kind == REDUCE_END else 0
                mark = e.t
            if unit is not None and unit.epilogue:
                ct.units.append(unit)
                prev, unit = mark, None
            if e.kind == EXIT:
                ct.exit = e.t
        traces.append(ct)
    return traces


def _stats(xs):
    xs = list(xs)
    if not xs:
        return None
    return {"median": statistics.median(xs), "max": max(xs), "min": min(xs), "count": len(xs)}


def summarize(traces: list[CtaTrace], flops: float | None = None, mhz: float = 2070.0) -> dict:
    """The breakdown of one launch (times in microseconds).

    ``flops`` (2MNK) turns the k-loop time into an FFMA efficiency: the flops
    of one k-tile are flops / (k-tiles over all units), and an SM's peak is
    128 FFMA x 2 per clock at ``mhz``.
    """
    if not traces:
        raise ValueError("no CTA recorded an entry")
    t0 = min(t.entry for t in traces)
    us = 1e-3
    exits = [t.exit for t in traces if t.exit is not None]
    ktiles = sum(u.ktiles for t in traces for u in t.units)
    kloop_ns = sum(u.kloop_ns for t in traces for u in t.units)
    out = {
        "ctas": len(traces),
        "span_us": (max(exits) - t0) * us if exits else None,
        "entry_skew_us": (max(t.entry for t in traces) - t0) * us,
        "exit_skew_us": (max(exits) - min(exits)) * us if exits else None,
        "start_latency_us": _stats((t.first_stage - t.entry) * us for t in traces
                                   if t.first_stage is not None),
        "producer_issue_us": _stats((t.producer_issued - t.entry) * us for t in traces
                                    if t.producer_issued is not None),
        "barriers_ready_us": _stats((t.barriers_ready - t.entry) * us for t in traces
                                    if t.barriers_ready is not None),
        "cta_synced_us": _stats((t.cta_synced - t.entry) * us for t in traces
                                if t.cta_synced is not None),
        "producer_start_us": _stats((t.producer_start - t.entry) * us for t in traces
                                    if t.producer_start is not None),
        "first_a_landed_us": _stats((t.first_a_landed - t.entry) * us for t in traces
                                    if t.first_a_landed is not None),
        "ktiles": ktiles,
        "ktile_us": (kloop_ns / ktiles) * us if ktiles else None,
        "ktile_us_by_unit": _stats(u.kloop_ns / u.ktiles * us for t in traces for u in t.units
                                   if u.ktiles),
        "ktiles_per_cta": _stats(sum(u.ktiles for u in t.units) for t in traces),
        "units_per_cta": _stats(len(t.units) for t in traces),
    }
    for name in ("store", "publish", "reduce"):
        out[f"{name}_us"] = _stats(u.epilogue_ns * us for t in traces for u in t.units
                                   if u.epilogue == name)
    units = [u for t in traces for u in t.units]
    out["owner_wait_us"] = _stats(u.wait_ns * us for u in units if u.waited is not None)
    out["owner_waits"] = {"all_arrived": sum(1 for u in units if u.waited is True),
                          "timed_out": sum(1 for u in units if u.waited is False)}
    out["published_then_last"] = sum(1 for u in units if u.epilogue == "reduce" and u.publish_ns)
    out["prefetched"] = sum(1 for u in units if u.prefetched)
    # The CTA that exits last: its phases, relative to the first entry.
    out["critical_cta"] = None
    if exits:
        crit = max((t for t in traces if t.exit is not None), key=lambda t: t.exit)
        tl = [("entry", crit.entry)]
        mark = crit.entry
        if crit.first_stage is not None:
            tl.append(("first stage landed", crit.first_stage))
            mark = crit.first_stage
        for u in crit.units:
            mark += u.kloop_ns
            kend = mark
            tl.append((f"tile {u.tile}: {u.ktiles} k-tiles computed", mark))
            if u.waited is not None:
                mark += u.wait_ns
                tl.append((f"tile {u.tile}: owner wait, {'all arrived' if u.waited else 'timed out'}",
                           mark))
            if u.publish_ns:
                mark += u.publish_ns
                tl.append((f"tile {u.tile}: partial published", mark))
            if kend + u.epilogue_ns != mark:
                mark = kend + u.epilogue_ns
                tl.append((f"tile {u.tile}: {u.epilogue} done", mark))
        tl.append(("exit", crit.exit))
        out["critical_cta"] = {"cta": crit.cta, "sm": crit.sm,
                               "timeline": [(label, (t - t0) * us) for label, t in tl]}
    if flops and ktiles and kloop_ns:
        per_ktile_flop = flops / ktiles
        sm_peak = FFMA_PER_CLK_PER_SM * 2 * mhz * 1e6          # flop/s per SM
        out["ffma_efficiency_in_kloop"] = per_ktile_flop / (kloop_ns / ktiles * 1e-9) / sm_peak
    return out


def format_summary(s: dict) -> str:
    def st(name, unit="us"):
        v = s.get(name)
        if v is None:
            return f"{name:<22} -"
        return (f"{name:<22} median {v['median']:8.3f} {unit}  max {v['max']:8.3f}  "
                f"min {v['min']:8.3f}  n={v['count']}")
    lines = [
        f"CTAs {s['ctas']}, first entry to last exit {s['span_us']:.2f} us, "
        f"entry skew {s['entry_skew_us']:.2f} us, exit skew {s['exit_skew_us']:.2f} us",
        st("start_latency_us"), st("barriers_ready_us"), st("cta_synced_us"),
        st("producer_start_us"), st("producer_issue_us"),
        st("first_a_landed_us"),
        f"{'ktile_us (weighted)':<22} {s['ktile_us']:.4f} us over {s['ktiles']} k-tiles",
        st("ktile_us_by_unit"), st("ktiles_per_cta", ""), st("units_per_cta", ""),
        st("store_us"), st("publish_us"), st("reduce_us"),
    ]
    if s.get("owner_wait_us"):
        lines.append(st("owner_wait_us"))
    lines.append(f"owner waits: {s['owner_waits']['all_arrived']} all arrived, "
                 f"{s['owner_waits']['timed_out']} timed out; "
                 f"published then last: {s['published_then_last']}; "
                 f"partials prefetched: {s.get('prefetched', 0)}")
    if "ffma_efficiency_in_kloop" in s:
        lines.append(f"FFMA efficiency inside the k-loop: {100 * s['ffma_efficiency_in_kloop']:.1f} %")
    if s.get("critical_cta"):
        c = s["critical_cta"]
        lines.append(f"last CTA to exit: {c['cta']} (SM {c['sm']})")
        lines.extend(f"  {t:9.3f} us  {label}" for label, t in c["timeline"])
    return "\n".join(lines)


# ------------------------------------------------------------------ GPU run
def run_traced(M: int, N: int, K: int, variant: int = -1, warmup: int = 3, dist: str = "uniform",
               seed: int = 1010):
    """One traced call of the C ABI on the current GPU; returns the decoded CTA traces."""
    import torch

    from . import _build, workloads
    path = _build.build_trace()
    lib = ctypes.CDLL(path)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    lib.sgemm_variant.argtypes = [ctypes.c_int, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp]
    lib.sgemm_variant.restype = ctypes.c_int
    lib.sgemm_trace_configure.argtypes = [vp, i64]
    lib.sgemm_trace_configure.restype = ctypes.c_int
    lib.sgemm_query_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.sgemm_query_device_status.restype = ctypes.c_int
    dev = torch.device("cuda")
    A = workloads.matrix(M, K, dist, seed, 0).to(dev)
    B = workloads.matrix(K, N, dist, seed, 1).to(dev)
    C = torch.empty(M, N, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4, device=dev)
    max_ctas = 4096
    buf = torch.zeros(max_ctas * SLOTS * 2, dtype=torch.int64, device=dev)

    def call():
        st = lib.sgemm_variant(variant, M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                               stream)
        if st != 0:
            raise RuntimeError(f"sgemm_variant returned {st}")

    if lib.sgemm_trace_configure(None, 0) != 0:
        raise RuntimeError("sgemm_trace_configure failed")
    for _ in range(warmup):
        flush.fill_(1.0)
        call()
    torch.cuda.synchronize()
    if lib.sgemm_trace_configure(buf.data_ptr(), max_ctas) != 0:
        raise RuntimeError("sgemm_trace_configure failed")
    flush.fill_(1.0)
    call()
    torch.cuda.synchronize()
    lib.sgemm_trace_configure(None, 0)
    detail = ctypes.c_uint32(0)
    st = lib.sgemm_query_device_status(stream, ctypes.byref(detail))
    if st != 0:
        raise RuntimeError(f"device status {st} (site {detail.value}) after the traced call")
    words = buf.cpu().numpy().view(np.uint64)
    events = decode(words, max_ctas)
    ctas = max((i + 1 for i, ev in enumerate(events) if ev), default=0)
    return per_cta(events[:ctas])


def main(argv=None):
    p = argparse.ArgumentParser(description="phase trace of one tile-kernel launch")
    p.add_argument("--m", type=int, default=1024)
    p.add_argument("--n", type=int, default=1024)
    p.add_argument("--k", type=int, default=1024)
    p.add_argument("--variant", default="auto")
    p.add_argument("--mhz", type=float, default=2070.0)
    p.add_argument("--json", action="store_true")
    args = p.parse_args(argv)
    from .binding import VARIANTS
    variant = -1 if args.variant == "auto" else VARIANTS[args.variant]
    traces = run_traced(args.m, args.n, args.k, variant)
    s = summarize(traces, flops=2.0 * args.m * args.n * args.k, mhz=args.mhz)
    print(f"{args.m}x{args.n}x{args.k} variant {args.variant}")
    print(format_summary(s))
    if args.json:
        print(json.dumps(s))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
