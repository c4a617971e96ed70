"""Host test of the phase-trace reader on a synthetic buffer (no GPU).

The traced diagnostic library writes, per CTA, records of two 64-bit words
(global time in ns; kind << 56 | a << 32 | b) in fixed slots (consumer records
from slot 0, producer records from slot 56).  The buffer below is built by
hand with known phases, so every figure of the summary is known in advance.
"""
import numpy as np
import pytest

from dense_fp32_gemm_03_gb300 import phase_trace as pt


def _buffer(ctas, records):
    w = np.zeros((ctas, pt.SLOTS, 2), dtype=np.uint64)
    for (cta, slot), (t, kind, a, b) in records.items():
        w[cta, slot, 0] = t
        w[cta, slot, 1] = (kind << 56) | (a << 32) | b
    return w.reshape(-1)


RECORDS = {
    # CTA 0: entry on SM 5, a split tile published, then a split tile it reduces.
    (0, 0): (1000, pt.ENTRY, 5, 0),
    (0, 1): (3000, pt.FIRST_STAGE, 0, 0),
    (0, 2): (13000, pt.KLOOP_END, 3, 10),
    (0, 3): (14000, pt.PUBLISH_END, 3, 0),
    (0, 4): (19000, pt.KLOOP_END, 4, 5),
    (0, 5): (20500, pt.REDUCE_END, 4, 2),
    (0, 6): (20600, pt.EXIT, 0, 0),
    (0, pt.PRODUCER_SLOT0): (1500, pt.PRODUCER_ISSUED, 0, 0),
    # CTA 1: one whole tile.
    (1, 0): (1200, pt.ENTRY, 9, 0),
    (1, 1): (3100, pt.FIRST_STAGE, 0, 0),
    (1, 2): (23100, pt.KLOOP_END, 7, 20),
    (1, 3): (23600, pt.STORE_END, 7, 0),
    (1, 4): (23700, pt.EXIT, 0, 0),
    (1, pt.PRODUCER_SLOT0): (1800, pt.PRODUCER_ISSUED, 0, 0),
}


def test_decode_and_phases():
    words = _buffer(3, RECORDS)          # the third CTA recorded nothing
    events = pt.decode(words, 3)
    assert [len(e) for e in events] == [8, 6, 0]
    traces = pt.per_cta(events)
    assert [t.cta for t in traces] == [0, 1]
    t0, t1 = traces
    assert (t0.sm, t0.entry, t0.first_stage, t0.exit, t0.producer_issued) == (5, 1000, 3000, 20600, 1500)
    assert [(u.tile, u.ktiles, u.kloop_ns, u.epilogue, u.epilogue_ns, u.partials_read)
            for u in t0.units] == [(3, 10, 10000, "publish", 1000, 0), (4, 5, 5000, "reduce", 1500, 2)]
    assert [(u.tile, u.ktiles, u.kloop_ns, u.epilogue, u.epilogue_ns) for u in t1.units] == \
        [(7, 20, 20000, "store", 500)]


def test_summary_figures():
    traces = pt.per_cta(pt.decode(_buffer(2, RECORDS), 2))
    sm_peak = pt.FFMA_PER_CLK_PER_SM * 2 * 2000.0 * 1e6
    # 35 k-tiles of 1 us each at half the peak of a 2000 MHz SM.
    flops = 35 * 0.5 * sm_peak * 1e-6
    s = pt.summarize(traces, flops=flops, mhz=2000.0)
    assert s["ctas"] == 2
    assert s["span_us"] == pytest.approx(22.7)
    assert s["entry_skew_us"] == pytest.approx(0.2)
    assert s["exit_skew_us"] == pytest.approx(3.1)
    assert s["start_latency_us"]["max"] == pytest.approx(2.0)
    assert s["start_latency_us"]["min"] == pytest.approx(1.9)
    assert s["producer_issue_us"]["max"] == pytest.approx(0.6)
    assert s["ktiles"] == 35 and s["ktile_us"] == pytest.approx(1.0)
    assert s["ktiles_per_cta"]["max"] == 20 and s["units_per_cta"]["max"] == 2
    assert s["publish_us"]["median"] == pytest.approx(1.0)
    assert s["reduce_us"]["median"] == pytest.approx(1.5)
    assert s["store_us"]["median"] == pytest.approx(0.5)
    assert s["ffma_efficiency_in_kloop"] == pytest.approx(0.5)
    text = pt.format_summary(s)
    assert "first entry to last exit 22.70 us" in text and "50.0 %" in text


def test_short_buffer_rejected():
    with pytest.raises(ValueError):
        pt.decode(np.zeros(10, dtype=np.uint64), 1)


def test_owner_wait_and_publish_then_last():
    """An owner that waited in time reduces without publishing; a sharer that published
    and then found itself last reduces after its publish; the critical CTA's timeline."""
    rec = {
        (0, 0): (0, pt.ENTRY, 1, 0),
        (0, 1): (2000, pt.FIRST_STAGE, 0, 0),
        (0, 2): (12000, pt.KLOOP_END, 5, 10),
        (0, 3): (13000, pt.OWNER_WAIT, 5, 1),
        (0, 4): (15000, pt.REDUCE_END, 5, 2),
        (0, 5): (15100, pt.EXIT, 0, 0),
        (1, 0): (100, pt.ENTRY, 2, 0),
        (1, 1): (2100, pt.FIRST_STAGE, 0, 0),
        (1, 2): (14100, pt.KLOOP_END, 6, 12),
        (1, 3): (16100, pt.OWNER_WAIT, 6, 0),
        (1, 4): (17100, pt.PUBLISH_END, 6, 1),
        (1, 5): (19100, pt.REDUCE_END, 6, 3),
        (1, 6): (19200, pt.EXIT, 0, 0),
    }
    traces = pt.per_cta(pt.decode(_buffer(2, rec), 2))
    u0, u1 = traces[0].units[0], traces[1].units[0]
    assert (u0.epilogue, u0.wait_ns, u0.waited, u0.publish_ns, u0.epilogue_ns) == ("reduce", 1000, True, 0, 3000)
    assert (u1.epilogue, u1.wait_ns, u1.waited, u1.publish_ns, u1.epilogue_ns) == ("reduce", 2000, False, 1000, 5000)
    s = pt.summarize(traces)
    assert s["owner_waits"] == {"all_arrived": 1, "timed_out": 1}
    assert s["published_then_last"] == 1
    assert s["critical_cta"]["cta"] == 1
    times = [t for _, t in s["critical_cta"]["timeline"]]
    assert times == pytest.approx([0.1, 2.1, 14.1, 16.1, 17.1, 19.1, 19.2])
    assert "last CTA to exit: 1" in pt.format_summary(s)
