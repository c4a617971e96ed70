"""Host tests of the tile kernel's work decomposition (no GPU).

``plan_launch`` (csrc/sgemm_plan.h) cuts a product into BM x BN tiles and,
for the persistent schedule, fills whole waves of resident CTAs with whole
tiles and cuts the k-iterations of the remaining tiles evenly over the CTAs
(Stream-K, "Beyond Kernel 7: Closing the Gap to cuBLAS on an H100 FP32 GEMM",
section "Kernel 14").  The host API and the size-specialized kernels both
evaluate it, so an error here is an error on the GPU.  A small host program
(tests/plan_probe.cpp) prints its plans; the checks below restate the
decomposition's contract independently:

* tiles cover M x N and k-tiles cover K;
* whole tiles fill complete waves; the split tiles number fewer than a wave;
* the CTAs' Stream-K shares partition the split tiles' iteration stream;
* every (split tile, sharing CTA) pair has its own workspace slot
  (slot = tile + CTA) below the slot count the workspace is sized for.
"""
from __future__ import annotations

import pytest

import plan_util

K_MIN_SK_ITERS = 4  # kMinSkIters in sgemm_plan.h: shorter shares are not worth splitting


@pytest.fixture(scope="module")
def probe():
    if not plan_util.available():
        pytest.skip("needs g++ and the CUDA headers")
    return plan_util.plans


def ceil_div(a, b):
    return -(-a // b)


# The configurations' shapes, ragged and degenerate ones, and tile counts at
# and around the number of resident CTAs.
SHAPES = [
    (256, 256, 256), (512, 512, 512), (768, 768, 768), (1024, 1024, 1024), (1536, 1536, 1536),
    (2048, 2048, 2048), (4096, 4096, 4096), (8192, 8192, 8192), (1024, 1024, 16384),
    (16384, 1024, 4096), (1, 1, 1), (1, 1, 100000), (129, 257, 17), (1000, 1000, 1000),
    (4095, 4097, 4093), (4096, 4096, 16), (4096, 4096, 48), (128 * 8, 256 * 19, 512),
    (128 * 8, 256 * 19 + 1, 512), (128 * 16, 256 * 19, 4096), (65536, 32800, 65540),
]
TILES = [(128, 256, 16), (128, 128, 16)]
RESIDENT = [152, 148, 1, 7]


def cases():
    return [(M, N, K, bm, bn, bk, res, sk)
            for (M, N, K) in SHAPES for (bm, bn, bk) in TILES for res in RESIDENT
            for sk in (True, False)]


def share(p, c):
    """Iterations [start, end) of the Stream-K stream owned by CTA c (the documented rule)."""
    start = c * p["sk_base"] + min(c, p["sk_extra"])
    return start, start + p["sk_base"] + (1 if c < p["sk_extra"] else 0)


def test_tiles_cover_the_product(probe):
    cs = cases()
    for case, p in zip(cs, probe(cs)):
        M, N, K, bm, bn, bk, res, sk = case
        assert p["ok"] == 1, case
        assert (p["tiles_m"], p["tiles_n"], p["ipt"]) == (ceil_div(M, bm), ceil_div(N, bn),
                                                          ceil_div(K, bk)), case
        assert p["group_m"] >= 1, case


def test_one_tile_per_cta_schedule(probe):
    cs = [c for c in cases() if not c[7]]
    for case, p in zip(cs, probe(cs)):
        tiles = p["tiles_m"] * p["tiles_n"]
        assert (p["dp_tiles"], p["sk_tiles"], p["grid"], p["slots"]) == (tiles, 0, tiles, 0), case


def test_stream_k_waves_and_shares(probe):
    cs = [c for c in cases() if c[7]]
    for case, p in zip(cs, probe(cs)):
        res = case[6]
        tiles = p["tiles_m"] * p["tiles_n"]
        assert p["dp_tiles"] + p["sk_tiles"] == tiles, case
        assert p["dp_tiles"] % res == 0 and p["sk_tiles"] < res, case
        assert p["grid"] <= res, case
        if p["sk_tiles"] == 0:
            assert p["slots"] == 0 and p["grid"] == min(tiles, res), case
            continue
        total = p["sk_tiles"] * p["ipt"]
        assert p["sk_tiles"] <= p["sk_ctas"] <= res, case
        assert 0 <= p["sk_extra"] < p["sk_ctas"], case
        assert p["sk_base"] * p["sk_ctas"] + p["sk_extra"] == total, case
        # Shares are never shorter than the splitting threshold unless every
        # split tile has a CTA of its own.
        assert p["sk_base"] >= K_MIN_SK_ITERS or p["sk_ctas"] == p["sk_tiles"], case
        # CTAs beyond the Stream-K sharers exist only to run whole-tile waves.
        assert p["grid"] == (res if p["dp_tiles"] > 0 else p["sk_ctas"]), case
        # The shares partition [0, total) in CTA order.
        pos = 0
        for c in range(p["sk_ctas"]):
            start, end = share(p, c)
            assert start == pos and end > start, (case, c)
            pos = end
        assert pos == total, case


def test_split_tiles_have_distinct_slots(probe):
    cs = [c for c in cases() if c[7]]
    for case, p in zip(cs, probe(cs)):
        if p["sk_tiles"] == 0:
            continue
        ipt = p["ipt"]
        used = set()
        for c in range(p["sk_ctas"]):
            start, end = share(p, c)
            first_tile, last_tile = start // ipt, (end - 1) // ipt
            for t in range(first_tile, last_tile + 1):
                kb = max(start, t * ipt) - t * ipt
                ke = min(end, (t + 1) * ipt) - t * ipt
                if kb == 0 and ke == ipt:
                    continue  # a whole tile inside the share: written straight to C
                slot = t + c
                assert slot < p["slots"], (case, t, c)
                assert slot not in used, (case, t, c)
                used.add(slot)


# The size-specialized instances (kSpecShapes in sgemm_plan.h): shape and tile.
SPECIALIZED = [((4096, 4096, 4096), (128, 256)), ((1024, 1024, 1024), (128, 128)),
               ((768, 768, 768), (128, 128))]


def test_specialized_instance_needs_the_compiled_sm_count(probe):
    """The selector takes a size-specialized instance only when the device runs exactly the
    152 CTAs its schedule was compiled for; any other SM count x CTAs per SM falls back."""
    cs = [(M, N, K, bm, bn, 16, res, True)
          for (M, N, K), (bm, bn) in SPECIALIZED for res in (152, 148, 144, 160, 304, 76, 1)]
    for case, p in zip(cs, probe(cs)):
        M, N, K, bm, bn, bk, res, sk = case
        want = [s for s, _ in SPECIALIZED].index((M, N, K)) if res == 152 else -1
        assert p["spec"] == want, case


def test_specialized_instance_only_for_its_shape_and_tile(probe):
    cs = [(4096, 4096, 4092, 128, 256, 16, 152, True), (1024, 1024, 2048, 128, 128, 16, 152, True),
          (1024, 1024, 1024, 128, 256, 16, 152, True), (4096, 4096, 4096, 128, 128, 16, 152, True),
          (2048, 2048, 2048, 128, 256, 16, 152, False), (1023, 1024, 1024, 128, 128, 16, 152, True),
          (2048, 2048, 2048, 128, 256, 16, 152, True), (1536, 1536, 1536, 128, 256, 16, 152, True)]
    for case, p in zip(cs, probe(cs)):
        assert p["spec"] == -1, case
