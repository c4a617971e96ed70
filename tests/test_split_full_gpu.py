"""Full-size parity where the Stream-K schedule splits tiles over CTAs.

Split tiles are where CTAs hand partial sums to each other, so they are
compared element by element at the configurations' full sizes:

* 1024 x 1024 x 16384 (long K): every tile is split, so the whole product is
  compared, through the selector, Stream-K on 128 x 256 tiles and Stream-K on
  128 x 128 tiles;
* 16384 x 1024 x 4096 (tall), 8192^3, 4096^3 and the sweep's 1536^3 and 2048^3
  (every tile split): whole tile-row blocks that hold
  split tiles.  The blocks are chosen from the schedule itself (plan_launch,
  read through tests/plan_probe.cpp): the test asserts that each block
  contains split tiles of the variant it runs.

Stream-K results are not bit-reproducible across schedules ("Beyond Kernel 7",
"What the result establishes"), so the check is the FP32 bound per element
and the pages' max|err|/max|ref| gate, not equality with another variant.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_fp32_gemm_03_gb300 as sg
from dense_fp32_gemm_03_gb300 import workloads

import plan_util
from parity import check_within_bound

pytestmark = pytest.mark.gpu

TILE = {sg.STREAMK: (128, 256), sg.STREAMK_SMALL: (128, 128), sg.SPECIALIZED: None}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not plan_util.available():
        pytest.skip("needs g++ and the CUDA headers for the schedule probe")
    import __graft_entry__
    __graft_entry__.build()
    yield
    st, site = sg.query_device_status()
    assert st == 0, f"device status {st} (site {site}) left after the module"


def _resident():
    # The tile kernels run one CTA per SM.
    return torch.cuda.get_device_properties(0).multi_processor_count


def _tile_of(variant, A, B, C):
    """(BM, BN) of the 16-deep tiles the variant runs for these operands."""
    if variant == sg.AUTO:
        variant = sg.select_variant(A, B, C)
    if variant == sg.SPECIALIZED:
        # The instance compiled for this shape: the tile whose plan it matches.
        M, K = A.shape
        N = B.shape[1]
        for tile in TILE.values():
            if tile and plan_util.plan(M, N, K, tile[0], tile[1], 16, _resident())["spec"] >= 0:
                return tile
        return None
    return TILE[variant]


def test_long_k_every_tile_split_full_compare():
    w = workloads.LONG_K
    A_h, B_h = workloads.operands(w)
    ref, E = oracle.sgemm_f64(A_h, B_h)
    A, B = A_h.cuda(), B_h.cuda()
    C = torch.empty(w.M, w.N, device="cuda")
    for v in (sg.AUTO, sg.STREAMK, sg.STREAMK_SMALL):
        tile = _tile_of(v, A, B, C)
        assert tile is not None
        p = plan_util.plan(w.M, w.N, w.K, tile[0], tile[1], 16, _resident())
        assert p["dp_tiles"] == 0 and p["sk_tiles"] == p["tiles_m"] * p["tiles_n"], p
        C.fill_(float("nan"))
        sg.sgemm(A, B, out=C, variant=v)
        torch.cuda.synchronize()
        check_within_bound(C.cpu().numpy(), ref, E, w.K, f"{w.name} variant {v} (full)")


SWEEP_LARGE = [s for s in workloads.SWEEP if s.M in (1536, 2048)]


@pytest.mark.parametrize("w", [workloads.TALL, workloads.SQUARE_8192, workloads.SQUARE_4096,
                               *SWEEP_LARGE], ids=lambda w: w.name)
@pytest.mark.parametrize("variant", [sg.AUTO, sg.STREAMK], ids=["auto", "streamk"])
def test_row_blocks_with_split_tiles(w, variant):
    A_h, B_h = workloads.operands(w)
    A, B = A_h.cuda(), B_h.cuda()
    C = torch.full((w.M, w.N), float("nan"), device="cuda")
    tile = _tile_of(variant, A, B, C)
    assert tile is not None
    bm, bn = tile
    p = plan_util.plan(w.M, w.N, w.K, bm, bn, 16, _resident())
    split = list(plan_util.split_tiles(p))
    assert split, f"{w.name}: the schedule splits no tile"
    # The tile rows of the first and the last split tile.
    rows_of_split = sorted({plan_util.tile_coords(p, t)[0] for t in split})
    blocks = sorted({rows_of_split[0], rows_of_split[-1]})
    sg.sgemm(A, B, out=C, variant=variant)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    assert np.all(np.isfinite(got)), f"{w.name}: tiles left unwritten"
    for tm in blocks:
        in_block = [t for t in split if plan_util.tile_coords(p, t)[0] == tm]
        assert in_block, (w.name, tm)
        rows = slice(tm * bm, min((tm + 1) * bm, w.M))
        ref, E = oracle.sgemm_f64(A_h[rows], B_h)
        check_within_bound(got[rows], ref, E, w.K,
                           f"{w.name} variant {variant} tile row {tm} ({len(in_block)} split tiles)")


# The owner of a split tile normally keeps its partial in registers and adds
# the other sharers' partials to it; with the test switch every sharer
# publishes and the last to arrive sums all partials from the workspace.  Both
# paths add the same partials in CTA order, so the results must be equal bit
# for bit.  The shapes cover both tile configurations, the size-specialized
# instances, ragged edges, up to five sharers of a tile (768^3) and the scaled
# epilogue.
SUM_PATHS = [((1024, 1024, 1024), sg.AUTO), ((1024, 1024, 1024), sg.STREAMK_SMALL),
             ((1024, 1024, 1024), sg.STREAMK), ((768, 768, 768), sg.AUTO),
             ((768, 768, 768), sg.STREAMK_SMALL), ((1000, 1100, 900), sg.STREAMK_SMALL),
             ((1000, 1100, 900), sg.STREAMK), ((1024, 1024, 16384), sg.STREAMK),
             ((4096, 4096, 4096), sg.AUTO)]


def _with_owner_publishing(fn):
    sg.debug_owner_publishes(True)
    try:
        return fn()
    finally:
        sg.debug_owner_publishes(False)


@pytest.mark.parametrize("shape,variant", SUM_PATHS,
                         ids=[f"{'x'.join(map(str, s))}-{sg.variant_name(v) if v >= 0 else 'auto'}"
                              for s, v in SUM_PATHS])
def test_split_tiles_summed_from_the_workspace_match_bit_for_bit(shape, variant):
    M, N, K = shape
    w = workloads.Workload(f"sumpath_{M}x{N}x{K}", M, N, K, "uniform", 2300 + M + K)
    A_h, B_h = workloads.operands(w)
    A, B = A_h.cuda(), B_h.cuda()
    C = torch.empty(M, N, device="cuda")
    tile = _tile_of(variant, A, B, C)
    assert tile is not None
    assert list(plan_util.split_tiles(plan_util.plan(M, N, K, tile[0], tile[1], 16, _resident()))), \
        "the schedule splits no tile"
    default = sg.sgemm(A, B, variant=variant)
    published = _with_owner_publishing(lambda: sg.sgemm(A, B, variant=variant))
    torch.cuda.synchronize()
    assert torch.equal(default, published)
    r, c = workloads.sample_indices(M, N, 2048, w.seed)
    ref, E = oracle.sgemm_entries_f64(A_h, B_h, r.numpy(), c.numpy())
    check_within_bound(published[r.cuda(), c.cuda()].cpu().numpy(), ref, E, K,
                       f"{w.name} variant {variant}, every partial from the workspace")


def test_split_tiles_summed_from_the_workspace_scaled_and_static():
    """The same equality through the scaled epilogue and the allocation-free entry point."""
    M = N = K = 1024
    w = workloads.Workload("sumpath_scaled_1024", M, N, K, "uniform", 2399)
    A_h, B_h = workloads.operands(w)
    A, B = A_h.cuda(), B_h.cuda()
    C0 = torch.randn(M, N, device="cuda")

    def scaled():
        C = C0.clone()
        sg.sgemm_ex(A, B, C, alpha=0.75, beta=-1.5)
        return C

    def static():
        C = torch.empty(M, N, device="cuda")
        st = sg.binding.sgemm_streamk_static_raw(M, N, K, A.data_ptr(), K, B.data_ptr(), N,
                                                 C.data_ptr(), N,
                                                 torch.cuda.current_stream().cuda_stream)
        assert st == 0, st
        return C

    for fn in (scaled, static):
        default = fn()
        published = _with_owner_publishing(fn)
        torch.cuda.synchronize()
        assert torch.equal(default, published), fn.__name__
