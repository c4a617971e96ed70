"""GPU parity of sgemm_host: C = A * B with A, B and C in host memory.

The library copies B, then A in row panels, multiplies each panel as its rows
land and copies C's panels back (include/sgemm.h).  Every check compares with
the CPU oracle: per element within the FP32 bound for random inputs, exactly
for integer-valued ones.  Shapes cover one panel, several panels with a ragged
last one, ragged K and N (device pitches rounded up to 4 floats), strided host
views, pageable memory, K == 0, two streams at once and staging regrowth.
"""
import os

import pytest
import torch

import oracle
import dense_fp32_gemm_03_gb300 as sg
from dense_fp32_gemm_03_gb300 import workloads

from parity import check_exact, check_within_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    yield
    st, site = sg.query_device_status()
    assert st == 0, f"device status {st} (site {site}) left after the module"


def _operands(M, N, K, seed, dist="uniform"):
    w = workloads.Workload(f"host_{M}x{N}x{K}", M, N, K, dist, seed)
    return workloads.operands(w)


# (M, N, K): one panel; ragged K and N; two panels with a ragged last one; four
# panels (M = 4096) with ragged N; a K that is not a multiple of 4 across panels.
SHAPES = [(256, 256, 256), (1000, 1100, 900), (2050, 1030, 520), (4096, 640, 384),
          (2304, 769, 1023)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_pinned_against_oracle(shape):
    M, N, K = shape
    A, B = _operands(M, N, K, 3100 + M + K)
    ref, E = oracle.sgemm_f64(A, B)
    C = sg.sgemm_host(A.pin_memory(), B.pin_memory())
    check_within_bound(C.numpy(), ref, E, K, f"sgemm_host {M}x{N}x{K}")


def test_integer_inputs_exact_across_panels():
    M, N, K = 4096, 256, 512                  # four panels
    A = workloads.matrix(M, K, "int8range", 3201, 0)
    B = workloads.matrix(K, N, "int8range", 3201, 1)
    ref, E = oracle.sgemm_f64(A, B)
    assert E.max() < 2 ** 24
    C = sg.sgemm_host(A.pin_memory(), B.pin_memory())
    check_exact(C.numpy(), ref, "sgemm_host integer 4096x256x512")


@pytest.mark.parametrize("panels", ["1", "3", "8"])
def test_panel_count_does_not_change_the_result_beyond_the_bound(panels):
    M, N, K = 2048, 512, 640
    A, B = _operands(M, N, K, 3301)
    ref, E = oracle.sgemm_f64(A, B)
    old = os.environ.get("SGEMM_HOST_PANELS")
    os.environ["SGEMM_HOST_PANELS"] = panels
    try:
        C = sg.sgemm_host(A.pin_memory(), B.pin_memory())
    finally:
        if old is None:
            del os.environ["SGEMM_HOST_PANELS"]
        else:
            os.environ["SGEMM_HOST_PANELS"] = old
    check_within_bound(C.numpy(), ref, E, K, f"sgemm_host with {panels} panel(s)")


def test_strided_views_and_pageable_memory():
    """Row-strided host views (lda > K, ldb > N, ldc > N), not page-locked."""
    M, N, K = 1500, 700, 333
    A_big = workloads.matrix(M, K + 5, "uniform", 3401, 0)
    B_big = workloads.matrix(K, N + 3, "uniform", 3402, 1)
    A, B = A_big[:, :K], B_big[:, :N]
    C_big = torch.full((M, N + 9), float("nan"))
    C = C_big[:, :N]
    sg.sgemm_host(A, B, out=C)
    ref, E = oracle.sgemm_f64(A.contiguous(), B.contiguous())
    check_within_bound(C.numpy(), ref, E, K, "sgemm_host strided pageable")
    assert torch.isnan(C_big[:, N:]).all(), "columns past N of the strided C were written"


def test_k_zero_writes_zeros_and_empty_is_a_no_op():
    C = torch.full((300, 200), float("nan")).pin_memory()
    A = torch.empty((300, 0))
    B = torch.empty((0, 200))
    sg.sgemm_host(A, B, out=C)
    assert bool((C == 0).all())
    empty = torch.full((0, 5), 1.0)
    sg.sgemm_host(torch.empty((0, 3)), torch.empty((3, 5)), out=empty)


def test_two_streams_at_once():
    """Each stream has its own staging: overlapping calls on two streams both come out right."""
    probs = [(2048, 768, 1024, 3501), (1536, 1280, 640, 3502)]
    streams = [torch.cuda.Stream() for _ in probs]
    outs, refs, inputs = [], [], []   # the pinned inputs must outlive the queued copies
    for (M, N, K, seed), s in zip(probs, streams):
        A, B = _operands(M, N, K, seed)
        refs.append((oracle.sgemm_f64(A, B), K))
        inputs.append((A.pin_memory(), B.pin_memory()))
        outs.append(sg.sgemm_host(*inputs[-1], stream=s, wait=False))
    for s in streams:
        s.synchronize()
    for C, ((ref, E), K) in zip(outs, refs):
        check_within_bound(C.numpy(), ref, E, K, "sgemm_host on two streams")


def test_staging_regrowth_on_one_stream():
    """A small call, a larger one (the staging is replaced), and a small one again."""
    s = torch.cuda.Stream()
    for M, N, K, seed in [(256, 256, 128, 3601), (3000, 1000, 700, 3602), (300, 250, 90, 3603)]:
        A, B = _operands(M, N, K, seed)
        ref, E = oracle.sgemm_f64(A, B)
        C = sg.sgemm_host(A.pin_memory(), B.pin_memory(), stream=s)
        check_within_bound(C.numpy(), ref, E, K, f"sgemm_host regrowth {M}x{N}x{K}")


def test_calls_queue_behind_earlier_work_on_the_stream():
    """Back-to-back calls on one stream share its staging: the second starts only
    after the first has copied its C out, so both finish correct."""
    M, N, K = 2048, 512, 256
    A1, B1 = _operands(M, N, K, 3701)
    A2, B2 = _operands(M, N, K, 3702)
    s = torch.cuda.Stream()
    pinned = [x.pin_memory() for x in (A1, B1, A2, B2)]   # alive until the stream is done
    C1 = sg.sgemm_host(pinned[0], pinned[1], stream=s, wait=False)
    C2 = sg.sgemm_host(pinned[2], pinned[3], stream=s, wait=False)
    s.synchronize()
    for C, A, B, tag in [(C1, A1, B1, "first"), (C2, A2, B2, "second")]:
        ref, E = oracle.sgemm_f64(A, B)
        check_within_bound(C.numpy(), ref, E, K, f"sgemm_host queued ({tag})")


def test_after_releasing_workspaces():
    sg.release_workspaces()
    M, N, K = 700, 600, 500
    A, B = _operands(M, N, K, 3801)
    ref, E = oracle.sgemm_f64(A, B)
    C = sg.sgemm_host(A.pin_memory(), B.pin_memory())
    check_within_bound(C.numpy(), ref, E, K, "sgemm_host after release")
