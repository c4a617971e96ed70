"""GPU parity: the CUDA path against the CPU oracle, element by element.

Every call goes through the C ABI (``libsgemm.so``) via the ctypes binding.
Inputs are the seeded host matrices of ``workloads``; the same host arrays go
to the oracle and, copied, to the GPU.  Random inputs must meet the bound
|C_gpu - C_ref| <= 4 K 2^-24 sum_k |A B|; integer inputs with partial sums
below 2^24 must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_fp32_gemm_03_gb300 as sg
from dense_fp32_gemm_03_gb300 import workloads

from parity import check_exact, check_within_bound

pytestmark = pytest.mark.gpu

FAST = [sg.TILED, sg.STREAMK, sg.TILED_SMALL, sg.STREAMK_SMALL, sg.SMALL]
ALL_VARIANTS = [sg.GUARDED, *FAST, sg.STAGED]
SENTINEL = float.fromhex("0x1.dead00p+100")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    yield
    st, site = sg.query_device_status()
    assert st == 0, f"device status {st} (site {site}) left after the module"


def _dev(x):
    return x.to("cuda", non_blocking=False)


def _run(A, B, variant=sg.AUTO, out=None):
    C = sg.sgemm(_dev(A), _dev(B), out=out, variant=variant)
    torch.cuda.synchronize()
    return C


def _ref(A, B):
    return oracle.sgemm_f64(A, B)


# ----------------------------------------------------------------- configs
def test_square_256_uniform_all_variants():
    w = workloads.SMALL_256
    A, B = workloads.operands(w)
    ref, E = _ref(A, B)
    for v in [sg.AUTO, *ALL_VARIANTS]:
        C = _run(A, B, v).cpu().numpy()
        check_within_bound(C, ref, E, w.K, f"256^3 variant {v}")


def test_square_256_integer_bit_exact_all_variants():
    w = workloads.SMALL_256_INT
    A, B = workloads.operands(w)
    ref, E = _ref(A, B)
    assert E.max() < 2 ** 24
    for v in [sg.AUTO, *ALL_VARIANTS]:
        check_exact(_run(A, B, v).cpu().numpy(), ref, f"int 256^3 variant {v}")


@pytest.mark.parametrize("w", [workloads.SQUARE_1024] + [s for s in workloads.SWEEP if s.M <= 1024],
                         ids=lambda w: w.name)
def test_full_compare_mid_sizes(w):
    A, B = workloads.operands(w)
    ref, E = _ref(A, B)
    for v in [sg.AUTO, sg.STREAMK, sg.TILED, sg.STREAMK_SMALL]:
        C = _run(A, B, v).cpu().numpy()
        check_within_bound(C, ref, E, w.K, f"{w.name} variant {v}")


def _sampled(w, variants, count=4096):
    A, B = workloads.operands(w)
    r, c = workloads.sample_indices(w.M, w.N, count, w.seed)
    ref, E = oracle.sgemm_entries_f64(A, B, r.numpy(), c.numpy())
    dA, dB = _dev(A), _dev(B)
    out = torch.empty((w.M, w.N), device="cuda")
    for v in variants:
        out.fill_(float("nan"))
        sg.sgemm(dA, dB, out=out, variant=v)
        torch.cuda.synchronize()
        assert bool(torch.isfinite(out).all()), f"{w.name} variant {v}: non-finite output"
        got = out[r.cuda(), c.cuda()].cpu().numpy()
        check_within_bound(got, ref, E, w.K, f"{w.name} variant {v} (sampled)")
    return out


@pytest.mark.parametrize("w", [s for s in workloads.SWEEP if s.M > 1024], ids=lambda w: w.name)
def test_sampled_sweep_large(w):
    _sampled(w, [sg.AUTO, sg.STREAMK, sg.TILED])


def test_sampled_4096():
    _sampled(workloads.SQUARE_4096, [sg.AUTO, sg.STREAMK, sg.TILED])


@pytest.mark.parametrize("w", [workloads.SQUARE_8192, workloads.LONG_K, workloads.TALL],
                         ids=lambda w: w.name)
def test_sampled_large_rectangular(w):
    _sampled(w, [sg.AUTO], count=2048)


def test_full_size_row_block_4096():
    """A full 128-row block of the 4096^3 product, compared element by element."""
    w = workloads.SQUARE_4096
    A, B = workloads.operands(w)
    C = _run(A, B).cpu().numpy()
    rows = slice(1536, 1664)
    ref, E = oracle.sgemm_f64(A[rows], B)
    check_within_bound(C[rows], ref, E, w.K, "4096^3 row block")


# ----------------------------------------------------------- shapes and edges
RAGGED = [(1, 1, 1), (1, 7, 3), (5, 1, 9), (3, 5, 1), (8, 8, 8), (127, 129, 65), (129, 127, 17),
          (128, 256, 16), (255, 257, 31), (300, 520, 200), (1000, 1000, 100), (130, 4, 1000),
          (4, 1030, 77), (513, 260, 1023)]


@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
def test_ragged_shapes_all_variants(shape):
    M, N, K = shape
    A = workloads.matrix(M, K, "normal", M * 7 + N, 0)
    B = workloads.matrix(K, N, "normal", M * 7 + N, 1)
    ref, E = _ref(A, B)
    for v in [sg.AUTO, *ALL_VARIANTS]:
        if v in FAST and (K % 4 or N % 4):
            # Row strides not multiple of 4: fast variants must refuse, AUTO must fall back.
            with pytest.raises(sg.SgemmError):
                _run(A, B, v)
            continue
        check_within_bound(_run(A, B, v).cpu().numpy(), ref, E, K, f"{shape} variant {v}")


def test_row_strides_and_views():
    big_a = workloads.matrix(300, 520, "uniform", 3, 0).cuda()
    big_b = workloads.matrix(260, 600, "uniform", 3, 1).cuda()
    A = big_a[10:210, 8:208]      # 200 x 200, lda = 520
    B = big_b[4:204, 12:340]      # 200 x 328, ldb = 600
    ref, E = _ref(A.cpu(), B.cpu())
    for v in [sg.AUTO, *ALL_VARIANTS]:
        C = sg.sgemm(A, B, variant=v)
        torch.cuda.synchronize()
        check_within_bound(C.cpu().numpy(), ref, E, 200, f"views variant {v}")


def test_misaligned_pointer_avoids_the_fast_variants():
    buf_a = workloads.matrix(1, 64 * 64 + 1, "uniform", 4, 0).cuda()
    A = buf_a[0, 1:].view(64, 64)  # 4-byte offset: not 16-byte aligned
    B = workloads.matrix(64, 64, "uniform", 4, 1).cuda()
    C = torch.empty(64, 64, device="cuda")
    assert sg.select_variant(A, B, C) in (sg.GUARDED, sg.STAGED)
    with pytest.raises(sg.SgemmError):
        sg.sgemm(A, B, out=C, variant=sg.TILED)
    sg.sgemm(A, B, out=C)
    torch.cuda.synchronize()
    ref, E = _ref(A.cpu(), B.cpu())
    check_within_bound(C.cpu().numpy(), ref, E, 64, "misaligned")


def test_output_canaries_untouched():
    """C inside a larger buffer: the guard band around it must keep its sentinel."""
    M, N, K = 261, 300, 140
    A = workloads.matrix(M, K, "normal", 11, 0)
    B = workloads.matrix(K, N, "normal", 11, 1)
    ref, E = _ref(A, B)
    for v in [sg.AUTO, *ALL_VARIANTS]:
        big = torch.full((M + 16, 320), SENTINEL, device="cuda")
        C = big[8:8 + M, 8:8 + N]
        sg.sgemm(_dev(A), _dev(B), out=C, variant=v)
        torch.cuda.synchronize()
        h = big.cpu().numpy()
        mask = np.ones_like(h, dtype=bool)
        mask[8:8 + M, 8:8 + N] = False
        assert np.all(h[mask] == np.float32(SENTINEL)), f"variant {v} wrote outside C"
        check_within_bound(h[8:8 + M, 8:8 + N], ref, E, K, f"canary variant {v}")


def test_k_zero_fills_zeros_and_empty_is_noop():
    A = torch.empty(37, 0, device="cuda")
    B = torch.empty(0, 45, device="cuda")
    C = torch.full((37, 45), float("nan"), device="cuda")
    sg.sgemm(A, B, out=C)
    torch.cuda.synchronize()
    assert bool((C == 0).all())
    C2 = torch.full((0, 45), 1.0, device="cuda")
    sg.sgemm(torch.empty(0, 5, device="cuda"), torch.ones(5, 45, device="cuda"), out=C2)
    C3 = torch.full((6, 3), 1.0, device="cuda")
    sg.sgemm(torch.ones(6, 5, device="cuda"), torch.empty(5, 0, device="cuda").view(5, 0),
             out=C3[:, :0])
    torch.cuda.synchronize()
    assert bool((C3 == 1.0).all())


def test_nan_and_inf_propagate():
    M, N, K = 256, 512, 64
    A = workloads.matrix(M, K, "uniform", 21, 0)
    B = workloads.matrix(K, N, "uniform", 21, 1)
    A[17, 5] = float("nan")
    B[9, 300] = float("inf")
    ref, _ = _ref(A, B)
    for v in [sg.AUTO, *ALL_VARIANTS]:
        C = _run(A, B, v).cpu().numpy().astype(np.float64)
        assert np.array_equal(np.isnan(C), np.isnan(ref)), f"variant {v}: NaN pattern differs"
        assert np.array_equal(np.isinf(C), np.isinf(ref)), f"variant {v}: Inf pattern differs"


def test_output_prior_contents_never_read():
    """beta = 0: NaN already in C must not leak into the result."""
    w = workloads.SMALL_256
    A, B = workloads.operands(w)
    ref, E = _ref(A, B)
    for v in ALL_VARIANTS:
        C = torch.full((256, 256), float("nan"), device="cuda")
        sg.sgemm(_dev(A), _dev(B), out=C, variant=v)
        torch.cuda.synchronize()
        check_within_bound(C.cpu().numpy(), ref, E, 256, f"nan-prefill variant {v}")


def test_streamk_is_deterministic():
    w = workloads.SQUARE_1024
    A, B = map(_dev, workloads.operands(w))
    first = sg.sgemm(A, B, variant=sg.STREAMK)
    for _ in range(3):
        again = sg.sgemm(A, B, variant=sg.STREAMK)
        torch.cuda.synchronize()
        assert torch.equal(first, again)


def test_integer_long_k_exact_through_split():
    """Long K with small integers: every partial sum exact, so Stream-K splits are exact."""
    M, N, K = 128, 256, 8192
    g = torch.Generator().manual_seed(5)
    A = torch.randint(-2, 3, (M, K), generator=g).float()
    B = torch.randint(-2, 3, (K, N), generator=g).float()
    ref, E = _ref(A, B)
    assert E.max() < 2 ** 24
    for v in [sg.AUTO, sg.STREAMK, sg.STREAMK_SMALL, sg.TILED]:
        check_exact(_run(A, B, v).cpu().numpy(), ref, f"int long-K variant {v}")


def test_nondefault_stream():
    w = workloads.SMALL_256
    A, B = map(_dev, workloads.operands(w))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = sg.sgemm(A, B, variant=sg.STREAMK)
    s.synchronize()
    ref, E = _ref(*workloads.operands(w))
    check_within_bound(C.cpu().numpy(), ref, E, 256, "side stream")


def test_selector_choices_are_valid():
    for w in workloads.ALL:
        A = torch.empty(w.M, w.K, device="cuda")
        B = torch.empty(w.K, w.N, device="cuda")
        C = torch.empty(w.M, w.N, device="cuda")
        assert sg.select_variant(A, B, C) in sg.VARIANTS.values()
        del A, B, C


def test_wait_expiry_is_reported_not_hung():
    assert sg.query_device_status() == (0, 0)
    assert sg.debug_expire_wait(2_000_000) == 0     # 2 ms limit on a barrier nobody completes
    st, site = sg.query_device_status()
    assert st == 3 and site == 3                     # SGEMM_ERR_TIMEOUT at the probe
    assert sg.query_device_status() == (0, 0)        # reading cleared it
    w = workloads.SMALL_256
    A, B = workloads.operands(w)
    ref, E = _ref(A, B)
    check_within_bound(_run(A, B).cpu().numpy(), ref, E, 256, "after expiry")


def test_workspace_reuse_across_split_layouts():
    """One cached workspace serves Stream-K calls of different shapes in a row."""
    shapes = [(1024, 1024, 1024), (1536, 1536, 1536), (640, 768, 2048), (1024, 1024, 1024),
              (2048, 2048, 512), (512, 512, 4096)]
    for i, (M, N, K) in enumerate(shapes):
        A = workloads.matrix(M, K, "normal", 300 + i, 0)
        B = workloads.matrix(K, N, "normal", 300 + i, 1)
        r, c = workloads.sample_indices(M, N, 2048, 300 + i)
        ref, E = oracle.sgemm_entries_f64(A, B, r.numpy(), c.numpy())
        for v in (sg.STREAMK, sg.STREAMK_SMALL):
            out = torch.full((M, N), float("nan"), device="cuda")
            sg.sgemm(_dev(A), _dev(B), out=out, variant=v)
            torch.cuda.synchronize()
            assert bool(torch.isfinite(out).all()), f"{(M, N, K)} variant {v}: tiles not written"
            check_within_bound(out[r.cuda(), c.cuda()].cpu().numpy(), ref, E, K, f"{(M, N, K)} v{v}")


def test_concurrent_streams_use_separate_workspaces():
    """Two Stream-K calls in flight at once on two streams: each keeps its own workspace."""
    shapes = [(1536, 1536, 1536, 81), (1024, 1024, 2048, 82)]
    ops, outs, streams = [], [], [torch.cuda.Stream(), torch.cuda.Stream()]
    for M, N, K, seed in shapes:
        ops.append((workloads.matrix(M, K, "normal", seed, 0), workloads.matrix(K, N, "normal", seed, 1)))
    dev = [(A.cuda(), B.cuda()) for A, B in ops]
    torch.cuda.synchronize()
    for rep in range(3):
        for (A, B), s in zip(dev, streams):
            with torch.cuda.stream(s):
                outs.append(sg.sgemm(A, B, variant=sg.STREAMK))
    torch.cuda.synchronize()
    for idx, ((A, B), (M, N, K, seed)) in enumerate(zip(ops, shapes)):
        r, c = workloads.sample_indices(M, N, 1024, seed)
        ref, E = oracle.sgemm_entries_f64(A, B, r.numpy(), c.numpy())
        for rep in range(3):
            got = outs[2 * rep + idx][r.cuda(), c.cuda()].cpu().numpy()
            check_within_bound(got, ref, E, K, f"stream {idx} rep {rep}")


def test_graph_capture_and_replay():
    """After one call has sized the stream's workspace, sgemm() captures into a CUDA graph."""
    w = workloads.SQUARE_1024
    A_h, B_h = workloads.operands(w)
    A, B = A_h.cuda(), B_h.cuda()
    C = torch.empty(w.M, w.N, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sg.sgemm(A, B, out=C)          # warm-up: workspace for this stream exists now
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        sg.sgemm(A, B, out=C)
    C.fill_(float("nan"))
    A.copy_(workloads.matrix(w.M, w.K, w.dist, 4242, 0))   # new inputs, same buffers
    graph.replay()
    torch.cuda.synchronize()
    ref, E = oracle.sgemm_f64(A.cpu(), B_h)
    check_within_bound(C.cpu().numpy(), ref, E, w.K, "graph replay")


def test_graph_replay_after_workspace_regrowth():
    """A graph captured with sgemm() keeps a valid workspace after a larger call on the
    same stream replaced the stream's cached workspace (the old one is retired, not freed)."""
    w = workloads.SQUARE_1024
    A_h, B_h = workloads.operands(w)
    A, B = A_h.cuda(), B_h.cuda()
    C = torch.empty(w.M, w.N, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sg.sgemm(A, B, out=C)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        sg.sgemm(A, B, out=C)
    # A product whose split tiles need more workspace than 1024^3 left in the cache
    # (the cache holds 1.25 x what a call asked for).
    need = 1.25 * sg.workspace_size(w.M, w.N, w.K)
    big = next(x for x in (workloads.Workload(f"regrow_{m}x{n}x{k}", m, n, k, "normal", 1300 + m)
                           for m, n, k in [(1536, 1536, 1536), (2048, 2048, 2048),
                                           (2560, 2560, 1024), (4096, 4096, 512)])
               if sg.workspace_size(x.M, x.N, x.K) > need)
    Ab, Bb = (x.cuda() for x in workloads.operands(big))
    with torch.cuda.stream(s):
        Cb = sg.sgemm(Ab, Bb)
    s.synchronize()
    C.fill_(float("nan"))
    A.copy_(workloads.matrix(w.M, w.K, w.dist, 4343, 0))
    graph.replay()
    torch.cuda.synchronize()
    ref, E = oracle.sgemm_f64(A.cpu(), B_h)
    check_within_bound(C.cpu().numpy(), ref, E, w.K, "graph replay after regrowth")
    r, c = workloads.sample_indices(big.M, big.N, 1024, big.seed)
    ref_b, E_b = oracle.sgemm_entries_f64(*workloads.operands(big), r.numpy(), c.numpy())
    check_within_bound(Cb[r.cuda(), c.cuda()].cpu().numpy(), ref_b, E_b, big.K, "regrown call")


def test_unknown_variant_rejected_on_a_device():
    A = torch.ones(64, 64, device="cuda")
    C = torch.full((64, 64), 7.0, device="cuda")
    for v in (len(sg.VARIANTS), -2):
        with pytest.raises(sg.SgemmError) as e:
            sg.sgemm(A, A, out=C, variant=v)
        assert e.value.status == sg.binding.ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())


def test_timeout_on_one_stream_leaves_other_streams_running():
    """A wait that expires on one stream while Stream-K calls run on another: the query
    that reports it must not clear the other stream's workspace under its kernels.  The
    other stream's results, and its next call, must still be exact."""
    w = workloads.SQUARE_1024
    A_h, B_h = workloads.operands(w)
    A, B = A_h.cuda(), B_h.cuda()
    s_probe, s_work = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s_work):
        first = sg.sgemm(A, B, variant=sg.STREAMK_SMALL)   # sizes s_work's workspace
    s_work.synchronize()
    outs = [torch.full((w.M, w.N), float("nan"), device="cuda") for _ in range(40)]
    with torch.cuda.stream(s_work):
        torch.cuda._sleep(2_000_000)      # about 1 ms: the calls below start after the probe
        for out in outs:
            sg.sgemm(A, B, out=out, variant=sg.STREAMK_SMALL)
    assert sg.debug_expire_wait(2_000_000, stream=s_probe) == 0   # expires after 2 ms
    st, site = sg.query_device_status(stream=s_probe)               # while s_work still runs
    assert (st, site) == (3, 3)
    with torch.cuda.stream(s_work):
        after = sg.sgemm(A, B, variant=sg.STREAMK_SMALL)          # counters cleared first
    torch.cuda.synchronize()
    for i, out in enumerate(outs):
        assert torch.equal(out, first), f"call {i} on the other stream changed"
    assert torch.equal(after, first)
    ref, E = oracle.sgemm_f64(A_h, B_h)
    check_within_bound(first.cpu().numpy(), ref, E, w.K, "stream-K beside an expiring wait")
    assert sg.query_device_status() == (0, 0)


def test_split_tile_handoffs_under_concurrent_kernels():
    """Stream-K calls on four streams at once compete for SMs, so some CTAs of a launch start
    late: owners then give up waiting for their sharers, the partial prefetch gives up, and
    other CTAs finish the split tiles.  Whoever finishes, the sums are added in the same
    order, so every result must equal the sequential one bit for bit."""
    w = workloads.SQUARE_1024
    A_h, B_h = workloads.operands(w)
    A, B = A_h.cuda(), B_h.cuda()
    variants = [sg.STREAMK_SMALL, sg.STREAMK]
    C = torch.empty(w.M, w.N, device="cuda")
    if sg.select_variant(A, B, C) == sg.SPECIALIZED:
        variants.append(sg.SPECIALIZED)   # compiled for this device's SM count
    ref = {v: sg.sgemm(A, B, variant=v) for v in variants}
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(4)]
    outs = []
    for rep in range(6):
        for i, s in enumerate(streams):
            v = variants[(rep + i) % len(variants)]
            with torch.cuda.stream(s):
                C = torch.full((w.M, w.N), float("nan"), device="cuda")
                sg.sgemm(A, B, out=C, variant=v)
            outs.append((v, C))
    torch.cuda.synchronize()
    assert sg.query_device_status() == (0, 0)
    for k, (v, C) in enumerate(outs):
        assert torch.equal(C, ref[v]), f"call {k} (variant {v}) differs from the sequential result"
    C_ref, E = oracle.sgemm_f64(A_h, B_h)
    check_within_bound(ref[sg.STREAMK_SMALL].cpu().numpy(), C_ref, E, w.K, "concurrent hand-offs")
