"""GPU parity of the staged variant: operands the TMA-fed kernels cannot read in place.

A contiguous matrix with a column count that is not a multiple of 4 has a
row stride TMA cannot take, and so has any view that starts at an address
not aligned to 16 bytes.  The staged variant copies such an A or B into an
aligned workspace buffer and writes such a C with 4-byte stores; results
must meet the same bound as every other variant (integer inputs: exact).
"""
import numpy as np
import pytest
import torch

import oracle
import dense_fp32_gemm_03_gb300 as sg
from dense_fp32_gemm_03_gb300 import workloads

from parity import check_exact, check_within_bound

pytestmark = pytest.mark.gpu
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


def _offset_view(host, offset):
    """A CUDA view of `host` whose first element sits `offset` floats into a buffer."""
    rows, cols = host.shape
    buf = torch.full((rows * cols + offset,), SENTINEL, device="cuda")
    view = buf[offset:].view(rows, cols)
    view.copy_(host)
    return view


def _padded_view(host, pad, offset=0):
    """A CUDA view of `host` with row stride cols + pad, starting `offset` floats in."""
    rows, cols = host.shape
    ld = cols + pad
    buf = torch.full((rows * ld + offset,), SENTINEL, device="cuda")
    view = buf[offset:].as_strided((rows, cols), (ld, 1))
    view.copy_(host)
    return view


# (M, N, K, which operands start one float past an aligned address)
CASES = [
    (300, 520, 201, ""),        # lda = 201
    (333, 521, 256, ""),        # ldb = ldc = 521: B copied, C written with 4-byte stores
    (257, 259, 263, ""),        # every stride odd
    (256, 512, 256, "A"),       # aligned strides, A misaligned
    (256, 512, 256, "B"),
    (256, 512, 256, "C"),
    (385, 130, 97, "ABC"),      # odd strides and offsets together
    (1, 1, 1, "ABC"),
    (2, 3, 5, ""),
    (129, 1, 1023, "A"),
    (1, 1025, 3, "B"),
    (1031, 1029, 1027, ""),    # several tiles, ragged in every direction, split over K
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:3])) + (c[3] or ""))
@pytest.mark.parametrize("variant", ["staged", "auto"])
def test_unaligned_operands(case, variant):
    M, N, K, off = case
    A = workloads.matrix(M, K, "normal", 600 + M + N, 0)
    B = workloads.matrix(K, N, "normal", 600 + M + N, 1)
    ref, E = oracle.sgemm_f64(A, B)
    dA = _offset_view(A, 1 if "A" in off else 0)
    dB = _offset_view(B, 1 if "B" in off else 0)
    C = _offset_view(torch.zeros(M, N), 1 if "C" in off else 0)
    C.fill_(float("nan"))
    v = sg.STAGED if variant == "staged" else sg.AUTO
    sg.sgemm(dA, dB, out=C, variant=v)
    torch.cuda.synchronize()
    check_within_bound(C.cpu().numpy(), ref, E, K, f"{case} {variant}")


def test_fast_variants_still_refuse_unaligned():
    A = torch.ones(64, 63, device="cuda")
    B = torch.ones(63, 64, device="cuda")
    for v in (sg.TILED, sg.STREAMK, sg.TILED_SMALL, sg.STREAMK_SMALL):
        with pytest.raises(sg.SgemmError):
            sg.sgemm(A, B, variant=v)


def test_selector_stages_large_and_guards_tiny():
    A = torch.empty(2048, 2047, device="cuda")
    B = torch.empty(2047, 2048, device="cuda")
    C = torch.empty(2048, 2048, device="cuda")
    assert sg.select_variant(A, B, C) == sg.STAGED
    a, b, c = torch.empty(8, 7, device="cuda"), torch.empty(7, 8, device="cuda"), torch.empty(
        8, 8, device="cuda")
    assert sg.select_variant(a, b, c) == sg.GUARDED
    # Aligned operands never take either.
    A4 = torch.empty(2048, 2048, device="cuda")
    assert sg.select_variant(A4, A4, C) in (sg.TILED, sg.STREAMK, sg.TILED_SMALL, sg.STREAMK_SMALL,
                                            sg.SPECIALIZED)


def test_canaries_around_misaligned_c():
    """C one float into a padded buffer: nothing outside C may change."""
    M, N, K = 261, 303, 141
    A = workloads.matrix(M, K, "uniform", 61, 0)
    B = workloads.matrix(K, N, "uniform", 61, 1)
    ref, E = oracle.sgemm_f64(A, B)
    for v in (sg.STAGED, sg.AUTO, sg.GUARDED):
        big = torch.full((M + 16, 331), SENTINEL, device="cuda")
        C = big[8:8 + M, 9:9 + N]    # ldc = 331, base 4 bytes past a 16-byte boundary
        sg.sgemm(_offset_view(A, 3), _padded_view(B, 5, 2), out=C, variant=v)
        torch.cuda.synchronize()
        h = big.cpu().numpy()
        mask = np.ones_like(h, dtype=bool)
        mask[8:8 + M, 9:9 + N] = False
        assert np.all(h[mask] == np.float32(SENTINEL)), f"variant {v} wrote outside C"
        check_within_bound(h[8:8 + M, 9:9 + N], ref, E, K, f"canary variant {v}")


def test_integer_inputs_exact_with_odd_strides():
    M, N, K = 255, 257, 253
    A = workloads.matrix(M, K, "int8range", 62, 0)
    B = workloads.matrix(K, N, "int8range", 62, 1)
    ref, E = oracle.sgemm_f64(A, B)
    assert E.max() < 2 ** 24
    C = torch.empty(M, N, device="cuda")
    sg.sgemm(A.cuda(), B.cuda(), out=C, variant=sg.STAGED)
    torch.cuda.synchronize()
    check_exact(C.cpu().numpy(), ref, "int staged")


@pytest.mark.parametrize("layout", ["row", "col"])
def test_alpha_beta_with_misaligned_c(layout):
    M, N, K = 301, 259, 130
    A = workloads.matrix(M, K, "normal", 63, 0).numpy()
    B = workloads.matrix(K, N, "normal", 63, 1).numpy()
    C0 = workloads.matrix(M, N, "normal", 63, 2).numpy()
    alpha, beta = -1.25, 0.5
    if layout == "row":
        dA, dB = _offset_view(torch.from_numpy(A), 1), _offset_view(torch.from_numpy(B), 2)
        C = _offset_view(torch.from_numpy(C0), 3)
        sg.sgemm_ex(dA, dB, C, alpha=alpha, beta=beta)
        torch.cuda.synchronize()
        got = C.cpu().numpy()
    else:
        # Column-major: store the transposes row-major, then view them back.
        dA = _offset_view(torch.from_numpy(np.ascontiguousarray(A.T)), 1).t()
        dB = _offset_view(torch.from_numpy(np.ascontiguousarray(B.T)), 1).t()
        C = _offset_view(torch.from_numpy(np.ascontiguousarray(C0.T)), 1).t()
        sg.sgemm_ex(dA, dB, C, alpha=alpha, beta=beta, layout=sg.COL_MAJOR)
        torch.cuda.synchronize()
        got = C.cpu().numpy()
    ref = oracle.sgemm_ex_f64(A, B, alpha=alpha, beta=beta, C0=C0)
    _, E = oracle.sgemm_f64(A, B)
    U24 = 2.0 ** -24
    lim = abs(alpha) * 4 * K * U24 * E + 4 * U24 * (abs(alpha) * E + abs(beta) * np.abs(C0))
    assert np.all(np.isfinite(got))
    bad = np.abs(got.astype(np.float64) - ref) > lim
    assert not np.any(bad), f"{layout}: {int(bad.sum())} elements outside the bound"


def test_staged_then_other_variants_share_the_workspace():
    """Copies and partial tiles share the stream's workspace: alternate calls."""
    M, N, K = 1029, 771, 517
    A = workloads.matrix(M, K, "uniform", 64, 0)
    B = workloads.matrix(K, N, "uniform", 64, 1)
    ref, E = oracle.sgemm_f64(A, B)
    dA, dB = A.cuda(), B.cuda()
    Kp = 520
    A4 = torch.zeros(M, Kp)
    A4[:, :K] = A
    B4 = torch.zeros(Kp, N + 1)
    B4[:K, :N] = B
    dA4, dB4 = A4.cuda(), B4.cuda()[:, :N]   # ldb = N + 1 = 772: aligned
    outs = []
    for v in (sg.STAGED, sg.STREAMK_SMALL, sg.STAGED, sg.STREAMK, sg.AUTO):
        C = torch.full((M, N + 1), float("nan"), device="cuda")[:, :N]   # ldc = 772
        if v == sg.STAGED or v == sg.AUTO:
            sg.sgemm(dA, dB, out=C, variant=v)
        else:
            sg.sgemm(dA4, dB4, out=C, variant=v)
        outs.append(C)
    torch.cuda.synchronize()
    for i, C in enumerate(outs):
        check_within_bound(C.cpu().numpy(), ref, E, K, f"call {i}")


def test_workspace_size_covers_both_copies():
    M, N, K = 1023, 1025, 1027
    need = sg.workspace_size(M, N, K, variant=sg.STAGED)
    assert need >= 4 * (M * 1028 + K * 1028)


def test_sampled_full_size_unaligned_4095():
    """4095 x 4097 x 4093: every operand copied, C scalar, sampled against the oracle."""
    M, N, K = 4095, 4097, 4093
    A = workloads.matrix(M, K, "uniform", 65, 0)
    B = workloads.matrix(K, N, "uniform", 65, 1)
    r, c = workloads.sample_indices(M, N, 4096, 65)
    ref, E = oracle.sgemm_entries_f64(A, B, r.numpy(), c.numpy())
    out = torch.full((M, N), float("nan"), device="cuda")
    assert sg.select_variant(A.cuda(), B.cuda(), out) == sg.STAGED
    sg.sgemm(A.cuda(), B.cuda(), out=out)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all())
    got = out[r.cuda(), c.cuda()].cpu().numpy()
    check_within_bound(got, ref, E, K, "4095x4097x4093 staged (sampled)")
