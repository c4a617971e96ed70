"""GPU parity of the opt-in TF32 tensor-core mode (``sgemm_tf32``) against the oracle.

TF32 keeps FP32's exponent and 10 of its 23 fraction bits, so each input
carries a relative error below 2^-10 (truncation; half that if rounded) and
each product below 2^-9 + 2^-20.  With FP32 accumulation in any order the
per-element error is then at most (2^-9 + 2^-20 + 2K 2^-24) sum_k |A B|; the
test allows twice that.  Integers of magnitude <= 8 are exact in TF32, so
integer inputs whose partial sums stay below 2^24 must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_fp32_gemm_03_gb300 as sg
from dense_fp32_gemm_03_gb300 import workloads

from parity import check_exact

pytestmark = pytest.mark.gpu


def tf32_bound(K, E):
    return (2.0 ** -8 + 4.0 * K * 2.0 ** -24) * E


def check_tf32(C_gpu, C_ref, E, K, what):
    C_gpu = np.asarray(C_gpu, dtype=np.float64)
    assert np.all(np.isfinite(C_gpu)), f"{what}: non-finite output"
    err = np.abs(C_gpu - C_ref)
    lim = tf32_bound(K, E)
    bad = err > lim
    assert not np.any(bad), (f"{what}: {int(bad.sum())} elements outside the TF32 bound; "
                             f"worst excess {(err - lim).max():.3e}")
    return float((err / np.maximum(E, 1e-30)).max())


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert sg.query_device_status() == (0, 0)


def test_tf32_single_tile_integers_exact():
    g = torch.Generator().manual_seed(3)
    A = torch.randint(-8, 9, (128, 32), generator=g).float()
    B = torch.randint(-8, 9, (32, 256), generator=g).float()
    C = sg.sgemm_tf32(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    ref, _ = oracle.sgemm_f64(A, B, with_abs=False)
    check_exact(C.cpu().numpy(), ref, "tf32 one tile")


def test_tf32_integer_workload_exact():
    w = workloads.SMALL_256_INT
    A, B = workloads.operands(w)
    C = sg.sgemm_tf32(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    ref, _ = oracle.sgemm_f64(A, B, with_abs=False)
    check_exact(C.cpu().numpy(), ref, "tf32 int 256^3")


@pytest.mark.parametrize("w", [workloads.SMALL_256, workloads.SQUARE_1024], ids=lambda w: w.name)
def test_tf32_within_bound_full(w):
    A, B = workloads.operands(w)
    C = sg.sgemm_tf32(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    ref, E = oracle.sgemm_f64(A, B)
    worst = check_tf32(C.cpu().numpy(), ref, E, w.K, w.name)
    assert worst > 0.0  # TF32 is not FP32: some rounding must show


@pytest.mark.parametrize("w", [workloads.SQUARE_4096, workloads.LONG_K], ids=lambda w: w.name)
def test_tf32_within_bound_sampled(w):
    A, B = workloads.operands(w)
    C = sg.sgemm_tf32(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    r, c = workloads.sample_indices(w.M, w.N, 2048, w.seed)
    ref, E = oracle.sgemm_entries_f64(A, B, r.numpy(), c.numpy())
    check_tf32(C[r.cuda(), c.cuda()].cpu().numpy(), ref, E, w.K, w.name)


@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 7, 3), (127, 129, 65), (300, 520, 200),
                                   (1000, 1000, 100), (130, 4, 1001), (257, 300, 33)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tf32_ragged_shapes_and_k_tails(shape):
    M, N, K = shape
    lda = (K + 3) // 4 * 4                      # A's row stride must be a multiple of 4
    A_big = workloads.matrix(M, lda, "normal", M + N, 0)
    A = A_big[:, :K]
    B = workloads.matrix(K, N, "normal", M + N, 1)   # B may have any stride
    ldc = (N + 3) // 4 * 4
    C_big = torch.full((M, ldc), float("nan"), device="cuda")
    C = C_big[:, :N]
    sg.sgemm_tf32(A.cuda() if A.is_contiguous() else A_big.cuda()[:, :K], B.cuda(), out=C)
    torch.cuda.synchronize()
    ref, E = oracle.sgemm_f64(np.ascontiguousarray(A.numpy()), B)
    check_tf32(C.cpu().numpy(), ref, E, K, f"tf32 {shape}")
    if ldc > N:
        assert bool(torch.isnan(C_big[:, N:]).all()), "wrote past N"


@pytest.mark.parametrize("shape", [(64, 64, 65), (300, 259, 201), (513, 771, 1027)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tf32_any_alignment(shape):
    """A starting 4 bytes off alignment with an odd stride (copied first), B with an odd
    stride (transposed first), C starting 4 bytes off alignment (4-byte stores)."""
    M, N, K = shape
    A = workloads.matrix(M, K, "normal", 99, 0)
    B = workloads.matrix(K, N, "normal", 99, 1)
    ref, E = oracle.sgemm_f64(A, B)
    bufA = torch.zeros(M * (K + 1) + 1, device="cuda")
    dA = bufA[1:].as_strided((M, K), (K + 1, 1))
    dA.copy_(A.cuda())
    dB = B.cuda()                                    # ldb = N, odd for two of the shapes
    big = torch.full((M * (N + 3) + 1,), float("nan"), device="cuda")
    C = big[1:].as_strided((M, N), (N + 3, 1))
    sg.sgemm_tf32(dA, dB, out=C)
    torch.cuda.synchronize()
    check_tf32(C.cpu().numpy(), ref, E, K, f"tf32 any alignment {shape}")


@pytest.mark.parametrize("shape", [(256, 256, 256), (384, 520, 96), (129, 300, 77), (300, 33, 1029)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tf32_b_in_place_and_transposed(shape):
    """B read in place (MN-major, 16-byte aligned rows) and B copied transposed first
    (a base 4 bytes off alignment) give results within the bound, on every tile edge."""
    M, N, K = shape
    lda = (K + 3) // 4 * 4
    A = workloads.matrix(M, K, "uniform", 90 + M, 0)
    B = workloads.matrix(K, N, "uniform", 90 + M, 1)
    ref, E = oracle.sgemm_f64(A, B)
    A_dev = torch.zeros(M, lda, device="cuda")
    A_dev[:, :K] = A.cuda()
    A_dev = A_dev[:, :K]
    ldb = (N + 3) // 4 * 4
    B_aligned = torch.zeros(K, ldb, device="cuda")
    B_aligned[:, :N] = B.cuda()
    B_aligned = B_aligned[:, :N]
    flat = torch.zeros(K * N + 1, device="cuda")
    B_offset = flat[1:].view(K, N)
    B_offset.copy_(B.cuda())
    ldc = (N + 3) // 4 * 4                       # C's row stride must be a multiple of 4
    for what, Bd in (("in place", B_aligned), ("transposed", B_offset)):
        C = torch.full((M, ldc), float("nan"), device="cuda")[:, :N]
        sg.sgemm_tf32(A_dev, Bd, out=C)
        torch.cuda.synchronize()
        check_tf32(C.cpu().numpy(), ref, E, K, f"tf32 {shape} B {what}")


@pytest.mark.parametrize("shape", [(200, 260, 64), (200, 261, 64), (300, 518, 96), (257, 515, 40),
                                   (513, 1024, 48), (1029, 2051, 64), (2600, 2301, 256)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tf32_edges_leave_neighbours_untouched(shape):
    """C inside a larger NaN-filled buffer (rows below it, columns right of it): stores at
    the M and N edges (TMA boxes clipped by the hardware, or row stores where N is not a
    multiple of 4) write C and nothing else, on integer inputs that must be exact."""
    M, N, K = shape
    A = workloads.matrix(M, K, "int8range", 71 + N, 0)
    B = workloads.matrix(K, N, "int8range", 71 + N, 1)
    ref, E = oracle.sgemm_f64(A, B)
    assert E.max() < 2 ** 24
    ldc = (N + 3) // 4 * 4 + 8                   # 8 or more canary columns on the right
    big = torch.full((M + 40, ldc), float("nan"), device="cuda")
    C = big[:M, :N]
    sg.sgemm_tf32(A.cuda(), B.cuda(), out=C)
    torch.cuda.synchronize()
    check_exact(C.cpu().numpy(), ref, f"tf32 edges {shape}")
    assert bool(torch.isnan(big[:M, N:]).all()), "wrote right of column N - 1"
    assert bool(torch.isnan(big[M:]).all()), "wrote below row M - 1"


def test_tf32_integers_exact_through_both_b_paths():
    M, N, K = 256, 512, 384
    A = workloads.matrix(M, K, "int8range", 95, 0)
    B = workloads.matrix(K, N, "int8range", 95, 1)
    ref, _ = oracle.sgemm_f64(A, B)
    flat = torch.zeros(K * N + 3, device="cuda")
    B_offset = flat[3:].view(K, N)
    B_offset.copy_(B.cuda())
    for Bd in (B.cuda(), B_offset):
        C = sg.sgemm_tf32(A.cuda(), Bd)
        torch.cuda.synchronize()
        check_exact(C.cpu().numpy(), ref, "tf32 integers")


@pytest.mark.parametrize("shape", [(1000, 1000, 2048), (4096, 4096, 512)], ids=lambda s: "x".join(map(str, s)))
def test_tf32_stream_k_deterministic_and_within_bound(shape):
    """Split tiles (Stream-K) are summed in a fixed order: repeated calls agree bit for bit."""
    M, N, K = shape
    A = workloads.matrix(M, K, "uniform", 97, 0)
    B = workloads.matrix(K, N, "uniform", 97, 1)
    dA, dB = A.cuda(), B.cuda()
    C1 = sg.sgemm_tf32(dA, dB)
    C2 = sg.sgemm_tf32(dA, dB)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    r, c = workloads.sample_indices(M, N, 2048, 97)
    ref, E = oracle.sgemm_entries_f64(A, B, r.numpy(), c.numpy())
    check_tf32(C1[r.cuda(), c.cuda()].cpu().numpy(), ref, E, K, f"tf32 {shape}")


@pytest.mark.parametrize("shape", [(2048, 2048, 2048), (1000, 1000, 2048), (4096, 4096, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tf32_split_tiles_summed_from_the_workspace_match_bit_for_bit(shape):
    """With the test switch the owner of a split tile publishes its partial instead of
    keeping it in tensor memory, and the last to arrive sums every partial from the
    workspace: the same additions in the same order, so the same bits."""
    M, N, K = shape
    A = workloads.matrix(M, K, "uniform", 98, 0).cuda()
    B = workloads.matrix(K, N, "uniform", 98, 1).cuda()
    default = sg.sgemm_tf32(A, B)
    sg.debug_owner_publishes(True)
    try:
        published = sg.sgemm_tf32(A, B)
    finally:
        sg.debug_owner_publishes(False)
    torch.cuda.synchronize()
    assert torch.equal(default, published)


_SINGLE_SM_SCRIPT = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import oracle
import dense_fp32_gemm_03_gb300 as sg
from dense_fp32_gemm_03_gb300 import workloads
for (M, N, K) in [(256, 512, 384), (1000, 1000, 2048), (4096, 4096, 512)]:
    A = workloads.matrix(M, K, "int8range", 98, 0)
    B = workloads.matrix(K, N, "int8range", 98, 1)
    C = sg.sgemm_tf32(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    r, c = workloads.sample_indices(M, N, 2048, 98)
    ref, E = oracle.sgemm_entries_f64(A, B, r.numpy(), c.numpy())
    assert E.max() < 2 ** 24
    got = C[r.cuda(), c.cuda()].cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref), (M, N, K)
# C inside NaN canaries (rows below, columns right; N % 4 = 1, 3, 1).
for (M, N, K) in [(200, 261, 64), (1029, 2051, 64), (2600, 2301, 256)]:
    A = workloads.matrix(M, K, "int8range", 71 + N, 0)
    B = workloads.matrix(K, N, "int8range", 71 + N, 1)
    ref, E = oracle.sgemm_f64(A, B)
    ldc = (N + 3) // 4 * 4 + 8
    big = torch.full((M + 40, ldc), float("nan"), device="cuda")
    sg.sgemm_tf32(A.cuda(), B.cuda(), out=big[:M, :N])
    torch.cuda.synchronize()
    assert np.array_equal(big[:M, :N].cpu().numpy().astype(np.float64), ref), (M, N, K)
    assert bool(torch.isnan(big[:M, N:]).all()) and bool(torch.isnan(big[M:]).all()), (M, N, K)
# Split tiles summed from the workspace (test switch) give the owner's bits.
for (M, N, K) in [(1000, 1000, 2048), (4096, 4096, 512)]:
    A = workloads.matrix(M, K, "uniform", 99, 0).cuda()
    B = workloads.matrix(K, N, "uniform", 99, 1).cuda()
    C0 = sg.sgemm_tf32(A, B)
    sg.debug_owner_publishes(True)
    C1 = sg.sgemm_tf32(A, B)
    sg.debug_owner_publishes(False)
    torch.cuda.synchronize()
    assert torch.equal(C0, C1), (M, N, K)
assert sg.query_device_status() == (0, 0)
print("single-SM path ok")
"""


def test_tf32_single_sm_kernel_in_a_subprocess():
    """The single-SM kernel (used where no CTA pair fits) stays exact on integers and writes
    nothing outside C."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = _SINGLE_SM_SCRIPT.format(root=root, tests=os.path.join(root, "tests"))
    env = dict(os.environ, SGEMM_TF32_PAIRS="0")
    r = subprocess.run([sys.executable, "-c", script], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "single-SM path ok" in r.stdout
