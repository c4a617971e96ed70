"""GPU parity of the small-product kernel (variant SMALL).

64 x 64 tiles with K split over CTAs; the shares of a tile are added in
share order by whichever CTA arrives last, so repeated calls agree bit for
bit.  Results must meet the FP32 bound (integer inputs: exact).
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


# Shapes: one tile and no split (K < 64), one tile split many ways, many tiles
# split a few ways, ragged edges in every dimension, K tails inside a share.
SHAPES = [(1, 1, 4), (8, 8, 8), (64, 64, 16), (64, 64, 1024), (128, 128, 128), (256, 256, 256),
          (100, 132, 300), (513, 260, 1020), (768, 768, 768), (65, 4, 4000), (4, 1000, 36),
          (300, 520, 200)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_against_oracle(shape):
    M, N, K = shape
    A = workloads.matrix(M, K, "normal", 700 + M + K, 0)
    B = workloads.matrix(K, N, "normal", 700 + M + K, 1)
    ref, E = oracle.sgemm_f64(A, B)
    # Row strides padded to multiples of 4 (the kernel's 128-bit loads).
    lda, ldb = (K + 3) // 4 * 4, (N + 3) // 4 * 4
    dA = torch.zeros(M, lda, device="cuda")
    dA[:, :K] = A.cuda()
    dB = torch.zeros(K, ldb, device="cuda")
    dB[:, :N] = B.cuda()
    ldc = (N + 3) // 4 * 4 + 4
    big = torch.full((M + 2, ldc + 4), SENTINEL, device="cuda")
    C = big[1:1 + M, 4:4 + N]            # ldc = ldc + 4 (a multiple of 4), 16-byte aligned
    sg.sgemm(dA[:, :K], dB[:, :N], out=C, variant=sg.SMALL)
    torch.cuda.synchronize()
    h = big.cpu().numpy()
    mask = np.ones_like(h, dtype=bool)
    mask[1:1 + M, 4:4 + N] = False
    assert np.all(h[mask] == np.float32(SENTINEL)), "wrote outside C"
    check_within_bound(h[1:1 + M, 4:4 + N], ref, E, K, f"small {shape}")


def test_small_split_deterministic_and_integer_exact():
    M, N, K = 192, 320, 2048                # 15 tiles, K split into many shares
    A = workloads.matrix(M, K, "int8range", 71, 0)
    B = workloads.matrix(K, N, "int8range", 71, 1)
    ref, E = oracle.sgemm_f64(A, B)
    assert E.max() < 2 ** 24
    C1 = sg.sgemm(A.cuda(), B.cuda(), variant=sg.SMALL)
    torch.cuda.synchronize()
    check_exact(C1.cpu().numpy(), ref, "small integers")
    R = workloads.matrix(M, K, "uniform", 72, 0).cuda()
    S = workloads.matrix(K, N, "uniform", 72, 1).cuda()
    first = sg.sgemm(R, S, variant=sg.SMALL)
    for _ in range(3):
        again = sg.sgemm(R, S, variant=sg.SMALL)
        torch.cuda.synchronize()
        assert torch.equal(first, again)


@pytest.mark.parametrize("alpha,beta", [(1.5, -0.5), (-2.0, 0.0)])
def test_small_alpha_beta(alpha, beta):
    M, N, K = 200, 132, 700
    A = workloads.matrix(M, K, "normal", 73, 0).numpy()
    B = workloads.matrix(K, N, "normal", 73, 1).numpy()
    C0 = workloads.matrix(M, N, "normal", 73, 2).numpy()
    C = torch.from_numpy(C0).cuda()
    if beta == 0.0:
        C.fill_(float("nan"))               # beta == 0 never reads C
    assert sg.select_variant(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), C) == sg.SMALL
    sg.sgemm_ex(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), C, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    ref = oracle.sgemm_ex_f64(A, B, alpha=alpha, beta=beta, C0=C0)
    _, E = oracle.sgemm_f64(A, B)
    U24 = 2.0 ** -24
    c0 = np.abs(C0) if beta != 0 else 0.0
    lim = abs(alpha) * 4 * K * U24 * E + 4 * U24 * (abs(alpha) * E + abs(beta) * c0)
    got = C.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert not np.any(np.abs(got - ref) > lim)


def test_small_refuses_unaligned_and_staged_small_works():
    A = torch.ones(64, 63, device="cuda")
    B = torch.ones(63, 64, device="cuda")
    with pytest.raises(sg.SgemmError):
        sg.sgemm(A, B, variant=sg.SMALL)
    # Odd strides: the selector stages the copies and may run this kernel on them.
    M, N, K = 150, 97, 231
    A = workloads.matrix(M, K, "normal", 74, 0)
    B = workloads.matrix(K, N, "normal", 74, 1)
    ref, E = oracle.sgemm_f64(A, B)
    C = sg.sgemm(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    check_within_bound(C.cpu().numpy(), ref, E, K, "staged small")


def test_selector_uses_small_for_small_products_only():
    def pick(n):
        A = torch.empty(n, n, device="cuda")
        return sg.select_variant(A, A, torch.empty(n, n, device="cuda"))
    assert pick(128) == sg.SMALL
    assert pick(256) == sg.SMALL
    assert pick(4096) != sg.SMALL
