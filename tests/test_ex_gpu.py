"""GPU parity of sgemm_ex: C = alpha * A B + beta * C, row- and column-major.

Expected values come from the oracle's scaled, two-layout form.  Tolerance:
the product term keeps the FP32 bound |alpha| 4 K 2^-24 sum|ab|; scaling by
alpha, adding beta * C and the final rounding add at most a few units of
2^-24 of |alpha| sum|ab| + |beta c0|.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_fp32_gemm_03_gb300 as sg
from dense_fp32_gemm_03_gb300 import workloads

pytestmark = pytest.mark.gpu
U24 = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert sg.query_device_status() == (0, 0)


def _check(got, A, B, alpha, beta, C0, what):
    K = A.shape[1]
    ref = oracle.sgemm_ex_f64(A, B, alpha=alpha, beta=beta, C0=C0)
    _, E = oracle.sgemm_f64(np.ascontiguousarray(A), np.ascontiguousarray(B))
    c0 = np.abs(C0.astype(np.float64)) if beta != 0 else 0.0
    lim = abs(alpha) * 4 * K * U24 * E + 4 * U24 * (abs(alpha) * E + abs(beta) * c0)
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    bad = np.abs(got - ref) > lim
    assert not np.any(bad), f"{what}: {int(bad.sum())} elements outside the bound"


# Shapes that reach each kernel: Stream-K with split tiles (large and small
# tiles), whole-tile waves, ragged edges, and the bounds-checked kernel.
SHAPES = [(1536, 1536, 512), (1024, 1024, 1024), (256, 512, 64), (300, 520, 200), (129, 77, 33)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("alpha,beta", [(1.5, -0.75), (-2.0, 0.0), (1.0, 1.0)])
def test_row_major_alpha_beta(shape, alpha, beta):
    M, N, K = shape
    A = workloads.matrix(M, K, "normal", 400 + M, 0).numpy()
    B = workloads.matrix(K, N, "normal", 400 + M, 1).numpy()
    C0 = workloads.matrix(M, N, "normal", 400 + M, 2).numpy()
    C = torch.from_numpy(C0).cuda()
    if beta == 0.0:
        C.fill_(float("nan"))   # beta == 0 must not read C
    sg.sgemm_ex(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), C, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    _check(C.cpu().numpy(), A, B, alpha, beta, C0, f"row {shape} a={alpha} b={beta}")


def _col(x):
    """A CUDA tensor with the values of x in column-major storage."""
    return torch.from_numpy(np.ascontiguousarray(x.T)).cuda().t()


@pytest.mark.parametrize("shape", [(1024, 768, 512), (300, 520, 200), (33, 17, 9)],
                         ids=lambda s: "x".join(map(str, s)))
def test_column_major(shape):
    M, N, K = shape
    A = workloads.matrix(M, K, "uniform", 500 + M, 0).numpy()
    B = workloads.matrix(K, N, "uniform", 500 + M, 1).numpy()
    C0 = workloads.matrix(M, N, "uniform", 500 + M, 2).numpy()
    C = _col(C0)
    sg.sgemm_ex(_col(A), _col(B), C, alpha=0.5, beta=2.0, layout=sg.COL_MAJOR)
    torch.cuda.synchronize()
    _check(C.cpu().numpy(), A, B, 0.5, 2.0, C0, f"col {shape}")


def test_alpha_zero_and_k_zero_scale_c():
    C0 = workloads.matrix(100, 60, "normal", 9, 2)
    A = torch.full((100, 40), float("nan"), device="cuda")   # alpha == 0: A, B unused
    B = torch.full((40, 60), float("nan"), device="cuda")
    C = C0.cuda()
    sg.sgemm_ex(A, B, C, alpha=0.0, beta=-3.0)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), -3.0 * C0)
    C = C0.cuda()
    sg.sgemm_ex(torch.empty(100, 0, device="cuda"), torch.empty(0, 60, device="cuda"), C,
                alpha=2.0, beta=0.5)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), 0.5 * C0)
    C = torch.full((100, 60), float("nan"), device="cuda")
    sg.sgemm_ex(torch.empty(100, 0, device="cuda"), torch.empty(0, 60, device="cuda"), C,
                alpha=2.0, beta=0.0)
    torch.cuda.synchronize()
    assert bool((C == 0).all())


def test_integer_alpha_beta_exact():
    w = workloads.SMALL_256_INT
    A, B = (x.numpy() for x in workloads.operands(w))
    C0 = workloads.matrix(256, 256, "int8range", 77, 2).numpy()
    C = torch.from_numpy(C0).cuda()
    sg.sgemm_ex(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), C, alpha=2.0, beta=-1.0)
    torch.cuda.synchronize()
    ref = oracle.sgemm_ex_f64(A, B, alpha=2.0, beta=-1.0, C0=C0)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), ref)


def test_layout_rejected_when_unknown():
    A = torch.ones(8, 8, device="cuda")
    C = torch.empty(8, 8, device="cuda")
    st = sg.binding.load().sgemm_ex(7, 8, 8, 8, 1.0, A.data_ptr(), 8, A.data_ptr(), 8, 0.0,
                                    C.data_ptr(), 8, 0)
    assert st == sg.binding.ERR_INVALID_VALUE
