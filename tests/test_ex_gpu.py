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


# ------------------------------------------------------------ sgemm_ex2: op(A), op(B)
TRANS = [(False, False), (True, False), (False, True), (True, True)]
TRANS_IDS = ["NN", "TN", "NT", "TT"]


def _stored(x, t):
    """The stored form of op(X) = x: x itself, or its transpose (contiguous)."""
    return np.ascontiguousarray(x.T) if t else np.ascontiguousarray(x)


def _check_op(got, opA, opB, A_st, B_st, ta, tb, alpha, beta, C0, what, col_major=False):
    K = opA.shape[1]
    ref = oracle.sgemm_op_f64(A_st, B_st, trans_a=ta, trans_b=tb, alpha=alpha, beta=beta, C0=C0,
                              col_major=col_major)
    _, E = oracle.sgemm_f64(opA, opB)
    c0 = np.abs(C0.astype(np.float64)) if beta != 0 else 0.0
    lim = abs(alpha) * 4 * K * U24 * E + 4 * U24 * (abs(alpha) * E + abs(beta) * c0)
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    bad = np.abs(got - ref) > lim
    assert not np.any(bad), f"{what}: {int(bad.sum())} elements outside the bound"


# Shapes that reach each path: Stream-K 128 x 256 with split tiles, the
# 1024^3 size (size-specialized instance when nothing is copied), the
# small-product kernel, ragged sizes whose transposed storage has row strides
# that are not multiples of 4 (copied, or the guarded kernel), and a thin one.
# 1023 x 1025 x 515: every stored matrix has an odd row stride, so the staged
# variant copies the operands: transposed copies and aligned copies together.
OP_SHAPES = [(1536, 1536, 512), (1024, 1024, 1024), (256, 512, 64), (300, 520, 200),
             (129, 77, 33), (1000, 1000, 100), (64, 4096, 256), (1023, 1025, 515)]


@pytest.mark.parametrize("shape", OP_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.5, -0.75)], ids=["plain", "scaled"])
@pytest.mark.parametrize("ta,tb", TRANS, ids=TRANS_IDS)
def test_transposed_operands_row_major(shape, alpha, beta, ta, tb):
    M, N, K = shape
    opA = workloads.matrix(M, K, "normal", 600 + M + N, 0).numpy()
    opB = workloads.matrix(K, N, "normal", 600 + M + N, 1).numpy()
    C0 = workloads.matrix(M, N, "normal", 600 + M + N, 2).numpy()
    A_st, B_st = _stored(opA, ta), _stored(opB, tb)
    C = torch.from_numpy(C0).cuda()
    if beta == 0.0:
        C.fill_(float("nan"))
    sg.sgemm_ex2(torch.from_numpy(A_st).cuda(), torch.from_numpy(B_st).cuda(), C, alpha=alpha,
                 beta=beta, trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    _check_op(C.cpu().numpy(), opA, opB, A_st, B_st, ta, tb, alpha, beta, C0,
              f"ex2 {shape} ta={ta} tb={tb} a={alpha} b={beta}")


@pytest.mark.parametrize("shape", [(1024, 768, 512), (300, 520, 200), (33, 17, 9)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("ta,tb", TRANS, ids=TRANS_IDS)
def test_transposed_operands_column_major(shape, ta, tb):
    M, N, K = shape
    opA = workloads.matrix(M, K, "uniform", 700 + M, 0).numpy()
    opB = workloads.matrix(K, N, "uniform", 700 + M, 1).numpy()
    C0 = workloads.matrix(M, N, "uniform", 700 + M, 2).numpy()
    A_st = np.ascontiguousarray(opA.T if ta else opA)
    B_st = np.ascontiguousarray(opB.T if tb else opB)
    C = _col(C0)
    sg.sgemm_ex2(_col(A_st), _col(B_st), C, alpha=0.5, beta=2.0, trans_a=ta, trans_b=tb,
                 layout=sg.COL_MAJOR)
    torch.cuda.synchronize()
    _check_op(C.cpu().numpy(), opA, opB, A_st, B_st, ta, tb, 0.5, 2.0, C0,
              f"ex2 col {shape} ta={ta} tb={tb}", col_major=True)


@pytest.mark.parametrize("shape", [(256, 256, 256), (1024, 1024, 1024), (1000, 772, 300)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("ta,tb", TRANS, ids=TRANS_IDS)
def test_transposed_integer_inputs_exact(shape, ta, tb):
    M, N, K = shape
    opA = workloads.matrix(M, K, "int8range", 800 + M, 0).numpy()
    opB = workloads.matrix(K, N, "int8range", 800 + M, 1).numpy()
    C0 = workloads.matrix(M, N, "int8range", 800 + M, 2).numpy()
    A_st, B_st = _stored(opA, ta), _stored(opB, tb)
    C = torch.from_numpy(C0).cuda()
    sg.sgemm_ex2(torch.from_numpy(A_st).cuda(), torch.from_numpy(B_st).cuda(), C, alpha=2.0,
                 beta=-1.0, trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    ref = oracle.sgemm_op_f64(A_st, B_st, trans_a=ta, trans_b=tb, alpha=2.0, beta=-1.0, C0=C0)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("ta,tb", TRANS, ids=TRANS_IDS)
def test_transposed_operands_match_explicit_transposes_bit_for_bit(ta, tb):
    """At 1024^3 the transposed forms run the schedule sgemm() runs on explicitly
    transposed copies (an M-major A lands in shared memory exactly as the transposed
    row-major A does; a transposed B is copied first), so the sums are the same."""
    w = workloads.SQUARE_1024
    opA, opB = (x.numpy() for x in workloads.operands(w))
    dA, dB = torch.from_numpy(opA).cuda(), torch.from_numpy(opB).cuda()
    plain = sg.sgemm(dA, dB)
    C = torch.full((w.M, w.N), float("nan"), device="cuda")
    sg.sgemm_ex2(torch.from_numpy(_stored(opA, ta)).cuda(), torch.from_numpy(_stored(opB, tb)).cuda(),
                 C, trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    assert torch.equal(C, plain)


def test_ex2_without_transposition_equals_ex():
    M, N, K = 700, 900, 333
    A = workloads.matrix(M, K, "normal", 901, 0).cuda()
    B = workloads.matrix(K, N, "normal", 901, 1).cuda()
    C0 = workloads.matrix(M, N, "normal", 901, 2).cuda()
    C1, C2 = C0.clone(), C0.clone()
    sg.sgemm_ex(A, B, C1, alpha=0.25, beta=3.0)
    sg.sgemm_ex2(A, B, C2, alpha=0.25, beta=3.0)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


def test_ex2_alpha_zero_k_zero_and_bad_flags():
    C0 = workloads.matrix(50, 40, "normal", 902, 2)
    A = torch.full((30, 50), float("nan"), device="cuda")      # stored K x M: trans_a
    B = torch.full((40, 30), float("nan"), device="cuda")      # stored N x K: trans_b
    C = C0.cuda()
    sg.sgemm_ex2(A, B, C, alpha=0.0, beta=-2.0, trans_a=True, trans_b=True)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), -2.0 * C0)
    C = torch.full((50, 40), float("nan"), device="cuda")
    sg.sgemm_ex2(torch.empty(0, 50, device="cuda"), torch.empty(40, 0, device="cuda"), C,
                 trans_a=True, trans_b=True)
    torch.cuda.synchronize()
    assert bool((C == 0).all())
    lib = sg.binding.load()
    for ta, tb in [(2, 0), (0, -1)]:
        st = lib.sgemm_ex2(0, ta, tb, 8, 8, 8, 1.0, A.data_ptr(), 8, B.data_ptr(), 8, 0.0,
                           C.data_ptr(), 8, 0)
        assert st == sg.binding.ERR_INVALID_VALUE
