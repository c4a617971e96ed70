"""Pins for the CPU oracle (CPU only).

The oracle restates the definition C[m, n] = sum_k A[m, k] B[k, n] ("Beyond
Kernel 7: Closing the Gap to cuBLAS on an H100 FP32 GEMM", section "The
operation: GEMM and the precision of the comparison").  The pages print no
worked numeric example, so it is pinned to facts fixed by mathematics instead:

* identity and permutation matrices (one nonzero product per output: exact);
* the rank-1 closed form (u v^T)(w z^T) = (v . w) u z^T, exact on dyadic inputs;
* brute force on every shape with M, N, K in 1..8 against exact rational
  arithmetic (Python ``fractions``), on integer and on random float inputs;
* an independent float64 library product (numpy matmul);
* K-split additivity and the transpose identity (AB)^T = B^T A^T;
* the magnitude E = |A| |B| and the sampled-entry routine.

Each pin is a function of a ``gemm`` callable so that ``test_pins_catch_mutants``
can show that plausible mistakes (a transposed operand, a dropped term, a shifted
index, a flipped sign, float32 accumulation) fail at least one pin.
"""
from fractions import Fraction
import itertools

import numpy as np
import pytest

import oracle
from dense_fp32_gemm_03_gb300 import workloads

U53 = 2.0 ** -53  # unit roundoff of float64


def _oracle_gemm(A, B):
    return oracle.sgemm_f64(A, B, with_abs=False)[0]


def _exact(A, B):
    """Exact rational product as a float64 array of correctly rounded values, plus E."""
    M, K = A.shape
    N = B.shape[1]
    C = np.zeros((M, N))
    E = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = Fraction(0)
            e = Fraction(0)
            for k in range(K):
                p = Fraction(float(A[m, k])) * Fraction(float(B[k, n]))
                s += p
                e += abs(p)
            C[m, n] = float(s)
            E[m, n] = float(e)
    return C, E


def _rng(seed):
    return np.random.default_rng(seed)


def _dyadic(rng, shape, bits=10):
    """Float32 values k/2^bits in [-1, 1]: products of two are exact in float32."""
    return (rng.integers(-(2 ** bits), 2 ** bits + 1, size=shape) / 2.0 ** bits).astype(np.float32)


# ----------------------------------------------------------------- the pins
def pin_identity(gemm):
    rng = _rng(1)
    A = rng.standard_normal((7, 5)).astype(np.float32)
    B = rng.standard_normal((5, 9)).astype(np.float32)
    assert np.array_equal(gemm(A, np.eye(5, dtype=np.float32)), A.astype(np.float64))
    assert np.array_equal(gemm(np.eye(5, dtype=np.float32), B), B.astype(np.float64))


def pin_permutation(gemm):
    rng = _rng(2)
    A = rng.standard_normal((6, 11)).astype(np.float32)
    B = rng.standard_normal((11, 4)).astype(np.float32)
    p = rng.permutation(11)
    P = np.eye(11, dtype=np.float32)[p]          # (P B)[i] = B[p[i]]
    assert np.array_equal(gemm(P, B), B[p].astype(np.float64))
    q = rng.permutation(11)
    Q = np.eye(11, dtype=np.float32)[:, q]       # (A Q)[:, j] = A[:, q[j]]
    assert np.array_equal(gemm(A, Q), A[:, q].astype(np.float64))


def pin_rank1(gemm):
    """(u v^T)(w z^T) = (v . w) u z^T with dyadic vectors: every step exact."""
    rng = _rng(3)
    M, K, N = 9, 13, 7
    u, v, w, z = (_dyadic(rng, s, bits=6) for s in (M, K, K, N))
    A = np.outer(u, v).astype(np.float32)  # exact: 12-bit products
    B = np.outer(w, z).astype(np.float32)
    assert np.array_equal(A.astype(np.float64), np.outer(u.astype(np.float64), v))
    vw = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(v, w))
    expect = np.array([[float(vw * Fraction(float(um)) * Fraction(float(zn))) for zn in z] for um in u])
    assert np.array_equal(gemm(A, B), expect)
    # Small-integer vectors: the same identity, in integers.
    ui, vi, wi, zi = (rng.integers(-8, 9, size=s) for s in (M, K, K, N))
    Ai = np.outer(ui, vi).astype(np.float32)
    Bi = np.outer(wi, zi).astype(np.float32)
    assert np.array_equal(gemm(Ai, Bi), (int(vi @ wi) * np.outer(ui, zi)).astype(np.float64))


def pin_bruteforce_integer(gemm):
    """All shapes 1..8: integer inputs, exact against Python integer sums."""
    rng = _rng(4)
    for M, N, K in itertools.product(range(1, 9), repeat=3):
        A = rng.integers(-8, 9, size=(M, K))
        B = rng.integers(-8, 9, size=(K, N))
        expect = np.array([[sum(int(A[m, k]) * int(B[k, n]) for k in range(K))
                            for n in range(N)] for m in range(M)], dtype=np.float64)
        got = gemm(A.astype(np.float32), B.astype(np.float32))
        assert np.array_equal(got, expect), (M, N, K)


def pin_bruteforce_random(gemm):
    """All shapes 1..8: random float inputs against exact rationals, float64 error bound."""
    rng = _rng(5)
    for M, N, K in itertools.product(range(1, 9), repeat=3):
        A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
        B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
        exact, E = _exact(A, B)
        got = gemm(A, B)
        # Recursive summation of K exact products: |err| <= (K-1) u / (1 - (K-1) u) * E,
        # plus the rounding of the exact value to float64 in ``_exact``.
        tol = (K * U53 * 1.001) * E + U53 * np.abs(exact)
        assert np.all(np.abs(got - exact) <= tol), (M, N, K)


def pin_library(gemm):
    """An independent float64 product (numpy's BLAS) agrees to float64 rounding."""
    rng = _rng(6)
    A = rng.standard_normal((37, 53)).astype(np.float32)
    B = rng.standard_normal((53, 29)).astype(np.float32)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    E = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    assert np.all(np.abs(gemm(A, B) - ref) <= 2 * 53 * U53 * E)


def pin_ksplit(gemm):
    rng = _rng(7)
    A = rng.integers(-8, 9, size=(10, 23)).astype(np.float32)
    B = rng.integers(-8, 9, size=(23, 12)).astype(np.float32)
    for k1 in (1, 9, 22):
        assert np.array_equal(gemm(A, B), gemm(A[:, :k1], B[:k1]) + gemm(A[:, k1:], B[k1:]))


def pin_transpose(gemm):
    """(A B)^T = B^T A^T, bit for bit: the same products are summed in the same k order."""
    rng = _rng(8)
    A = rng.standard_normal((5, 19)).astype(np.float32)
    B = rng.standard_normal((19, 8)).astype(np.float32)
    lhs = gemm(A, B).T
    rhs = gemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T))
    assert np.array_equal(lhs, rhs)


PINS = [pin_identity, pin_permutation, pin_rank1, pin_bruteforce_integer,
        pin_bruteforce_random, pin_library, pin_ksplit, pin_transpose]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(_oracle_gemm)


# ------------------------------------------------------- mutants must fail a pin
def _mut_transposed_b(A, B):
    """Reads B[k, n] at flat index n*K + k instead of k*N + n (a swapped index)."""
    K, N = B.shape
    Bw = np.ascontiguousarray(B).reshape(-1).reshape(N, K).T
    return A.astype(np.float64) @ Bw.astype(np.float64)


def _mut_drop_last_k(A, B):
    return A[:, :-1].astype(np.float64) @ B[:-1].astype(np.float64)


def _mut_shift_index(A, B):
    return A.astype(np.float64) @ np.roll(B.astype(np.float64), 1, axis=0)


def _mut_sign(A, B):
    C = A.astype(np.float64) @ B.astype(np.float64)
    C[-1, -1] = -C[-1, -1]
    return C


def _mut_f32_accumulate(A, B):
    M, K = A.shape
    C = np.zeros((M, B.shape[1]), dtype=np.float32)
    for k in range(K):
        C = C + np.outer(A[:, k], B[k]).astype(np.float32)
    return C.astype(np.float64)


MUTANTS = [_mut_transposed_b, _mut_drop_last_k, _mut_shift_index, _mut_sign, _mut_f32_accumulate]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda f: f.__name__)
def test_pins_catch_mutants(mutant):
    failed = 0
    for pin in PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed >= 1, f"no pin caught {mutant.__name__}"


# --------------------------------------------------------- properties of the API
def test_abs_magnitude_is_product_of_absolutes():
    rng = _rng(9)
    A = rng.standard_normal((14, 31)).astype(np.float32)
    B = rng.standard_normal((31, 17)).astype(np.float32)
    _, E = oracle.sgemm_f64(A, B)
    C_abs, _ = oracle.sgemm_f64(np.abs(A), np.abs(B), with_abs=False)
    assert np.array_equal(E, C_abs)


def test_entries_match_full_product():
    A, B = workloads.matrix(40, 70, "normal", 5, 0), workloads.matrix(70, 33, "normal", 5, 1)
    C, E = oracle.sgemm_f64(A, B)
    r, c = workloads.sample_indices(40, 33, 100, 3)
    ce, ee = oracle.sgemm_entries_f64(A, B, r.numpy(), c.numpy())
    assert np.array_equal(ce, C[r.numpy(), c.numpy()])
    assert np.array_equal(ee, E[r.numpy(), c.numpy()])


def test_row_strides():
    rng = _rng(10)
    big_a = rng.standard_normal((12, 40)).astype(np.float32)
    big_b = rng.standard_normal((25, 50)).astype(np.float32)
    A, B = big_a[:, 3:28], big_b[:, 5:16]       # row strides 40 and 50, not the widths
    assert A.strides[0] == 160 and B.strides[0] == 200
    got = oracle.sgemm_f64(A, B, with_abs=False)[0]
    ref = oracle.sgemm_f64(np.ascontiguousarray(A), np.ascontiguousarray(B), with_abs=False)[0]
    assert np.array_equal(got, ref)


def test_degenerate_shapes():
    z = oracle.sgemm_f64(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32))
    assert np.array_equal(z[0], np.zeros((3, 4))) and np.array_equal(z[1], np.zeros((3, 4)))
    assert oracle.sgemm_f64(np.zeros((0, 5), np.float32), np.ones((5, 4), np.float32))[0].shape == (0, 4)
    assert oracle.sgemm_f64(np.ones((3, 5), np.float32), np.ones((5, 0), np.float32))[0].shape == (3, 0)
    with pytest.raises(ValueError):
        oracle.sgemm_f64(np.ones((3, 5), np.float32), np.ones((4, 2), np.float32))


def test_nan_propagates_along_its_row_and_column():
    A = np.ones((4, 6), np.float32)
    B = np.ones((6, 5), np.float32)
    A[2, 3] = np.nan
    C = oracle.sgemm_f64(A, B, with_abs=False)[0]
    assert np.all(np.isnan(C[2])) and not np.any(np.isnan(np.delete(C, 2, axis=0)))
    B2 = np.ones((6, 5), np.float32)
    B2[1, 4] = np.inf
    C2 = oracle.sgemm_f64(np.ones((4, 6), np.float32), B2, with_abs=False)[0]
    assert np.all(np.isinf(C2[:, 4])) and np.all(np.isfinite(C2[:, :4]))


def test_integer_workload_partial_sums_stay_exact():
    """The integer workload keeps every partial sum below 2^24 (256 * 64 = 16384)."""
    w = workloads.SMALL_256_INT
    A, B = workloads.operands(w)
    assert float(A.abs().max()) <= 8 and float(B.abs().max()) <= 8
    assert w.K * 8 * 8 < 2 ** 24
    _, E = oracle.sgemm_f64(A, B)
    assert E.max() < 2 ** 24


# ------------------------------------------------- the scaled, two-layout form
def test_ex_reduces_to_the_plain_definition():
    rng = _rng(11)
    A = rng.standard_normal((9, 13)).astype(np.float32)
    B = rng.standard_normal((13, 6)).astype(np.float32)
    plain = oracle.sgemm_f64(A, B, with_abs=False)[0]
    assert np.array_equal(oracle.sgemm_ex_f64(A, B), plain)
    # A power-of-two alpha scales exactly.
    assert np.array_equal(oracle.sgemm_ex_f64(A, B, alpha=-4.0), -4.0 * plain)


def test_ex_beta_reads_c_and_beta_zero_ignores_it():
    rng = _rng(12)
    A = rng.integers(-8, 9, size=(7, 5)).astype(np.float32)
    B = rng.integers(-8, 9, size=(5, 4)).astype(np.float32)
    C0 = rng.integers(-8, 9, size=(7, 4)).astype(np.float32)
    expect = 3.0 * (A.astype(np.int64) @ B.astype(np.int64)) - 2.0 * C0
    assert np.array_equal(oracle.sgemm_ex_f64(A, B, alpha=3.0, beta=-2.0, C0=C0), expect)
    nan_c = np.full((7, 4), np.nan, dtype=np.float32)
    assert np.array_equal(oracle.sgemm_ex_f64(A, B, alpha=1.0, beta=0.0, C0=nan_c),
                          (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))
    # alpha = 0 leaves beta * C0 (A and B only multiply a zero).
    assert np.array_equal(oracle.sgemm_ex_f64(A, B, alpha=0.0, beta=0.5, C0=C0), 0.5 * C0)


def test_ex_column_major_is_the_same_product():
    rng = _rng(13)
    A = rng.standard_normal((6, 11)).astype(np.float32)
    B = rng.standard_normal((11, 8)).astype(np.float32)
    C0 = rng.standard_normal((6, 8)).astype(np.float32)
    row = oracle.sgemm_ex_f64(A, B, alpha=0.5, beta=2.0, C0=C0)
    col = oracle.sgemm_ex_f64(np.asfortranarray(A), np.asfortranarray(B), alpha=0.5, beta=2.0,
                              C0=np.asfortranarray(C0), col_major=True)
    assert np.array_equal(row, col)


# ------------------------------- per-operand transposition: the op() form
# op(A) = A or A^T and op(B) = B or B^T, the stored arrays being A (M x K or
# K x M) and B (K x N or N x K).  Pins, each a function of an ``op`` callable
# (stored A, stored B, trans_a, trans_b, col_major, alpha, beta, C0) so that
# planted mistakes can be shown to fail one:
# * small integers: exact against numpy int64 products of explicit transposes,
#   with alpha, beta and both storage orders, on square and non-square shapes;
# * random floats: bit-identical to the plain pinned oracle applied to the
#   explicitly transposed (contiguous) operands -- the same products summed
#   in the same k order;
# * the transpose identity (op(A) op(B))^T = op(B)^T op(A)^T, bit-exact.
TRANS = [(False, False), (True, False), (False, True), (True, True)]


def _op_oracle(A, B, ta, tb, col_major=False, alpha=1.0, beta=0.0, C0=None):
    return oracle.sgemm_op_f64(A, B, trans_a=ta, trans_b=tb, alpha=alpha, beta=beta, C0=C0,
                               col_major=col_major)


def _stored(x, t):
    return np.ascontiguousarray(x.T if t else x).astype(np.float32)


def pin_op_integer_exact(op):
    rng = _rng(21)
    for M, N, K in [(7, 5, 9), (6, 6, 6)]:
        for ta, tb in TRANS:
            for cm in (False, True):
                opA = rng.integers(-8, 9, size=(M, K)).astype(np.int64)
                opB = rng.integers(-8, 9, size=(K, N)).astype(np.int64)
                C0 = rng.integers(-8, 9, size=(M, N)).astype(np.int64)
                expect = (3 * (opA @ opB) - 2 * C0).astype(np.float64)
                got = op(_stored(opA, ta), _stored(opB, tb), ta, tb, cm, alpha=3.0, beta=-2.0,
                         C0=C0.astype(np.float32))
                assert np.array_equal(got, expect), (M, N, K, ta, tb, cm)


def pin_op_explicit_transposes(op):
    rng = _rng(22)
    for M, N, K in [(9, 4, 13), (8, 8, 8)]:
        opA = rng.standard_normal((M, K)).astype(np.float32)
        opB = rng.standard_normal((K, N)).astype(np.float32)
        plain = oracle.sgemm_f64(opA, opB, with_abs=False)[0]
        for ta, tb in TRANS:
            got = op(_stored(opA, ta), _stored(opB, tb), ta, tb)
            assert np.array_equal(got, plain), (M, N, K, ta, tb)


def pin_op_transpose_identity(op):
    rng = _rng(23)
    for M, N, K in [(5, 11, 7), (6, 6, 6)]:
        opA = rng.standard_normal((M, K)).astype(np.float32)
        opB = rng.standard_normal((K, N)).astype(np.float32)
        for ta, tb in TRANS:
            A, B = _stored(opA, ta), _stored(opB, tb)
            C = op(A, B, ta, tb)
            # op(B)^T is the stored B read with the other flag; likewise op(A)^T.
            Ct = op(B, A, not tb, not ta)
            assert np.array_equal(C.T, Ct), (M, N, K, ta, tb)


OP_PINS = [pin_op_integer_exact, pin_op_explicit_transposes, pin_op_transpose_identity]


@pytest.mark.parametrize("pin", OP_PINS, ids=lambda p: p.__name__)
def test_op_oracle_pin(pin):
    pin(_op_oracle)


def _op_reference_parts(A, B, ta, tb):
    opA = (A.T if ta else A).astype(np.float64)
    opB = (B.T if tb else B).astype(np.float64)
    return opA, opB


def _opmut_swapped_flags(A, B, ta, tb, col_major=False, alpha=1.0, beta=0.0, C0=None):
    """Applies trans_b to A and trans_a to B."""
    opA, opB = _op_reference_parts(A, B, tb, ta)
    r = alpha * (opA @ opB)
    return r + beta * C0.astype(np.float64) if beta != 0 else r


def _opmut_ignores_trans_a(A, B, ta, tb, col_major=False, alpha=1.0, beta=0.0, C0=None):
    opA, opB = _op_reference_parts(A, B, False, tb)
    r = alpha * (opA @ opB)
    return r + beta * C0.astype(np.float64) if beta != 0 else r


def _opmut_c0_transposed(A, B, ta, tb, col_major=False, alpha=1.0, beta=0.0, C0=None):
    """Reads C0 transposed whenever A is transposed."""
    opA, opB = _op_reference_parts(A, B, ta, tb)
    r = alpha * (opA @ opB)
    if beta != 0:
        c = C0.astype(np.float64)
        r = r + beta * (c.T if ta else c)
    return r


def _opmut_beta_sign(A, B, ta, tb, col_major=False, alpha=1.0, beta=0.0, C0=None):
    opA, opB = _op_reference_parts(A, B, ta, tb)
    r = alpha * (opA @ opB)
    return r - beta * C0.astype(np.float64) if beta != 0 else r


def _opmut_drops_alpha_when_transposed(A, B, ta, tb, col_major=False, alpha=1.0, beta=0.0, C0=None):
    opA, opB = _op_reference_parts(A, B, ta, tb)
    r = (1.0 if (ta or tb) else alpha) * (opA @ opB)
    return r + beta * C0.astype(np.float64) if beta != 0 else r


OP_MUTANTS = [_opmut_swapped_flags, _opmut_ignores_trans_a, _opmut_c0_transposed, _opmut_beta_sign,
              _opmut_drops_alpha_when_transposed]


@pytest.mark.parametrize("mutant", OP_MUTANTS, ids=lambda f: f.__name__)
def test_op_pins_catch_mutants(mutant):
    failed = 0
    for pin in OP_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed >= 1, f"no pin caught {mutant.__name__}"


def test_op_without_transposition_is_the_ex_form():
    rng = _rng(24)
    A = rng.standard_normal((10, 7)).astype(np.float32)
    B = rng.standard_normal((7, 12)).astype(np.float32)
    C0 = rng.standard_normal((10, 12)).astype(np.float32)
    for cm in (False, True):
        assert np.array_equal(
            oracle.sgemm_op_f64(A, B, alpha=0.75, beta=-1.5, C0=C0, col_major=cm),
            oracle.sgemm_ex_f64(A, B, alpha=0.75, beta=-1.5, C0=C0, col_major=cm))


def test_op_beta_zero_never_reads_c():
    rng = _rng(25)
    A = rng.integers(-4, 5, size=(6, 9)).astype(np.float32)
    B = rng.integers(-4, 5, size=(5, 6)).astype(np.float32)   # stored N x K: trans_b
    nan_c = np.full((9, 5), np.nan, dtype=np.float32)
    got = oracle.sgemm_op_f64(A, B, trans_a=True, trans_b=True, beta=0.0, C0=nan_c)
    assert np.array_equal(got, (A.T.astype(np.int64) @ B.T.astype(np.int64)).astype(np.float64))
