"""Pins of the FP32 acceptance bound itself (CPU).

The GPU results must satisfy |C_gpu - C_ref| <= 4 K 2^-24 sum_k |A B| per
element (tests/parity.py).  Two things make that bound the right one:

* it covers every legitimate FP32 evaluation.  The classical error bound for
  a K-term dot product accumulated in any order with unit roundoff u = 2^-24
  is gamma_K = K u / (1 - K u) times sum |a b|; rounding the final value
  adds u (1 + gamma_K).  The bound is at least that sum for every K the
  library accepts (closed form below), and FP32 accumulation in k order and
  split over K, emulated here, stays inside it;
* it is tight enough to catch plausible mistakes: at the 256^3 workload a
  dropped k-term, inputs rounded to bf16, and inputs rounded to TF32 (the
  tensor-core precision the pages contrast with FP32: "Beyond Kernel 7:
  Closing the Gap to cuBLAS on an H100 FP32 GEMM", section "The operation:
  GEMM and the precision of the comparison") each break it.  Integer inputs
  cannot show TF32 (small integers are exact in it), so this random-input
  bound is what separates the two precisions.
"""
from __future__ import annotations

import numpy as np

import oracle
from dense_fp32_gemm_03_gb300 import workloads
from parity import bound

U = 2.0 ** -24


def gamma(K: int) -> float:
    return K * U / (1.0 - K * U)


def test_bound_covers_gamma_k_and_the_final_rounding():
    for K in (1, 2, 3, 16, 255, 256, 1024, 4096, 16384, 65540, 1 << 20, 1 << 22):
        assert 4.0 * K * U >= gamma(K) + U * (1.0 + gamma(K)), K


def fp32_accumulate(A, B):
    """C = A B accumulated in FP32 in k order, one rounding per multiply-add
    (the product of two floats is exact in float64, so rounding the float64
    sum to float32 is the fused multiply-add's single rounding)."""
    acc = np.zeros((A.shape[0], B.shape[1]), np.float32)
    for k in range(A.shape[1]):
        acc = (acc.astype(np.float64)
               + np.outer(A[:, k].astype(np.float64), B[k, :].astype(np.float64))).astype(np.float32)
    return acc


def round_mantissa(x, keep_bits):
    """Round float32 values to `keep_bits` fraction bits (nearest, ties away)."""
    drop = 23 - keep_bits
    b = x.view(np.uint32).astype(np.uint64)
    b = ((b + (1 << (drop - 1))) & ~np.uint64((1 << drop) - 1) & np.uint64(0xFFFFFFFF))
    return b.astype(np.uint32).view(np.float32)


def _workload():
    w = workloads.SMALL_256
    A, B = workloads.operands(w)
    A, B = A.numpy(), B.numpy()
    C, E = oracle.sgemm_f64(A, B)
    return A, B, C, bound(w.K, E)


def test_fp32_orders_stay_inside():
    A, B, C, lim = _workload()
    assert np.all(np.abs(fp32_accumulate(A, B) - C) <= lim)
    # Split over K in four shares, partials added in share order (Stream-K's way).
    parts = [fp32_accumulate(A[:, i * 64:(i + 1) * 64], B[i * 64:(i + 1) * 64]) for i in range(4)]
    split = ((parts[0] + parts[1]) + parts[2]) + parts[3]
    assert np.all(np.abs(split - C) <= lim)


def test_plausible_mistakes_break_it():
    A, B, C, lim = _workload()
    dropped = fp32_accumulate(A[:, 1:], B[1:])
    assert np.any(np.abs(dropped - C) > lim), "a dropped k-term passed"
    bf16 = fp32_accumulate(round_mantissa(A, 7), round_mantissa(B, 7))
    assert np.any(np.abs(bf16 - C) > lim), "bf16 inputs passed"
    tf32 = fp32_accumulate(round_mantissa(A, 10), round_mantissa(B, 10))
    assert np.any(np.abs(tf32 - C) > lim), "TF32 inputs passed"
