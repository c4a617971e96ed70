"""GPU parity with operands of more than 2^31 elements (8.6 GB each).

Offsets into A, B and C must be computed in 64 bits everywhere.  The
matrices are small integers given by formulas of their indices, built on the
GPU in row blocks; the oracle computes sampled rows or columns from the same
formulas on the host.  Every partial sum stays below 2^24, so results must
match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_fp32_gemm_03_gb300 as sg

from parity import check_exact

pytestmark = pytest.mark.gpu
BIG = 2 ** 31 + 2 ** 20   # elements, just past the 32-bit range


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if torch.cuda.get_device_properties(0).total_memory < 40 * 2 ** 30:
        pytest.skip("needs about 20 GB of device memory")
    import __graft_entry__
    __graft_entry__.build()
    yield
    st, site = sg.query_device_status()
    assert st == 0, f"device status {st} (site {site}) left after the module"


def _a_val(r, c):
    """A[r, c] in {-8..8}."""
    return ((r * 7 + c * 13) % 17 - 8)


def _b_val(r, c):
    """B[r, c] in {-3..3}."""
    return ((r * 5 + c * 3) % 7 - 3)


def _fill(rows, cols, fn, device="cuda", block=4096):
    """rows x cols float32 matrix fn(row, col), built in row blocks on `device`."""
    out = torch.empty(rows, cols, device=device)
    c = torch.arange(cols, device=device, dtype=torch.int64)
    for r0 in range(0, rows, block):
        r = torch.arange(r0, min(rows, r0 + block), device=device, dtype=torch.int64)[:, None]
        out[r0:r0 + r.shape[0]] = fn(r, c[None, :]).to(torch.float32)
    return out


def _host(rows_idx, cols, fn):
    r = np.asarray(rows_idx, dtype=np.int64)[:, None]
    c = np.arange(cols, dtype=np.int64)[None, :]
    return fn(r, c).astype(np.float32)


def test_a_beyond_2_31_elements():
    M, K, N = 32768, 65540, 128            # A: 2.148e9 elements
    assert M * K > BIG - 2 ** 20
    A = _fill(M, K, _a_val)
    B = _fill(K, N, _b_val)
    C = sg.sgemm(A, B)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 12345, M // 2 + 7, M - 2, M - 1])
    ref, E = oracle.sgemm_f64(_host(rows, K, _a_val), _host(np.arange(K), N, _b_val))
    assert E.max() < 2 ** 24
    r = torch.from_numpy(rows).cuda()
    check_exact(C[r].cpu().numpy(), ref, "A > 2^31 elements")
    # The bounds-checked kernel and the TF32 mode (small integers are exact in TF32).
    for what, run in (("guarded", lambda: sg.sgemm(A, B, variant=sg.GUARDED)),
                      ("tf32", lambda: sg.sgemm_tf32(A, B))):
        C = run()
        torch.cuda.synchronize()
        check_exact(C[r].cpu().numpy(), ref, f"A > 2^31 elements, {what}")
    del A, B, C
    torch.cuda.empty_cache()


def test_b_beyond_2_31_elements():
    M, K, N = 64, 65540, 32768             # B: 2.148e9 elements
    A = _fill(M, K, _a_val)
    B = _fill(K, N, _b_val)
    C = sg.sgemm(A, B)
    torch.cuda.synchronize()
    cols = np.array([0, 3, 9999, N // 2 + 1, N - 1])
    # Columns of B from the formula: B[:, cols] = transpose of rows `cols` of B^T.
    bt = _host(cols, K, lambda c, r: _b_val(r, c))
    ref, E = oracle.sgemm_f64(_host(np.arange(M), K, _a_val), np.ascontiguousarray(bt.T))
    assert E.max() < 2 ** 24
    check_exact(C[:, torch.from_numpy(cols).cuda()].cpu().numpy(), ref, "B > 2^31 elements")
    del A, B, C
    torch.cuda.empty_cache()


def test_c_beyond_2_31_elements():
    M, K, N = 65536, 16, 32800             # C: 2.150e9 elements
    A = _fill(M, K, _a_val)
    B = _fill(K, N, _b_val)
    C = torch.full((M, N), float("nan"), device="cuda")
    sg.sgemm(A, B, out=C)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 40000, M - 1, M - 1, 65535])
    cols = np.array([0, 32799, 16000, 0, 32799, 12345])
    ref, E = oracle.sgemm_entries_f64(_host(np.arange(M), K, _a_val),
                                      _host(np.arange(K), N, _b_val), rows, cols)
    ri, ci = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    check_exact(C[ri, ci].cpu().numpy(), ref, "C > 2^31 elements")
    assert not bool(torch.isnan(C[-1]).any()), "last row of C not written"
    for what, run in (("guarded", lambda: sg.sgemm(A, B, out=C, variant=sg.GUARDED)),
                      ("tf32", lambda: sg.sgemm_tf32(A, B, out=C))):
        C.fill_(float("nan"))
        run()
        torch.cuda.synchronize()
        check_exact(C[ri, ci].cpu().numpy(), ref, f"C > 2^31 elements, {what}")
        assert not bool(torch.isnan(C[-1]).any()), f"{what}: last row of C not written"
    del A, B, C
    torch.cuda.empty_cache()
