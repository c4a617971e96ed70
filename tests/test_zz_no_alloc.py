"""The allocation-free Stream-K entry point, ``sgemm_streamk_static``.

Some callers cannot let a library allocate device memory: code running while
its stream is being captured, code that must never wait on the whole device
(cudaMalloc and cudaFree may synchronise it), and code with a memory budget
fixed before work starts.  For them the library keeps the Stream-K scratch
in one fixed array in its device image and this entry point uses only that.

The test calls it through the C ABI twice in a row on shapes whose Stream-K
schedule splits tiles (so the array's counters and partial sums are used and
reused), and checks each result against the regular entry point's result
within the parity tolerance of the other GPU tests, 4 K 2^-24 sum_k |A B|.
It runs last (file name) so that a failure here leaves every other test run.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_fp32_gemm_03_gb300 as sg
from dense_fp32_gemm_03_gb300 import binding, workloads

from parity import bound, check_within_bound

pytestmark = pytest.mark.gpu

STATIC_BYTES = 32 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _static_call(A, B, C):
    M, K = A.shape
    N = B.shape[1]
    return binding.sgemm_streamk_static_raw(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(),
                                            B.stride(0), C.data_ptr(), C.stride(0),
                                            torch.cuda.current_stream().cuda_stream)


def test_static_scratch_matches_regular_entry_point_twice():
    shapes = [(1024, 1024, 1024, 71), (640, 1536, 2048, 72)]
    for M, N, K, seed in shapes:
        assert 0 < sg.workspace_size(M, N, K, sg.STREAMK) <= STATIC_BYTES, "shape must use scratch"
        A_h = workloads.matrix(M, K, "uniform", seed, 0)
        B_h = workloads.matrix(K, N, "uniform", seed, 1)
        A, B = A_h.cuda(), B_h.cuda()
        regular = sg.sgemm(A, B, variant=sg.STREAMK)
        static = torch.full((M, N), float("nan"), device="cuda")
        assert _static_call(A, B, static) == sg.binding.OK
        torch.cuda.synchronize()
        assert sg.query_device_status() == (0, 0)
        _, E = oracle.sgemm_f64(A_h, B_h)
        got = static.cpu().numpy().astype(np.float64)
        ref = regular.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), f"{(M, N, K)}: tiles left unwritten"
        assert np.all(np.abs(got - ref) <= bound(K, E)), f"{(M, N, K)}: differs from sgemm()"
        C_ref, _ = oracle.sgemm_f64(A_h, B_h, with_abs=False)
        check_within_bound(got, C_ref, E, K, f"static scratch {(M, N, K)}")


def test_static_scratch_rejects_shapes_beyond_the_array():
    # 2 x 131 tiles of 128 x 256 leave 110 tiles to split over 152 CTAs: more
    # partial-sum slots than 32 MiB holds.  Nothing is launched.
    M, N, K = 256, 131 * 256, 1024
    need = sg.workspace_size(M, N, K, sg.STREAMK)
    if need <= STATIC_BYTES:
        pytest.skip(f"this device's schedule needs only {need} bytes here")
    A = torch.zeros(M, K, device="cuda")
    B = torch.zeros(K, N, device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    assert _static_call(A, B, C) == sg.binding.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())
