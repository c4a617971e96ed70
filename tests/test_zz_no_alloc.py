"""The allocation-free Stream-K entry point, ``sgemm_streamk_static``.

Some callers cannot let a library allocate device memory: code that must
never wait on the whole device (cudaMalloc and cudaFree may synchronise it),
code with a memory budget fixed before work starts, and code inside a
framework whose own allocator owns the device memory.  For them the library
keeps the Stream-K scratch in one fixed array in its device image and this
entry point uses only that.

The tests call it through the C ABI twice in a row on shapes whose Stream-K
schedule splits tiles (so the array's counters and partial sums are used and
reused), check each result against the regular entry point's result within
the parity tolerance of the other GPU tests, 4 K 2^-24 sum_k |A B|, and check
that the device's free memory does not change across such calls.  The file
runs last (file name) so that a failure here leaves every other test run.
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


def test_static_calls_leave_device_memory_unchanged():
    """Two calls after the first (which looks up the array's address) change the device's
    free memory by nothing: the library allocates no device memory on this path."""
    shapes = [(1024, 1024, 1024, 73), (768, 1280, 1536, 74)]
    ops = []
    for M, N, K, seed in shapes:
        A_h = workloads.matrix(M, K, "normal", seed, 0)
        B_h = workloads.matrix(K, N, "normal", seed, 1)
        ops.append((A_h, B_h, A_h.cuda(), B_h.cuda(), torch.full((M, N), float("nan"), device="cuda")))
    A0, B0, C0 = ops[0][2], ops[0][3], ops[0][4]
    assert _static_call(A0, B0, C0) == sg.binding.OK      # set-up on this device
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for _, _, A, B, C in ops:
        C.fill_(float("nan"))
    torch.cuda.synchronize()
    for _, _, A, B, C in ops:
        assert _static_call(A, B, C) == sg.binding.OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert sg.query_device_status() == (0, 0)
    for (A_h, B_h, _, _, C), (M, N, K, _) in zip(ops, shapes):
        ref, E = oracle.sgemm_f64(A_h, B_h)
        check_within_bound(C.cpu().numpy(), ref, E, K, f"static scratch, no allocation {(M, N, K)}")
