"""GPU parity of the size-specialized instances (M = N = K = 768, 1024, 4096).

The specialized instance runs the same Stream-K schedule as the generic
kernel with the shape compiled in, so its output must equal the generic
variant's bit for bit, and meet the oracle's bound like every variant.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_fp32_gemm_03_gb300 as sg
from dense_fp32_gemm_03_gb300 import binding, workloads

from parity import check_within_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the specialized schedules are compiled for 152 SMs")
    yield
    st, site = sg.query_device_status()
    assert st == 0, f"device status {st} (site {site}) left after the module"


def _sweep(n):
    return next(w for w in workloads.SWEEP if w.M == n)


@pytest.mark.parametrize("w,generic", [(_sweep(768), sg.STREAMK_SMALL),
                                       (workloads.SQUARE_1024, sg.STREAMK_SMALL),
                                       (workloads.SQUARE_4096, sg.STREAMK)],
                         ids=["768", "1024", "4096"])
def test_selected_and_bit_identical_to_generic(w, generic):
    A, B = (x.cuda() for x in workloads.operands(w))
    C_spec = torch.full((w.M, w.N), float("nan"), device="cuda")
    C_gen = torch.full((w.M, w.N), float("nan"), device="cuda")
    assert sg.select_variant(A, B, C_spec) == sg.SPECIALIZED
    sg.sgemm(A, B, out=C_spec, variant=sg.SPECIALIZED)
    sg.sgemm(A, B, out=C_gen, variant=generic)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(C_spec).all())
    assert torch.equal(C_spec, C_gen)


def test_1024_full_compare():
    w = workloads.SQUARE_1024
    A, B = workloads.operands(w)
    ref, E = oracle.sgemm_f64(A, B)
    C = sg.sgemm(A.cuda(), B.cuda(), variant=sg.SPECIALIZED)
    torch.cuda.synchronize()
    check_within_bound(C.cpu().numpy(), ref, E, w.K, "1024^3 specialized")


def test_768_full_compare():
    w = _sweep(768)
    A, B = workloads.operands(w)
    ref, E = oracle.sgemm_f64(A, B)
    C = sg.sgemm(A.cuda(), B.cuda(), variant=sg.SPECIALIZED)
    torch.cuda.synchronize()
    check_within_bound(C.cpu().numpy(), ref, E, w.K, "768^3 specialized")


def test_4096_sampled_and_row_block():
    w = workloads.SQUARE_4096
    A, B = workloads.operands(w)
    C = sg.sgemm(A.cuda(), B.cuda(), variant=sg.SPECIALIZED).cpu().numpy()
    r, c = workloads.sample_indices(w.M, w.N, 4096, w.seed)
    ref, E = oracle.sgemm_entries_f64(A, B, r.numpy(), c.numpy())
    check_within_bound(C[r.numpy(), c.numpy()], ref, E, w.K, "4096^3 specialized (sampled)")
    rows = slice(3968, 4096)     # the last tile row: split (Stream-K) tiles
    ref, E = oracle.sgemm_f64(A[rows], B)
    check_within_bound(C[rows], ref, E, w.K, "4096^3 specialized, last tile row")


def test_integer_inputs_exact_at_1024():
    A = workloads.matrix(1024, 1024, "int8range", 71, 0)
    B = workloads.matrix(1024, 1024, "int8range", 71, 1)
    ref, E = oracle.sgemm_f64(A, B)
    assert E.max() < 2 ** 24
    C = sg.sgemm(A.cuda(), B.cuda(), variant=sg.SPECIALIZED)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("shape", [(512, 512, 512), (1024, 1024, 1020), (4096, 4096, 4092),
                                   (1024, 1024, 2048), (1536, 1536, 1536), (2048, 2048, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
def test_other_shapes_unsupported(shape):
    M, N, K = shape
    A = torch.zeros(M, K, device="cuda")
    B = torch.zeros(K, N, device="cuda")
    C = torch.empty(M, N, device="cuda")
    assert sg.select_variant(A, B, C) != sg.SPECIALIZED
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm(A, B, out=C, variant=sg.SPECIALIZED)
    assert e.value.status == binding.ERR_UNSUPPORTED


def test_alpha_beta_at_a_specialized_shape_uses_the_generic_instance():
    w = workloads.SQUARE_1024
    A, B = workloads.operands(w)
    C0 = workloads.matrix(1024, 1024, "uniform", 72, 2)
    C = C0.cuda()
    sg.sgemm_ex(A.cuda(), B.cuda(), C, alpha=0.5, beta=-2.0)
    torch.cuda.synchronize()
    ref = oracle.sgemm_ex_f64(A.numpy(), B.numpy(), alpha=0.5, beta=-2.0, C0=C0.numpy())
    _, E = oracle.sgemm_f64(A, B)
    U24 = 2.0 ** -24
    lim = 0.5 * 4 * 1024 * U24 * E + 4 * U24 * (0.5 * E + 2.0 * np.abs(C0.numpy()))
    assert not np.any(np.abs(C.cpu().numpy().astype(np.float64) - ref) > lim)


def test_misaligned_c_at_a_specialized_shape():
    """A C the plain instance cannot store (ldc = 1025) at the specialized shape."""
    w = workloads.SQUARE_1024
    A, B = workloads.operands(w)
    ref, E = oracle.sgemm_f64(A, B)
    big = torch.full((1024, 1025), float("nan"), device="cuda")
    C = big[:, :1024]
    assert sg.select_variant(A.cuda(), B.cuda(), C) == sg.STAGED
    sg.sgemm(A.cuda(), B.cuda(), out=C)
    torch.cuda.synchronize()
    check_within_bound(C.cpu().numpy(), ref, E, w.K, "1024^3 ldc 1025")
