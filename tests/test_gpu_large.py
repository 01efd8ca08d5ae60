"""Operands and outputs of more than 2**31 elements: every address in the
kernels is formed in 64 bits.  The inputs are drawn on the device; rows of C on
both sides of the 2**31-element boundary (and the last row) are checked against
the fp64 oracle on the gathered rows of A, which gives exactly those rows of C.

Tolerance: 1e-6 * K * max|A| * max|B| (FP32 path), 1e-5 * ... (3xTF32 path)."""
import numpy as np
import pytest

from dense_fp32_gemm_09_gb300 import check, load, sgemm, sgemm_run_op

pytestmark = pytest.mark.gpu


def device_uniform(torch, shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.rand(shape, device="cuda", generator=g) * 2 - 1


def rows_across(boundary_row, last_row):
    return sorted({0, boundary_row - 1, boundary_row, boundary_row + 1, last_row})


@pytest.fixture
def big(cuda):
    torch = cuda
    yield torch
    torch.cuda.empty_cache()


def test_a_past_2_31_elements(big, oracle_mod):
    torch = big
    M, N, K = 67000, 64, 32768                    # A: 2.2e9 elements (8.8 GB)
    A = device_uniform(torch, (M, K), 1)
    B = device_uniform(torch, (K, N), 2)
    C = sgemm(A, B)
    torch.cuda.synchronize()
    rows = rows_across((1 << 31) // K, M - 1)
    ref = oracle_mod.gemm_f64(A[rows].cpu().numpy(), B.cpu().numpy())
    got = C[rows].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref)) <= 1e-6 * K
    del A, B, C


def test_c_past_2_31_elements(big, oracle_mod):
    torch = big
    M, N, K = 50000, 45000, 8                      # C: 2.25e9 elements (9 GB)
    A = device_uniform(torch, (M, K), 3)
    B = device_uniform(torch, (K, N), 4)
    C = sgemm(A, B)
    torch.cuda.synchronize()
    rows = rows_across((1 << 31) // N, M - 1)
    ref = oracle_mod.gemm_f64(A[rows].cpu().numpy(), B.cpu().numpy())
    got = C[rows].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref)) <= 1e-6 * K
    del A, B, C


def test_transposed_a_past_2_31_elements(big, oracle_mod):
    torch = big
    M, N, K = 67000, 64, 32768                    # A stored K x M (8.8 GB), transposed inside
    At = device_uniform(torch, (K, M), 5)
    B = device_uniform(torch, (K, N), 6)
    C = torch.empty(M, N, device="cuda")
    assert sgemm_run_op(1, 0, M, N, K, 1.0, At.data_ptr(), M, B.data_ptr(), N, 0.0,
                        C.data_ptr(), N) == 0
    torch.cuda.synchronize()
    rows = rows_across((1 << 31) // K, M - 1)
    ref = oracle_mod.gemm_f64(At[:, rows].t().contiguous().cpu().numpy(), B.cpu().numpy())
    got = C[rows].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref)) <= 1e-6 * K
    del At, B, C


def test_tf32x3_a_past_2_31_elements(big, oracle_mod):
    torch = big
    lib = load()
    M, N, K = 67000, 64, 32768
    A = device_uniform(torch, (M, K), 7)
    B = device_uniform(torch, (K, N), 8)
    C = torch.empty(M, N, device="cuda")
    check(lib.sgemm_tf32x3_run_ex(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0,
                                  C.data_ptr(), N, None, 0,
                                  torch.cuda.current_stream().cuda_stream), "tf32x3")
    torch.cuda.synchronize()
    check(lib.sgemm_device_status(), "device status")
    rows = rows_across((1 << 31) // K, M - 1)
    ref = oracle_mod.gemm_f64(A[rows].cpu().numpy(), B.cpu().numpy())
    got = C[rows].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref)) <= 1e-5 * K
    del A, B, C
