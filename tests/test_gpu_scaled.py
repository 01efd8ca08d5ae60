"""GPU parity of the scaled form C = alpha * A.B + beta * C (sgemm_run_ex) with the
fp64 oracle's oracle_gemm_f64_ex.

Tolerance: 1e-6 * (|alpha| * K * max|A| * max|B| + |beta| * max|C0|), the FP32
product tolerance extended by the beta term.  Exact cases (small integers, alpha
= 0, K = 0) must match bit for bit."""
import numpy as np
import pytest

from conftest import padded_device
from dense_fp32_gemm_09_gb300 import SgemmError, kernel_table, load, sgemm
from dense_fp32_gemm_09_gb300.workloads import make_inputs, random_pair, small_int_pair

pytestmark = pytest.mark.gpu


def tol(alpha, beta, A, B, C0):
    K = A.shape[1]
    return 1e-6 * (abs(alpha) * K * float(A.abs().max()) * float(B.abs().max())
                   + abs(beta) * float(C0.abs().max()))


def _ids():
    try:
        return [k["name"] for k in kernel_table()]
    except Exception:
        return []


@pytest.mark.parametrize("kname", _ids())
def test_each_kernel_scaled(cuda, oracle_mod, kname):
    torch = cuda
    kid = {k["name"]: k["kernel_id"] for k in kernel_table()}[kname]
    vec4 = {k["name"]: k["vec"] for k in kernel_table()}[kname] == 4
    for (M, N, K) in [(65, 63, 129), (300, 260, 1000), (257, 383, 77)]:
        A, B = random_pair(M, N, K, seed=M + N)
        # leading dimensions padded to multiples of 4 so 16-byte entries can run
        dA, dB = padded_device(torch, A, (-K) % 4 + 4), padded_device(torch, B, (-N) % 4 + 4)
        C0 = torch.randn(M, N, generator=torch.Generator().manual_seed(K))
        for alpha, beta in [(1.5, -0.75), (-2.0, 0.0), (0.5, 1.0)]:
            for schedule in (1, 2):
                ldc = N + (-N) % 4 + (4 if vec4 else 1)
                buf = torch.full((M, ldc), 7.0, device="cuda")
                C = buf[:, :N]
                C.copy_(C0)
                sgemm(dA, dB, out=C, alpha=alpha, beta=beta, kernel_id=kid, schedule=schedule)
                torch.cuda.synchronize()
                assert torch.all(buf[:, N:] == 7.0), "write outside C"
                ref = oracle_mod.gemm_f64_ex(alpha, A.numpy(), B.numpy(), beta, C0.numpy())
                err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
                assert err <= tol(alpha, beta, A, B, C0), (kname, (M, N, K), alpha, beta, err)


@pytest.mark.parametrize("name", ["sgemm_1024", "sgemm_ragged_3001x2047x1999"])
def test_workload_scaled(cuda, oracle_mod, name):
    torch = cuda
    A, B = make_inputs(name)
    M, N = A.shape[0], B.shape[1]
    C0 = torch.randn(M, N, generator=torch.Generator().manual_seed(1))
    C = C0.cuda()
    sgemm(A.cuda(), B.cuda(), out=C, alpha=0.75, beta=-1.25)
    ref = oracle_mod.gemm_f64_ex(0.75, A.numpy(), B.numpy(), -1.25, C0.numpy())
    err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
    assert err <= tol(0.75, -1.25, A, B, C0)


def test_scaled_small_integers_bit_exact(cuda, oracle_mod):
    torch = cuda
    A, B = small_int_pair(777, 515, 1999, seed=3)
    C0 = torch.randint(-1000, 1001, (777, 515), generator=torch.Generator().manual_seed(2)).float()
    C = C0.cuda()
    sgemm(A.cuda(), B.cuda(), out=C, alpha=2.0, beta=-3.0)
    ref = oracle_mod.gemm_f64_ex(2.0, A.numpy(), B.numpy(), -3.0, C0.numpy()).astype(np.float32)
    assert np.array_equal(C.cpu().numpy(), ref)


def test_beta_zero_ignores_old_C(cuda, oracle_mod):
    torch = cuda
    A, B = random_pair(300, 200, 500, seed=8)
    C = torch.full((300, 200), float("nan"), device="cuda")
    sgemm(A.cuda(), B.cuda(), out=C, alpha=3.0, beta=0.0)
    ref = oracle_mod.gemm_f64_ex(3.0, A.numpy(), B.numpy(), 0.0, None)
    assert torch.isfinite(C).all()
    assert np.max(np.abs(C.cpu().numpy() - ref)) <= 3.0 * 1e-6 * 500


def test_alpha_zero_and_empty_K_scale_C_only(cuda):
    torch = cuda
    C0 = torch.randn(50, 70)
    A = torch.full((50, 30), float("nan"), device="cuda")   # not read when alpha == 0
    B = torch.full((30, 70), float("nan"), device="cuda")
    C = C0.cuda()
    sgemm(A, B, out=C, alpha=0.0, beta=0.5)
    assert torch.equal(C.cpu(), C0 * np.float32(0.5))
    C = C0.cuda()
    sgemm(torch.empty(50, 0, device="cuda"), torch.empty(0, 70, device="cuda"), out=C,
          alpha=2.0, beta=-1.5)
    assert torch.equal(C.cpu(), C0 * np.float32(-1.5))
    C = torch.full((50, 70), float("nan"), device="cuda")
    sgemm(A, B, out=C, alpha=0.0, beta=0.0)
    assert torch.all(C == 0)


def test_nan_scalars_rejected(cuda):
    torch = cuda
    A = torch.ones(4, 4, device="cuda")
    C = torch.zeros(4, 4, device="cuda")
    with pytest.raises(SgemmError, match="INVALID_ARG"):
        sgemm(A, A, out=C, alpha=float("nan"), beta=1.0)
    lib = load()
    assert lib.sgemm_run_ex(4, 4, 4, 1.0, A.data_ptr(), 4, A.data_ptr(), 4, float("nan"),
                            C.data_ptr(), 4, -1, 0, None) == -1
