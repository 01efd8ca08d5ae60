"""GPU parity of transposed operands, C = alpha * op(A).op(B) + beta * C
(sgemm_run_op, and ``sgemm`` on ``X.t()`` views), with the fp64 oracle's
oracle_gemm_f64_op.

Tolerance: 1e-6 * (|alpha| * K * max|A| * max|B| + |beta| * max|C0|), as for the
scaled form.  Small-integer products must match bit for bit."""
import numpy as np
import pytest

from dense_fp32_gemm_09_gb300 import SgemmError, load, sgemm, sgemm_run_op
from dense_fp32_gemm_09_gb300.workloads import make_inputs, random_pair, small_int_pair

pytestmark = pytest.mark.gpu

COMBOS = [(0, 0), (0, 1), (1, 0), (1, 1)]


def tol(alpha, beta, A, B, C0):
    K = A.shape[1]
    return 1e-6 * (abs(alpha) * K * float(A.abs().max()) * float(B.abs().max())
                   + abs(beta) * float(C0.abs().max()))


def stored_device(torch, X, trans, pad, offset):
    """The logical operand X stored as X or X^T in a NaN-filled device buffer with
    leading dimension width + pad, `offset` floats in (1 breaks 16-byte alignment)."""
    S = X.t().contiguous() if trans else X
    rows, cols = S.shape
    ld = cols + pad
    flat = torch.full((offset + rows * ld + 8,), float("nan"), device="cuda")
    view = flat[offset:offset + rows * ld].view(rows, ld)[:, :cols]
    view.copy_(S)
    return view, ld


@pytest.mark.parametrize("ta,tb", COMBOS)
@pytest.mark.parametrize("M,N,K", [(257, 131, 199), (1000, 333, 64), (33, 1, 7), (1, 50, 20),
                                   (640, 512, 1024)])
def test_op_ragged_against_oracle(cuda, oracle_mod, ta, tb, M, N, K):
    torch = cuda
    A, B = random_pair(M, N, K, seed=M + 3 * N + 7 * K)
    C0 = torch.randn(M, N, generator=torch.Generator().manual_seed(K))
    for (alpha, beta, pad, offset) in [(1.0, 0.0, 0, 0), (1.5, -0.75, 3, 1), (-2.0, 1.0, 4, 4)]:
        dA, lda = stored_device(torch, A, ta, pad, offset)
        dB, ldb = stored_device(torch, B, tb, pad + 1, offset)
        ldc = N + 5
        buf = torch.full((M + 2, ldc), 7.0, device="cuda")
        C = buf[1:M + 1, :N]
        C.copy_(C0)
        st = sgemm_run_op(ta, tb, M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(), ldb, beta,
                          C.data_ptr(), ldc)
        assert st == 0, load().sgemm_last_error().decode()
        torch.cuda.synchronize()
        mask = torch.ones_like(buf, dtype=torch.bool)
        mask[1:M + 1, :N] = False
        assert torch.all(buf[mask] == 7.0), "write outside C"
        ref = oracle_mod.gemm_f64_op(ta, tb, dA.cpu().numpy(), dB.cpu().numpy(), alpha, beta,
                                     C0.numpy())
        err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
        assert err <= tol(alpha, beta, A, B, C0), ((ta, tb), (M, N, K), alpha, beta, err)


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_op_small_integers_bit_exact(cuda, oracle_mod, ta, tb):
    torch = cuda
    M, N, K = 515, 389, 1201
    A, B = small_int_pair(M, N, K, seed=21)
    dA, lda = stored_device(torch, A, ta, 1, 1)
    dB, ldb = stored_device(torch, B, tb, 2, 0)
    C = torch.empty(M, N, device="cuda")
    assert sgemm_run_op(ta, tb, M, N, K, 1.0, dA.data_ptr(), lda, dB.data_ptr(), ldb, 0.0,
                        C.data_ptr(), N) == 0
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64_op(ta, tb, dA.cpu().numpy(), dB.cpu().numpy())
    assert np.array_equal(C.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("ta,tb", [(0, 1), (1, 0), (1, 1)])
def test_torch_transposed_views(cuda, oracle_mod, ta, tb):
    """sgemm() on X.t() views takes the transposed path with the views' own
    storage (no copies on the Python side)."""
    torch = cuda
    A, B = make_inputs("sgemm_1024")
    dA = A.t().contiguous().cuda().t() if ta else A.cuda()
    dB = B.t().contiguous().cuda().t() if tb else B.cuda()
    assert (dA.stride(0) == 1) == bool(ta) and (dB.stride(0) == 1) == bool(tb)
    C = sgemm(dA, dB)
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
    assert err <= tol(1.0, 0.0, A, B, torch.zeros(1))


def test_op_k_zero_and_empty(cuda):
    torch = cuda
    C = torch.full((7, 5), 3.0, device="cuda")
    A = torch.empty(1, device="cuda")
    # K == 0: beta * C (here 0.5 * 3)
    assert sgemm_run_op(1, 1, 7, 5, 0, 1.0, A.data_ptr(), 7, A.data_ptr(), 1, 0.5,
                        C.data_ptr(), 5) == 0
    torch.cuda.synchronize()
    assert torch.all(C == 1.5)
    assert sgemm_run_op(1, 0, 0, 5, 3, 1.0, 0, 1, A.data_ptr(), 5, 0.0, C.data_ptr(), 5) == 0


def test_op_rejects_bad_arguments(cuda):
    torch = cuda
    X = torch.zeros(64, 64, device="cuda")
    p = X.data_ptr()
    lib = load()
    assert sgemm_run_op(2, 0, 8, 8, 8, 1.0, p, 8, p, 8, 0.0, p + 4 * 64 * 32, 8) == -1
    # transa: A stored K x M needs lda >= M
    C = torch.zeros(16, 16, device="cuda")
    assert sgemm_run_op(1, 0, 16, 8, 8, 1.0, p, 8, p, 8, 0.0, C.data_ptr(), 16) == -1
    assert b"leading dimension" in lib.sgemm_last_error()
    # transb: B stored N x K needs ldb >= K
    assert sgemm_run_op(0, 1, 8, 8, 16, 1.0, p, 16, p, 8, 0.0, C.data_ptr(), 16) == -1
    with pytest.raises(SgemmError):
        sgemm(X.t(), X, out=X)   # C overlaps A
