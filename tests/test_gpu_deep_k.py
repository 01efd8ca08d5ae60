"""Very deep K on a small C: one or a few tiles whose K range is shared by every
CTA of the persistent grid (stream-K with up to 152 contributors per tile), each
CTA summing tens of thousands of k in registers before the fixed-order reduction.
Checked element by element against the fp64 oracle at the 1e-6*K*max|A|*max|B|
bound, on 16-byte-aligned operands and on operands that take the 4-byte kernels."""
import numpy as np
import pytest

from dense_fp32_gemm_09_gb300 import sgemm, sgemm_query_config
from dense_fp32_gemm_09_gb300.workloads import random_pair

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,min_split", [
    (64, 64, 2_000_000, 100),      # one 64 x 64 tile, every CTA shares its K range
    (128, 128, 1_000_000, 30),     # four tiles
    (1, 1, 1 << 24, 100),          # a dot product of 2^24 terms (ldb = 1: 4-byte loads)
    (3, 70, 1 << 20, 50),          # ldb = 70: 4-byte loads, ragged tile
])
def test_deep_k_matches_oracle(cuda, oracle_mod, M, N, K, min_split):
    torch = cuda
    cfg = sgemm_query_config(M, N, K)
    assert cfg["split_k"] >= min_split and cfg["sk_tiles"] == cfg["tiles"], cfg
    A, B = random_pair(M, N, K, seed=80)
    dA, dB = A.cuda(), B.cuda()
    C = torch.full((M, N), float("nan"), device="cuda")
    sgemm(dA, dB, out=C)
    torch.cuda.synchronize()
    exact = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    tol = 1e-6 * K * float(A.abs().max()) * float(B.abs().max())
    err = float(np.max(np.abs(C.cpu().numpy().astype(np.float64) - exact)))
    assert np.isfinite(err) and err <= tol, (err, tol)
    # Run to run: the partial sums are added in a fixed order.
    C2 = torch.full((M, N), float("nan"), device="cuda")
    sgemm(dA, dB, out=C2)
    torch.cuda.synchronize()
    assert torch.equal(C, C2)
