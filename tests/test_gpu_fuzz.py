"""Seeded random cases across the whole entry-point surface, each checked element
by element against the fp64 oracle (oracle_gemm_f64_op): random M, N, K, leading
dimension padding, 4-byte misalignment of the bases, alpha/beta (including 0 and
1) and transpose flags; C lives inside a canary-filled buffer.  The 3xTF32 path
gets its own random cases at its own tolerance, and random cluster splits theirs."""
import numpy as np
import pytest

from dense_fp32_gemm_09_gb300 import check, load, sgemm_run_op

pytestmark = pytest.mark.gpu

CANARY = -7.25


def case(rng):
    M, N, K = (int(x) for x in rng.integers(1, 700, size=3))
    if rng.random() < 0.1:
        K = int(rng.integers(1, 5))
    ta, tb = int(rng.integers(0, 2)), int(rng.integers(0, 2))
    alpha = float(rng.choice([1.0, 0.0, -1.5, 0.25]))
    beta = float(rng.choice([0.0, 1.0, -0.5, 2.0]))
    pads = [int(x) for x in rng.integers(0, 6, size=3)]
    offs = [int(x) for x in rng.integers(0, 2, size=3)]
    return M, N, K, ta, tb, alpha, beta, pads, offs


def place(torch, X, pad, off, fill):
    rows, cols = X.shape
    ld = cols + pad
    flat = torch.full((off + rows * ld + 4,), fill, dtype=torch.float32, device="cuda")
    view = flat[off:off + rows * ld].view(rows, ld)[:, :cols]
    view.copy_(X)
    return flat, view, ld


@pytest.mark.parametrize("seed", range(120))
def test_random_ffma_cases(cuda, oracle_mod, seed):
    torch = cuda
    rng = np.random.default_rng(1000 + seed)
    M, N, K, ta, tb, alpha, beta, pads, offs = case(rng)
    g = torch.Generator().manual_seed(seed)
    A = torch.rand(M, K, generator=g) * 2 - 1                  # logical operands
    B = torch.rand(K, N, generator=g) * 2 - 1
    C0 = torch.rand(M, N, generator=g) * 2 - 1
    _, dA, lda = place(torch, A.t().contiguous() if ta else A, pads[0], offs[0], float("nan"))
    _, dB, ldb = place(torch, B.t().contiguous() if tb else B, pads[1], offs[1], float("nan"))
    cbuf, dC, ldc = place(torch, C0, pads[2], offs[2], CANARY)
    st = sgemm_run_op(ta, tb, M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(), ldb, beta,
                      dC.data_ptr(), ldc)
    assert st == 0, (M, N, K, ta, tb, load().sgemm_last_error())
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64_op(ta, tb, dA.cpu().numpy(), dB.cpu().numpy(), alpha, beta,
                                 C0.numpy())
    err = np.max(np.abs(dC.cpu().numpy().astype(np.float64) - ref))
    tol = 1e-6 * (abs(alpha) * K + abs(beta)) + 1e-30
    assert err <= tol, ((M, N, K, ta, tb, alpha, beta, pads, offs), err, tol)
    # nothing outside C was written
    flat = cbuf.cpu().numpy()
    mask = np.ones(flat.size, dtype=bool)
    base = offs[2]
    for r in range(M):
        mask[base + r * ldc: base + r * ldc + N] = False
    assert np.all(flat[mask] == CANARY)


@pytest.mark.parametrize("seed", range(30))
def test_random_tf32x3_cases(cuda, oracle_mod, seed):
    torch = cuda
    lib = load()
    rng = np.random.default_rng(2000 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 900, size=3))
    alpha = float(rng.choice([1.0, -2.0, 0.5]))
    beta = float(rng.choice([0.0, 1.0, -0.75]))
    pads = [int(x) for x in rng.integers(0, 6, size=3)]
    offs = [int(x) for x in rng.integers(0, 2, size=3)]
    g = torch.Generator().manual_seed(100 + seed)
    A = torch.rand(M, K, generator=g) * 2 - 1
    B = torch.rand(K, N, generator=g) * 2 - 1
    C0 = torch.rand(M, N, generator=g) * 2 - 1
    _, dA, lda = place(torch, A, pads[0], offs[0], float("nan"))
    _, dB, ldb = place(torch, B, pads[1], offs[1], float("nan"))
    cbuf, dC, ldc = place(torch, C0, pads[2], offs[2], CANARY)
    check(lib.sgemm_tf32x3_run_ex(M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(), ldb, beta,
                                  dC.data_ptr(), ldc, None, 0,
                                  torch.cuda.current_stream().cuda_stream), "tf32x3")
    torch.cuda.synchronize()
    check(lib.sgemm_device_status(), "device status")
    ref = oracle_mod.gemm_f64_ex(alpha, A.numpy(), B.numpy(), beta, C0.numpy())
    err = np.max(np.abs(dC.cpu().numpy().astype(np.float64) - ref))
    tol = 1e-5 * (abs(alpha) * K + abs(beta)) + 1e-30
    assert err <= tol, ((M, N, K, alpha, beta, pads, offs), err, tol)
    flat = cbuf.cpu().numpy()
    mask = np.ones(flat.size, dtype=bool)
    for r in range(M):
        mask[offs[2] + r * ldc: offs[2] + r * ldc + N] = False
    assert np.all(flat[mask] == CANARY)


def wide_case(rng):
    """Large shapes drawn around the tile chooser's boundaries: narrow C with M >= 4096
    (512 x 64 tiles), 64 < N <= 128, K around 2048 (slice depth), the smallest problems
    (32 x 32 tiles), long K, short K, short and wide C (M <= 64), N from 129 to 256 with
    M >= 4096 (64-wide tiles), small C with deep K, and N <= 128 with short K.
    Operands 16-byte aligned."""
    kind = int(rng.integers(0, 10))
    lo_hi = [((4000, 4600), (1, 65), (1, 2500)), ((4000, 4600), (65, 129), (1, 1500)),
             ((1000, 2600), (1000, 2600), (900, 2100)), ((1, 400), (1, 400), (1, 1100)),
             ((500, 1400), (500, 1400), (1, 4000)), ((1, 2500), (1, 2500), (1, 64)),
             ((1, 100), (2000, 9000), (1, 3000)), ((4000, 8300), (129, 257), (1, 2500)),
             ((200, 900), (200, 900), (2000, 6000)), ((4000, 9000), (65, 129), (64, 1500))][kind]
    M, N, K = (int(rng.integers(a, b)) for a, b in lo_hi)
    return M, N, K


@pytest.mark.parametrize("seed", range(100))
def test_random_wide_cases(cuda, oracle_mod, monkeypatch, seed):
    """Wide random cases on 16-byte-aligned operands (the 16-byte entries), with random
    alpha/beta and stream-K gaps forced to 0..3 or left to the planner."""
    torch = cuda
    rng = np.random.default_rng(3000 + seed)
    M, N, K = wide_case(rng)
    alpha = float(rng.choice([1.0, -1.5, 0.25]))
    beta = float(rng.choice([0.0, 1.0, -0.5]))
    gap = str(rng.choice(["", "0", "1", "2", "3"]))
    if gap:
        monkeypatch.setenv("SGEMM_SK_GAP", gap)
    else:
        monkeypatch.delenv("SGEMM_SK_GAP", raising=False)
    pads = [(-d) % 4 + 4 * int(rng.integers(0, 2)) for d in (K, N, N)]
    g = torch.Generator().manual_seed(3000 + seed)
    A = torch.rand(M, K, generator=g) * 2 - 1
    B = torch.rand(K, N, generator=g) * 2 - 1
    C0 = torch.rand(M, N, generator=g) * 2 - 1
    _, dA, lda = place(torch, A, pads[0], 0, float("nan"))
    _, dB, ldb = place(torch, B, pads[1], 0, float("nan"))
    cbuf, dC, ldc = place(torch, C0, pads[2], 0, CANARY)
    st = sgemm_run_op(0, 0, M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(), ldb, beta,
                      dC.data_ptr(), ldc)
    assert st == 0, (M, N, K, load().sgemm_last_error())
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64_ex(alpha, A.numpy(), B.numpy(), beta, C0.numpy())
    err = np.max(np.abs(dC.cpu().numpy().astype(np.float64) - ref))
    tol = 1e-6 * (abs(alpha) * K + abs(beta)) + 1e-30
    assert err <= tol, ((M, N, K, alpha, beta, gap), err, tol)
    flat = cbuf.cpu().numpy()
    mask = np.ones(flat.size, dtype=bool)
    for r in range(M):
        mask[r * ldc: r * ldc + N] = False
    assert np.all(flat[mask] == CANARY)


@pytest.mark.parametrize("seed", range(30))
def test_random_misaligned_cases_around_the_copy_threshold(cuda, oracle_mod, seed):
    """Operands with 4-byte-misaligned bases or odd leading dimensions, with M, N and K
    drawn around the point from which sgemm copies them to aligned buffers (K >= 768
    and M*N*K >= 5e8): both the copied path and the 4-byte-load kernels, checked
    element by element against the oracle inside canaried C."""
    torch = cuda
    rng = np.random.default_rng(5000 + seed)
    M, N = (int(x) for x in rng.integers(500, 1300, size=2))
    K = int(rng.integers(500, 1400))
    alpha = float(rng.choice([1.0, -1.5]))
    beta = float(rng.choice([0.0, 1.0]))
    pads = [int(x) for x in rng.integers(0, 4, size=3)]
    offs = [int(x) for x in rng.integers(0, 2, size=3)]
    if not any(pads[:2]) and not any(offs[:2]):
        offs[0] = 1                      # at least one operand misaligned
    g = torch.Generator().manual_seed(5000 + seed)
    A = torch.rand(M, K, generator=g) * 2 - 1
    B = torch.rand(K, N, generator=g) * 2 - 1
    C0 = torch.rand(M, N, generator=g) * 2 - 1
    _, dA, lda = place(torch, A, pads[0], offs[0], float("nan"))
    _, dB, ldb = place(torch, B, pads[1], offs[1], float("nan"))
    cbuf, dC, ldc = place(torch, C0, pads[2], offs[2], CANARY)
    st = sgemm_run_op(0, 0, M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(), ldb, beta,
                      dC.data_ptr(), ldc)
    assert st == 0, (M, N, K, load().sgemm_last_error())
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64_ex(alpha, A.numpy(), B.numpy(), beta, C0.numpy())
    err = np.max(np.abs(dC.cpu().numpy().astype(np.float64) - ref))
    tol = 1e-6 * (abs(alpha) * K + abs(beta)) + 1e-30
    assert err <= tol, ((M, N, K, pads, offs), err, tol)
    flat = cbuf.cpu().numpy()[offs[2]:]
    mask = np.ones(flat.size, dtype=bool)
    for r in range(M):
        mask[r * ldc: r * ldc + N] = False
    assert np.all(flat[mask] == CANARY)


@pytest.mark.parametrize("seed", range(60))
def test_random_cluster_split_cases(cuda, oracle_mod, monkeypatch, seed):
    """Random shapes run as cluster splits (schedule 3, clusters of up to 2, 4 or 8
    CTAs per tile) with random alpha/beta, leading-dimension padding and 4-byte
    misaligned bases (the 4-byte-load entries take the cluster sum too), against the
    oracle, with canaries around C."""
    torch = cuda
    lib = load()
    rng = np.random.default_rng(4000 + seed)
    M, N = (int(x) for x in rng.integers(1, 1500, size=2))
    K = int(rng.integers(1, 3000))
    alpha = float(rng.choice([1.0, -1.5, 0.25]))
    beta = float(rng.choice([0.0, 1.0, -0.5]))
    monkeypatch.setenv("SGEMM_CLUSTER", str(int(rng.choice([2, 4, 8]))))
    pads = [int(x) for x in rng.integers(0, 6, size=3)]
    offs = [int(x) for x in rng.integers(0, 2, size=3)]
    g = torch.Generator().manual_seed(4000 + seed)
    A = torch.rand(M, K, generator=g) * 2 - 1
    B = torch.rand(K, N, generator=g) * 2 - 1
    C0 = torch.rand(M, N, generator=g) * 2 - 1
    _, dA, lda = place(torch, A, pads[0], offs[0], float("nan"))
    _, dB, ldb = place(torch, B, pads[1], offs[1], float("nan"))
    cbuf, dC, ldc = place(torch, C0, pads[2], offs[2], CANARY)
    st = lib.sgemm_run_ex(M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(), ldb, beta,
                          dC.data_ptr(), ldc, -1, 3, torch.cuda.current_stream().cuda_stream)
    assert st == 0, (M, N, K, lib.sgemm_last_error())
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64_ex(alpha, A.numpy(), B.numpy(), beta, C0.numpy())
    err = np.max(np.abs(dC.cpu().numpy().astype(np.float64) - ref))
    tol = 1e-6 * (abs(alpha) * K + abs(beta)) + 1e-30
    assert err <= tol, ((M, N, K, alpha, beta, pads, offs), err, tol)
    flat = cbuf.cpu().numpy()
    mask = np.ones(flat.size, dtype=bool)
    for r in range(M):
        mask[offs[2] + r * ldc: offs[2] + r * ldc + N] = False
    assert np.all(flat[mask] == CANARY)
