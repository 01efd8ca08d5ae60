"""The 3xTF32 tensor-core variant (tcgen05 / TMEM / TMA) against the fp64 oracle.

Tolerance: max|C - C_ref| <= 1e-5 * K * max|A| * max|B| (split-TF32 products
keep about 21 significant bits of each operand; FP32-class, not bit-comparable
with the CUDA-core path)."""
import numpy as np
import pytest

from dense_fp32_gemm_09_gb300 import check, load
from dense_fp32_gemm_09_gb300.workloads import make_inputs, random_pair, small_int_pair

pytestmark = pytest.mark.gpu


def tol(A, B):
    return 1e-5 * A.shape[1] * float(A.abs().max()) * float(B.abs().max())


def run(torch, A, B, C=None, alpha=1.0, beta=0.0, lda=None, ldb=None):
    lib = load()
    M, K = A.shape
    N = B.shape[1]
    if C is None:
        C = torch.empty(M, N, device="cuda")
    st = lib.sgemm_tf32x3_run_ex(M, N, K, alpha, A.data_ptr(), lda or A.stride(0),
                                 B.data_ptr(), ldb or B.stride(0), beta, C.data_ptr(),
                                 C.stride(0), None, 0, torch.cuda.current_stream().cuda_stream)
    check(st, "sgemm_tf32x3_run_ex")
    torch.cuda.synchronize()
    check(lib.sgemm_device_status(), "sgemm_device_status")
    return C


@pytest.fixture(params=["auto", "128/dp", "256/dp", "128/sk", "256/sk"])
def tile_width(request, monkeypatch):
    """Run with the library's choice of tile width and schedule, then forced to each
    width with data-parallel tiles only (dp) and with stream-K on every partial
    wave (sk)."""
    if request.param == "auto":
        monkeypatch.delenv("SGEMM_TF32X3_BN", raising=False)
        monkeypatch.delenv("SGEMM_TF32X3_SCHEDULE", raising=False)
    else:
        bn, sched = request.param.split("/")
        monkeypatch.setenv("SGEMM_TF32X3_BN", bn)
        monkeypatch.setenv("SGEMM_TF32X3_SCHEDULE", "1" if sched == "dp" else "2")
    return request.param


@pytest.mark.parametrize("M,N,K", [(128, 256, 32), (1, 1, 1), (5, 7, 3), (128, 256, 64),
                                   (129, 257, 33), (300, 500, 1000), (1000, 333, 77),
                                   (2048, 64, 4096)])
def test_shapes(cuda, oracle_mod, tile_width, M, N, K):
    torch = cuda
    A, B = random_pair(M, N, K, seed=M + 3 * N + 7 * K)
    C = run(torch, A.cuda(), B.cuda())
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
    assert err <= tol(A, B), ((M, N, K), err, tol(A, B))


@pytest.mark.parametrize("name", ["sgemm_1024", "sgemm_2048", "sgemm_ragged_3001x2047x1999"])
def test_workloads(cuda, oracle_mod, tile_width, name):
    torch = cuda
    A, B = make_inputs(name)
    C = run(torch, A.cuda(), B.cuda())
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
    assert err <= tol(A, B), (name, err)


def test_workload_4096_sampled_rows(cuda, oracle_mod):
    torch = cuda
    A, B = make_inputs("sgemm_4096")
    C = run(torch, A.cuda(), B.cuda())
    rows = np.unique(np.r_[0, 4095, np.random.default_rng(1).integers(0, 4096, 40)]).astype(np.int32)
    ref = oracle_mod.gemm_f64_rows(A.numpy(), B.numpy(), rows)
    got = C.cpu().numpy()[rows].astype(np.float64)
    assert np.max(np.abs(got - ref)) <= tol(A, B)


def test_small_integers_exact(cuda, oracle_mod):
    # |a|, |b| <= 8 are exact in TF32 (lo = 0), products and sums stay exact.
    torch = cuda
    A, B = small_int_pair(257, 300, 1000, seed=5)
    C = run(torch, A.cuda(), B.cuda())
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy()).astype(np.float32)
    assert np.array_equal(C.cpu().numpy(), ref)


def test_split_matters(cuda, oracle_mod):
    """Values that are not TF32-representable: a single TF32 pass would miss the
    tolerance by far; the three-term split meets it."""
    torch = cuda
    g = torch.Generator().manual_seed(4)
    A = 1.0 + torch.rand(256, 512, generator=g) * 2 ** -12   # low mantissa bits only
    B = 1.0 + torch.rand(512, 384, generator=g) * 2 ** -12
    C = run(torch, A.cuda(), B.cuda())
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    assert np.max(np.abs(C.cpu().numpy() - ref)) <= 1e-6 * 512 * 4   # far below TF32 alone


def test_strided_and_scaled(cuda, oracle_mod, tile_width):
    torch = cuda
    A, B = random_pair(300, 200, 150, seed=9)
    dA = torch.full((300, 153), float("nan"), device="cuda")
    dA[:, :150] = A.cuda()
    dB = torch.full((150, 203), float("nan"), device="cuda")
    dB[:, :200] = B.cuda()
    C0 = torch.randn(300, 200)
    C = C0.cuda()
    run(torch, dA[:, :150], dB[:, :200], C=C, alpha=-1.5, beta=0.25, lda=153, ldb=203)
    ref = oracle_mod.gemm_f64_ex(-1.5, A.numpy(), B.numpy(), 0.25, C0.numpy())
    err = np.max(np.abs(C.cpu().numpy() - ref))
    assert err <= 1.5 * tol(A, B) + 1e-6 * 0.25 * float(C0.abs().max())


def test_caller_workspace_and_sizes(cuda):
    torch = cuda
    import ctypes
    lib = load()
    out = ctypes.c_size_t(0)
    assert lib.sgemm_tf32x3_workspace_size(100, 200, 300, ctypes.byref(out)) == 0
    need = out.value
    assert need >= 4 * 2 * (100 + 200) * 300
    A, B = random_pair(100, 200, 300, seed=1)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(100, 200, device="cuda")
    ws = torch.empty(need // 4 + 64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.sgemm_tf32x3_run_ex(100, 200, 300, 1.0, dA.data_ptr(), 300, dB.data_ptr(), 200,
                                   0.0, C.data_ptr(), 200, ws.data_ptr(), need, s) == 0
    assert lib.sgemm_tf32x3_run_ex(100, 200, 300, 1.0, dA.data_ptr(), 300, dB.data_ptr(), 200,
                                   0.0, C.data_ptr(), 200, ws.data_ptr(), need - 4, s) == -6
    torch.cuda.synchronize()
    assert lib.sgemm_device_status() == 0


@pytest.mark.parametrize("sched", ["0", "2"])
def test_stream_k_deterministic(cuda, monkeypatch, sched):
    """Split tiles are summed in a fixed order: two runs agree bit for bit."""
    torch = cuda
    monkeypatch.setenv("SGEMM_TF32X3_SCHEDULE", sched)
    A, B = random_pair(1000, 700, 2000, seed=9)
    dA, dB = A.cuda(), B.cuda()
    C1 = run(torch, dA, dB).clone()
    C2 = run(torch, dA, dB)
    assert torch.equal(C1, C2)


def test_stream_k_scaled_into_split_tiles(cuda, oracle_mod, monkeypatch):
    """alpha/beta on tiles finished by the split-tile reduction."""
    torch = cuda
    monkeypatch.setenv("SGEMM_TF32X3_SCHEDULE", "2")
    M, N, K = 384, 640, 1536
    A, B = random_pair(M, N, K, seed=10)
    C0 = torch.randn(M, N, generator=torch.Generator().manual_seed(3))
    C = run(torch, A.cuda(), B.cuda(), C=C0.cuda(), alpha=0.5, beta=-1.25)
    ref = oracle_mod.gemm_f64_ex(0.5, A.numpy(), B.numpy(), -1.25, C0.numpy())
    err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
    assert err <= 0.5 * tol(A, B) + 1e-5 * 1.25 * float(C0.abs().max())


@pytest.mark.parametrize("M,N,K,lda_pad", [(512, 512, 512, 0), (1000, 700, 1999, 1),
                                           (3001, 2047, 1999, 5), (129, 300, 33, 3),
                                           (2048, 64, 4096, 0), (1024, 1024, 1024, 4)])
def test_hi_read_in_place_is_bit_identical(cuda, tile_width, monkeypatch, M, N, K, lda_pad):
    """When TMA can read A (16-byte aligned rows), the one-call path feeds A itself as
    the hi operand instead of writing Ahi: the tensor core reads an fp32 operand as
    TF32 by dropping its 13 low mantissa bits, which is the split's hi.  The product
    must equal, bit for bit, the one with Ahi written (SGEMM_TF32X3_SPLIT_A=1),
    with padded leading dimensions, K not a multiple of 4 and alpha/beta."""
    torch = cuda
    A, B = random_pair(M, N, K, seed=M + N + K)
    lda = K + lda_pad
    lda += (-lda) % 4                      # 16-byte rows: the in-place path applies
    buf = torch.full((M, lda), float("nan"), device="cuda")
    buf[:, :K] = A.cuda()
    dA, dB = buf[:, :K], B.cuda()
    C0 = torch.randn(M, N, device="cuda")
    monkeypatch.delenv("SGEMM_TF32X3_SPLIT_A", raising=False)
    direct = run(torch, dA, dB, C0.clone(), alpha=0.75, beta=0.5, lda=lda)
    monkeypatch.setenv("SGEMM_TF32X3_SPLIT_A", "1")
    split = run(torch, dA, dB, C0.clone(), alpha=0.75, beta=0.5, lda=lda)
    assert torch.equal(direct, split)
