"""Parity of the CUDA path (called through the C ABI) with the fp64 CPU oracle.

Tolerance for FP32 results: max |C_gpu - C_ref| <= 1e-6 * K * max|A| * max|B|,
with the maxima over the drawn inputs.  Where the arithmetic is exact in any
summation order (small integers, identity and permutation matrices) the bar is
bit equality with the oracle rounded to fp32.
"""
import numpy as np
import pytest

from dense_fp32_gemm_09_gb300 import kernel_table, sgemm, sgemm_query_config
from dense_fp32_gemm_09_gb300.workloads import (WORKLOADS, make_inputs, random_pair,
                                                small_int_pair)

pytestmark = pytest.mark.gpu

SENTINEL = 1234.5


def tolerance(A, B):
    K = A.shape[1]
    return 1e-6 * K * float(A.abs().max()) * float(B.abs().max())


def canaried(torch, M, N, ldc_pad=5, rows_pad=2):
    """An (M, N) view with leading dimension N + ldc_pad inside a sentinel-filled
    buffer with rows_pad extra rows above and below."""
    buf = torch.full((M + 2 * rows_pad, N + ldc_pad), SENTINEL, dtype=torch.float32,
                     device="cuda")
    return buf, buf[rows_pad:rows_pad + M, :N]


def check_canary(buf, M, N, rows_pad=2):
    b = buf.cpu().numpy()
    mask = np.ones(b.shape, dtype=bool)
    mask[rows_pad:rows_pad + M, :N] = False
    assert np.all(b[mask] == SENTINEL), "a write landed outside the M x N region"


def padded(torch, X, pad, offset=0):
    """X copied into a device buffer with leading dimension cols + pad, starting
    `offset` elements into the buffer (offset 1 breaks 16-byte alignment)."""
    rows, cols = X.shape
    ld = cols + pad
    flat = torch.full((offset + rows * ld + 8,), float("nan"), dtype=torch.float32,
                      device="cuda")
    view = flat[offset:offset + rows * ld].view(rows, ld)[:, :cols]
    view.copy_(X)
    return view


# --------------------------------------------------------------------------
# the named workloads, in the configuration sgemm_run picks (the bench's)
# --------------------------------------------------------------------------


@pytest.mark.parametrize("name", ["sgemm_256", "sgemm_1024", "sgemm_2048",
                                  "sgemm_ragged_3001x2047x1999", "sgemm_4096"])
def test_workload_full_parity(cuda, oracle_mod, name):
    torch = cuda
    A, B = make_inputs(name)
    C = sgemm(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
    assert err <= tolerance(A, B), (name, err, tolerance(A, B))


@pytest.mark.parametrize("name", ["sgemm_8192", "sgemm_tall_16384x64x4096"])
def test_workload_sampled_rows(cuda, oracle_mod, name):
    """256 seeded rows plus the first and the last, and two rows in every band of
    BM rows (one CTA tile high), so that every tile, the split ones included, has
    rows in the sample; each sampled row is compared over all N columns."""
    torch = cuda
    w = WORKLOADS[name]
    A, B = make_inputs(name)
    C = sgemm(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    bm = sgemm_query_config(w.M, w.N, w.K)["bm"]
    bands = [min(r, w.M - 1) for b in range(0, w.M, bm)
             for r in (b + (b // bm * 37) % bm, b + bm - 1)]
    rng = np.random.default_rng(12345)
    rows = np.unique(np.concatenate([[0, w.M - 1], rng.integers(0, w.M, 256),
                                     bands])).astype(np.int32)
    ref = oracle_mod.gemm_f64_rows(A.numpy(), B.numpy(), rows)
    got = C[torch.from_numpy(rows.astype(np.int64)).cuda()].cpu().numpy().astype(np.float64)
    err = np.max(np.abs(got - ref))
    assert err <= tolerance(A, B), (name, err, tolerance(A, B))
    assert torch.isfinite(C).all()


def test_tall_skinny_full_parity(cuda, oracle_mod):
    A, B = make_inputs("sgemm_tall_16384x64x4096")
    C = sgemm(A.cuda(), B.cuda()).cpu().numpy().astype(np.float64)
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    assert np.max(np.abs(C - ref)) <= tolerance(A, B)


# --------------------------------------------------------------------------
# every tile-table entry, both schedules, ragged shapes, canaried output
# --------------------------------------------------------------------------

SHAPES = [(1, 1, 1), (3, 5, 7), (9, 4, 2), (31, 33, 17), (65, 63, 129), (127, 129, 65),
          (129, 127, 300), (257, 383, 1000), (300, 260, 33), (1000, 70, 517)]


def _ids():
    try:
        return [k["name"] for k in kernel_table()]
    except Exception:   # library not built: the test fixture reports it
        return []


@pytest.mark.parametrize("kname", _ids())
@pytest.mark.parametrize("schedule", [1, 2, 3])
def test_each_kernel_ragged_shapes(cuda, oracle_mod, kname, schedule):
    torch = cuda
    table = {k["name"]: k for k in kernel_table()}
    kid = table[kname]["kernel_id"]
    for (M, N, K) in SHAPES:
        A, B = random_pair(M, N, K, seed=M * 7 + N * 3 + K)
        # ld padded to a multiple of 4 so that 16-byte entries may run too
        dA = padded(torch, A, (-K) % 4 + 4)
        dB = padded(torch, B, (-N) % 4 + 4)
        buf, C = canaried(torch, M, N, ldc_pad=(-N) % 4 + 4)
        sgemm(dA, dB, out=C, kernel_id=kid, schedule=schedule)
        torch.cuda.synchronize()
        check_canary(buf, M, N)
        ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
        err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
        assert err <= tolerance(A, B), (kname, schedule, (M, N, K), err)


@pytest.mark.parametrize("kname", [k for k in _ids() if k.endswith("_v1")])
def test_unaligned_operands(cuda, oracle_mod, kname):
    torch = cuda
    kid = {k["name"]: k for k in kernel_table()}[kname]["kernel_id"]
    for (M, N, K) in [(33, 17, 65), (130, 131, 129), (301, 205, 199)]:
        A, B = random_pair(M, N, K, seed=K)
        dA = padded(torch, A, 1, offset=1)     # odd lda, 4-byte aligned base
        dB = padded(torch, B, 3, offset=3)
        buf, C = canaried(torch, M, N, ldc_pad=1)
        sgemm(dA, dB, out=C, kernel_id=kid, schedule=2)
        torch.cuda.synchronize()
        check_canary(buf, M, N)
        ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
        err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
        assert err <= tolerance(A, B)


def test_vec4_entry_refuses_unaligned(cuda):
    torch = cuda
    from dense_fp32_gemm_09_gb300 import SgemmError
    kid = [k for k in kernel_table() if k["vec"] == 4][0]["kernel_id"]
    A, B = random_pair(8, 8, 9, seed=0)
    with pytest.raises(SgemmError, match="UNSUPPORTED"):
        sgemm(A.cuda(), B.cuda(), kernel_id=kid)


# --------------------------------------------------------------------------
# exact cases: bit equality
# --------------------------------------------------------------------------


@pytest.mark.parametrize("M,N,K", [(3001, 2047, 1999), (512, 640, 4096), (77, 1031, 263)])
def test_small_integers_bit_exact(cuda, oracle_mod, M, N, K):
    A, B = small_int_pair(M, N, K, seed=M + N + K)
    C = sgemm(A.cuda(), B.cuda()).cpu().numpy()
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy()).astype(np.float32)
    assert np.array_equal(C, ref)


@pytest.mark.parametrize("n,cols", [(129, 77), (1000, 333)])
def test_identity_and_permutation_bit_exact(cuda, n, cols):
    torch = cuda
    g = torch.Generator().manual_seed(n)
    X = torch.randn(n, cols, generator=g)
    I = torch.eye(n)
    assert torch.equal(sgemm(I.cuda(), X.cuda()).cpu(), X)
    perm = torch.randperm(n, generator=g)
    P = torch.zeros(n, n)
    P[torch.arange(n), perm] = 1.0
    assert torch.equal(sgemm(P.cuda(), X.cuda()).cpu(), X[perm])
    Y = torch.randn(cols, n, generator=g)
    assert torch.equal(sgemm(Y.cuda(), P.cuda()).cpu(), Y[:, torch.argsort(perm)])


def test_ones_give_K(cuda):
    torch = cuda
    for M, N, K in [(1, 1, 1), (200, 300, 4097), (5, 64, 12345)]:
        C = sgemm(torch.ones(M, K, device="cuda"), torch.ones(K, N, device="cuda"))
        assert torch.all(C == K)


# --------------------------------------------------------------------------
# degenerate sizes, determinism, entry points
# --------------------------------------------------------------------------


def test_zero_K_writes_zeros_only_inside(cuda):
    torch = cuda
    buf, C = canaried(torch, 37, 45)
    A = torch.empty(37, 0, device="cuda")
    B = torch.empty(0, 45, device="cuda")
    sgemm(A, B, out=C)
    torch.cuda.synchronize()
    check_canary(buf, 37, 45)
    assert torch.all(C == 0)


def test_empty_M_or_N(cuda):
    torch = cuda
    assert sgemm(torch.ones(0, 5, device="cuda"), torch.ones(5, 7, device="cuda")).shape == (0, 7)
    assert sgemm(torch.ones(4, 5, device="cuda"), torch.ones(5, 0, device="cuda")).shape == (4, 0)


def test_run_to_run_deterministic(cuda):
    torch = cuda
    A, B = make_inputs("sgemm_4096")
    dA, dB = A.cuda(), B.cuda()
    C1 = sgemm(dA, dB).clone()
    C2 = sgemm(dA, dB)
    assert torch.equal(C1, C2)
    for kid in {k["kernel_id"] for k in kernel_table() if k["vec"] == 4}:
        a = sgemm(dA[:1000, :3000], dB[:3000, :700], kernel_id=kid, schedule=2).clone()
        b = sgemm(dA[:1000, :3000], dB[:3000, :700], kernel_id=kid, schedule=2)
        assert torch.equal(a, b)


def test_stream_k_matches_data_parallel_within_tolerance(cuda, oracle_mod):
    torch = cuda
    A, B = random_pair(700, 900, 2500, seed=9)
    dA, dB = A.cuda(), B.cuda()
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    for kid in {k["kernel_id"] for k in kernel_table() if k["vec"] == 4}:
        for schedule in (1, 2):
            C = sgemm(dA, dB, kernel_id=kid, schedule=schedule).cpu().numpy()
            assert np.max(np.abs(C - ref)) <= tolerance(A, B)


@pytest.mark.parametrize("gap", ["0", "1", "2", "3"])
def test_stream_k_gap_parity(cuda, oracle_mod, monkeypatch, gap):
    """Stream-K ranges with 0..3 placeholder slices between split tiles: every
    kernel, on shapes whose tiles are all split or whose last wave is, matches the
    oracle, writes nothing outside C, repeats bit for bit, and reports the gap."""
    torch = cuda
    monkeypatch.setenv("SGEMM_SK_GAP", gap)
    monkeypatch.setenv("SGEMM_CLUSTER", "0")   # the stream-K form of every split
    used = 0
    for (M, N, K) in [(1024, 1024, 1024), (700, 900, 2500), (1001, 517, 1999)]:
        A, B = random_pair(M, N, K, seed=M + N + K)
        ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
        dA = padded(torch, A, (-K) % 4 + 4)
        dB = padded(torch, B, (-N) % 4 + 4)
        for k in kernel_table():
            buf, C = canaried(torch, M, N, ldc_pad=(-N) % 4 + 4)
            sgemm(dA, dB, out=C, kernel_id=k["kernel_id"], schedule=2)
            first = C.clone()
            sgemm(dA, dB, out=C, kernel_id=k["kernel_id"], schedule=2)
            torch.cuda.synchronize()
            check_canary(buf, M, N)
            assert torch.equal(first, C), (k["name"], gap)
            err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
            assert err <= tolerance(A, B), (k["name"], gap, (M, N, K), err)
        cfg = sgemm_query_config(M, N, K, dA.stride(0), dB.stride(0), N, dA.data_ptr(),
                                 dB.data_ptr(), None)
        used += cfg["sk_gap"] == int(gap)
    assert used > 0


def test_chained_products_see_their_inputs_complete(cuda, oracle_mod):
    """Back-to-back products on one stream, each reading the one before (the main
    kernels start as programmatic dependents of the previous kernel, and wait for it
    before touching memory).  The chain runs a stream-K product whose reduction writes
    the next one's A, a product whose B is first packed (odd ld, large), and a scaled
    product that reads C.  Each stage matches the oracle applied to the final value of
    its inputs."""
    torch = cuda
    g = torch.Generator().manual_seed(21)

    def u(r, c, scale):
        return ((torch.rand(r, c, generator=g) - 0.5) * scale).cuda()

    X0, B1, B2 = u(1100, 1000, 1.0), u(1000, 1024, 0.1), u(1024, 1024, 0.1)
    B3 = u(1024, 2047, 0.1)            # ld 2047: packed before the product (M*N*K > 2^31)
    B4, C4 = u(2047, 512, 0.1), u(1100, 512, 1.0)
    C4_init = C4.clone()
    C1 = sgemm(X0, B1)
    C2 = sgemm(C1, B2)
    C3 = sgemm(C2, B3)
    sgemm(C3, B4, out=C4, alpha=0.5, beta=2.0)
    torch.cuda.synchronize()
    assert sgemm_query_config(1100, 2047, 1024, 1024, 2047, 2047, C2.data_ptr(),
                              B3.data_ptr(), C3.data_ptr())["packed"] == 2

    def check(A, B, C, alpha=1.0, beta=0.0, C0=None):
        a, b = A.cpu(), B.cpu()
        ref = alpha * oracle_mod.gemm_f64(a.numpy(), b.numpy())
        if C0 is not None:
            ref = ref + beta * C0.cpu().numpy().astype(np.float64)
        err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
        tol = abs(alpha) * tolerance(a, b) + (1e-6 * abs(beta) * float(C0.abs().max())
                                              if C0 is not None else 0.0)
        assert err <= tol, (tuple(A.shape), tuple(B.shape), err, tol)

    check(X0, B1, C1)
    check(C1, B2, C2)
    check(C2, B3, C3)
    check(C3, B4, C4, 0.5, 2.0, C4_init)


def test_caller_workspace_entry_point(cuda, oracle_mod):
    torch = cuda
    from dense_fp32_gemm_09_gb300 import check, sgemm_run_ws, sgemm_workspace_size
    A, B = make_inputs("sgemm_1024")
    M, K = A.shape
    N = B.shape[1]
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, device="cuda")
    need = sgemm_workspace_size(M, N, K, K, N, N, dA.data_ptr(), dB.data_ptr(), C.data_ptr())
    ws = torch.full((max(need, 16) // 4 + 64,), 7.0, device="cuda")   # dirty on purpose
    for _ in range(2):
        check(sgemm_run_ws(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, C.data_ptr(), N,
                           ws.data_ptr(), ws.numel() * 4), "sgemm_run_ws")
        torch.cuda.synchronize()
        ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
        assert np.max(np.abs(C.cpu().numpy() - ref)) <= tolerance(A, B)
    if need > 0:
        st = sgemm_run_ws(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, C.data_ptr(), N,
                          ws.data_ptr(), need - 4)
        assert st == -6


def test_library_workspace_reused_across_layouts(cuda, oracle_mod):
    """Consecutive split-tile calls with different tile sizes and grids share the
    library workspace on one stream; each must still be exact to tolerance."""
    torch = cuda
    table = {k["name"]: k["kernel_id"] for k in kernel_table()}
    cases = [("128x256x64_t8x16_s2_f2_v4", (1500, 1700, 3000)),
             ("128x64x16_t16x8_s4_f2_v4", (6000, 64, 2048)),
             ("64x64x16_t4x4_s3_f1_v4", (300, 260, 3000)),
             ("256x128x64_t8x16_s2_f2_v4", (700, 900, 5000))]
    for rep in range(2):
        for name, (M, N, K) in cases:
            A, B = random_pair(M, N, K, seed=M + rep)
            C = sgemm(A.cuda(), B.cuda(), kernel_id=table[name], schedule=2)
            ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
            err = np.max(np.abs(C.cpu().numpy() - ref))
            assert err <= tolerance(A, B), (name, (M, N, K), rep, err)


def test_host_buffer_entry_point(cuda, oracle_mod):
    torch = cuda
    from dense_fp32_gemm_09_gb300 import check, sgemm_run_host
    A, B = make_inputs("sgemm_ragged_3001x2047x1999")
    M, K = A.shape
    N = B.shape[1]
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.empty(M, N).pin_memory()
    dA = torch.empty(M, K, device="cuda")
    dB = torch.empty(K, N, device="cuda")
    dC = torch.empty(M, N, device="cuda")
    check(sgemm_run_host(M, N, K, hA.data_ptr(), K, hB.data_ptr(), N, hC.data_ptr(), N,
                         dA.data_ptr(), dB.data_ptr(), dC.data_ptr()), "sgemm_run_host")
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    assert np.max(np.abs(hC.numpy() - ref)) <= tolerance(A, B)


@pytest.mark.parametrize("panels", ["1", "3", "7"])
@pytest.mark.parametrize("M,N,K", [(1000, 333, 257), (130, 64, 40), (515, 96, 0)])
def test_host_entry_row_panels(cuda, oracle_mod, monkeypatch, panels, M, N, K):
    """The host-buffer entry in 1, 3 and 7 row panels (ragged last panel, padded
    leading dimensions, K == 0) on a side stream matches the oracle."""
    torch = cuda
    from dense_fp32_gemm_09_gb300 import check, sgemm_run_host
    monkeypatch.setenv("SGEMM_HOST_PANELS", panels)
    A, B = random_pair(M, N, K, seed=11)
    lda, ldb, ldc = K + 3, N + 1, N + 2
    hA = torch.zeros(M, lda).pin_memory()
    hB = torch.zeros(K, ldb).pin_memory()
    hA[:, :K] = A
    hB[:, :N] = B
    hC = torch.full((M, ldc), SENTINEL).pin_memory()
    dA = torch.empty(M * lda + 1, device="cuda")
    dB = torch.empty(K * ldb + 1, device="cuda")
    dC = torch.full((M * ldc + 1,), SENTINEL, device="cuda")
    side = torch.cuda.Stream()
    check(sgemm_run_host(M, N, K, hA.data_ptr(), lda, hB.data_ptr(), ldb, hC.data_ptr(), ldc,
                         dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), stream=side),
          "sgemm_run_host")
    side.synchronize()
    got = hC.numpy()
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy()) if K > 0 else np.zeros((M, N))
    assert np.max(np.abs(got[:, :N] - ref)) <= (tolerance(A, B) if K > 0 else 0.0)
    assert np.all(got[:, N:] == SENTINEL)


@pytest.mark.parametrize("panels", ["4", "1"])
def test_host_entry_is_ordered_on_the_callers_stream(cuda, oracle_mod, monkeypatch, panels):
    """Work queued on the stream before the call finishes before the call's
    copies and products start, and work queued after it sees the finished C: with
    4 panels on the library's own streams, and with 1 on the caller's stream."""
    torch = cuda
    from dense_fp32_gemm_09_gb300 import check, sgemm_run_host
    monkeypatch.setenv("SGEMM_HOST_PANELS", panels)
    M, N, K = 1024, 512, 384
    A, B = random_pair(M, N, K, seed=12)
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.empty(M, N).pin_memory()
    dA = torch.empty(M, K, device="cuda")
    dB = torch.empty(K, N, device="cuda")
    dC = torch.empty(M, N, device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(50_000_000)        # tens of milliseconds of GPU time
        dC.fill_(float("nan"))               # must land before the product
        check(sgemm_run_host(M, N, K, hA.data_ptr(), K, hB.data_ptr(), N, hC.data_ptr(), N,
                             dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), stream=side),
              "sgemm_run_host")
        after = dC.clone()                   # must see the finished product
    side.synchronize()
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    tol = tolerance(A, B)
    assert np.max(np.abs(hC.numpy() - ref)) <= tol
    assert np.max(np.abs(after.cpu().numpy() - ref)) <= tol
    assert torch.equal(after, dC)


def test_query_config_matches_bench_choice(cuda):
    cfg = sgemm_query_config(4096, 4096, 4096)
    assert cfg["grid"] > 0 and cfg["tiles"] == (4096 // cfg["bm"]) * (4096 // cfg["bn"])
    assert cfg["ctas_per_sm"] >= 1
    rag = sgemm_query_config(3001, 2047, 1999)
    assert rag["packed"] == 3 and rag["vec"] == 4   # odd ld: copied to aligned buffers
    small = sgemm_query_config(301, 205, 199)
    assert small["packed"] == 0 and small["vec"] == 1   # too small to be worth copying


@pytest.mark.parametrize("M,N,K,name", [
    (16384, 64, 4096, "512x64x32_t8x16_s2_f2_v4"),
    (4096, 36, 1000, "512x64x32_t8x16_s2_f2_v4"),
    (2048, 64, 4096, "64x64x16_t8x8_s3_f2_v4"),
    (8192, 128, 4096, "256x128x64_t8x16_s2_f2_v4"),
    (8192, 96, 4096, "256x128x64_t8x16_s2_f2_v4"),
    (4096, 4096, 4096, "128x256x64_t8x16_s2_f2_v4"),
    (2048, 2048, 2048, "256x128x64_t8x16_s2_f2_v4"),
    (1024, 1024, 1024, "128x256x32_t8x16_s4_f2_v4"),
    (1536, 1536, 1536, "128x256x32_t8x16_s4_f2_v4"),
    (256, 256, 256, "32x32x16_t4x4_s3_f2_v4"),
    (384, 384, 384, "32x32x16_t4x4_s3_f2_v4"),
    (512, 512, 512, "64x64x16_t8x8_s3_f2_v4"),
    (2048, 4096, 1024, "256x128x64_t8x16_s2_f2_v4"),
    (3008, 2048, 2000, "256x128x64_t8x16_s2_f2_v4_burst"),
    (4096, 4096, 1024, "128x256x64_t8x16_s2_f2_v4"),
    (768, 768, 4096, "128x256x32_t8x16_s4_f2_v4"),
    (384, 384, 4096, "128x128x32_t8x8_s3_f2_v4"),
])
def test_narrow_c_tile_choice(cuda, M, N, K, name):
    """Narrow C gets tiles no wider than it: 512 x 64 for N <= 64 once M fills eight
    of them, 256 x 128 for N <= 128.  Square-ish C takes 64-deep slices when K >= 2048
    or every CTA gets about 20 of them (128 x 256 tiles with double-buffered fragments
    once every CTA gets about 44), 32-deep ones on 128 x 256 tiles below; the
    smallest problems take 32 x 32 tiles."""
    assert sgemm_query_config(M, N, K)["name"] == name


def test_narrow_c_parity(cuda, oracle_mod):
    """The narrow-C choices above, full products against the oracle."""
    torch = cuda
    for (M, N, K) in [(4100, 61, 777), (4096, 128, 512), (5000, 100, 300)]:
        A, B = random_pair(M, N, K, seed=M + N)
        C = sgemm(A.cuda(), B.cuda())
        ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
        err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
        assert err <= tolerance(A, B), ((M, N, K), err)


def test_launch_counter_counts(cuda):
    torch = cuda
    from dense_fp32_gemm_09_gb300 import launch_count
    A = torch.ones(64, 64, device="cuda")
    n0 = launch_count()
    sgemm(A, A)
    assert launch_count() == n0 + 1


def test_large_unaligned_operands_are_packed(cuda, oracle_mod):
    """M*N*K >= 2^31 with rows off 16-byte alignment: sgemm_run copies the operands
    to aligned buffers first (reported by sgemm_query_config) and the result
    still matches the oracle, with nothing written outside C."""
    torch = cuda
    M, N, K = 1100, 1500, 1401
    A, B = random_pair(M, N, K, seed=77)
    dA = padded(torch, A, 2, offset=1)      # lda = 1403, base 4-byte aligned only
    dB = padded(torch, B, 1, offset=2)      # ldb = 1501
    cfg = sgemm_query_config(M, N, K, 1403, 1501, N + 3, dA.data_ptr(), dB.data_ptr(), None)
    assert cfg["packed"] == 3 and cfg["vec"] == 4
    buf, C = canaried(torch, M, N, ldc_pad=3)
    sgemm(dA, dB, out=C)
    torch.cuda.synchronize()
    check_canary(buf, M, N)
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    assert np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref)) <= tolerance(A, B)


@pytest.mark.parametrize("M,N,K,a_off,name,packed", [
    (64, 8192, 1024, 0, "64x64x16_t8x8_s3_f2_v4", 0),        # short, wide C
    (32, 4000, 1000, 0, "32x32x16_t4x4_s3_f2_v4", 0),
    (8192, 192, 1000, 0, "512x64x32_t8x16_s2_f2_v4", 0),     # 64-wide tiles fit N
    (4096, 128, 1024, 0, "256x128x32_t8x16_s4_f2_v4", 0),    # slices on offer
    (4096, 128, 512, 0, "128x128x32_t8x8_s3_f2_v4", 0),
    (448, 448, 4096, 0, "128x256x32_t8x16_s4_f2_v4", 0),     # small C, deep K
    (384, 384, 2048, 0, "128x128x32_t8x8_s3_f2_v4", 0),
    (2048, 128, 2048, 0, "256x128x32_t8x16_s4_f2_v4", 0),
    (1000, 1000, 300, 1, "128x128x16_t16x8_s4_f2_v1", 0),    # 4-byte loads, mid band
    (1000, 1000, 1000, 1, "128x256x32_t8x16_s4_f2_v4", 1),   # misaligned A copied
])
def test_rule_choices_through_the_automatic_path(cuda, oracle_mod, M, N, K, a_off, name,
                                                  packed):
    """Each tile-choice rule, taken by sgemm_run itself (no forced entry), against
    the oracle; a_off = 1 shifts A by 4 bytes so its rows are not 16-byte aligned."""
    torch = cuda
    A, B = random_pair(M, N, K, seed=M + N + K)
    buf = torch.empty(M * K + a_off, device="cuda")
    dA = buf[a_off:].view(M, K)
    dA.copy_(A)
    dB = B.cuda()
    cfg = sgemm_query_config(M, N, K, K, N, N, dA.data_ptr(), dB.data_ptr(), None)
    assert (cfg["name"], cfg["packed"]) == (name, packed)
    C = torch.full((M, N), float("nan"), device="cuda")
    sgemm(dA, dB, out=C)
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    err = float(np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref)))
    assert np.isfinite(err) and err <= tolerance(A, B), err
