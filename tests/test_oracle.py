"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test compares the oracle with something the source pages or plain
mathematics fix: the printed output of the pages' worked example, exact
rational arithmetic, exact integer products, identity / permutation
invariants, constant matrices, and an independent library routine.
"""
import math
import random
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden

# --------------------------------------------------------------------------
# helpers (test-side, independent of the oracle)
# --------------------------------------------------------------------------


def round_fraction_to_f32(x: Fraction) -> float:
    """Correctly rounded (nearest, ties to even) fp32 value of an exact rational."""
    if x == 0:
        return 0.0
    sign = -1.0 if x < 0 else 1.0
    ax = abs(x)
    e = ax.numerator.bit_length() - ax.denominator.bit_length()
    while Fraction(2) ** e > ax:
        e -= 1
    while Fraction(2) ** (e + 1) <= ax:
        e += 1
    q = Fraction(2) ** max(e - 23, -149)       # spacing of fp32 values near x
    n = ax / q
    lo = n.numerator // n.denominator
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    v = float(lo * q)
    return sign * float(np.float32(v))


def exact_product(A: np.ndarray, B: np.ndarray):
    M, K = A.shape
    N = B.shape[1]
    Af = [[Fraction(float(A[i, k])) for k in range(K)] for i in range(M)]
    Bf = [[Fraction(float(B[k, j])) for j in range(N)] for k in range(K)]
    C = [[sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0)) for j in range(N)]
         for i in range(M)]
    S = [[sum((abs(Af[i][k] * Bf[k][j]) for k in range(K)), Fraction(0)) for j in range(N)]
         for i in range(M)]
    return C, S


def p1_inputs(K=1024):
    # A[i] = (i % 7) * 0.1f, B[i] = (i % 5) * 0.2f, both with fp32 products.
    A = (np.arange(4 * K) % 7).astype(np.float32) * np.float32(0.1)
    B = (np.arange(4 * K) % 5).astype(np.float32) * np.float32(0.2)
    return A.reshape(4, K), B.reshape(K, 4)


# --------------------------------------------------------------------------
# the pages' worked example
# --------------------------------------------------------------------------


def test_p1_printed_output_fp32_fma(oracle_mod):
    rows = {r[0]: r[1:] for r in read_golden("p1_micro_gemm_4x4.txt")}
    K = int(rows["K"][0])
    A, B = p1_inputs(K)
    C = oracle_mod.gemm_f32_fma_seq(A, B)
    printed = ["%f" % float(v) for v in C[0]]
    assert printed == rows["C_row0_printed"]


def test_p1_fp32_close_to_f64(oracle_mod):
    A, B = p1_inputs()
    c32 = oracle_mod.gemm_f32_fma_seq(A, B).astype(np.float64)
    c64 = oracle_mod.gemm_f64(A, B)
    # The fp32 sequential result differs from the fp64 sum by accumulation error
    # only; the page's print agrees with the fp64 oracle to about 3e-4.
    assert np.max(np.abs(c32 - c64)) < 1e-3


def test_p1_closed_form_decimal(oracle_mod):
    """Rational arithmetic on the decimal definition 0.1*(i%7), 0.2*(i%5): the fp64
    oracle on the fp32-rounded inputs must agree to within the input rounding."""
    K = 1024
    A, B = p1_inputs(K)
    C = oracle_mod.gemm_f64(A, B)
    for i in range(4):
        for j in range(4):
            exact = sum(Fraction((i * K + k) % 7, 10) * Fraction(2 * ((k * 4 + j) % 5), 10)
                        for k in range(K))
            assert abs(C[i, j] - float(exact)) < 1e-5, (i, j, C[i, j], float(exact))
    # Row 0 of the closed form, to two decimals (the page prints these to 6).
    assert [round(float(sum(Fraction(k % 7, 10) * Fraction(2 * ((k * 4 + j) % 5), 10)
                            for k in range(K))), 2) for j in range(4)] == \
        [122.72, 122.46, 122.70, 122.74]


def test_p3_printed_diffs_are_ulp_multiples():
    """The two printed max|diff| values of the tiled test are whole multiples of the
    fp32 spacing of numbers near K/4 (what uniform[0,1) inputs give), which is the
    reading used for the inputs of the 1024^3 and 2048^3 workloads."""
    for M, N, K, diff, _ms, _gf in read_golden("p3_tiled_test_runs.txt"):
        K = int(K)
        spacing = 2.0 ** (math.floor(math.log2(K / 4)) - 23)
        ratio = float(diff) / spacing
        assert abs(ratio - round(ratio)) < 1e-3 and round(ratio) >= 1


def test_p3_printed_rates_are_2mnk_over_time():
    for M, N, K, _d, ms, gf in read_golden("p3_tiled_test_runs.txt"):
        rate = 2.0 * int(M) * int(N) * int(K) / (float(ms) * 1e-3) / 1e9
        assert abs(rate - float(gf)) / float(gf) < 2e-3


# --------------------------------------------------------------------------
# brute force on tiny inputs
# --------------------------------------------------------------------------


@pytest.mark.parametrize("seed", range(6))
def test_f64_against_exact_rationals(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    M, N, K = (int(x) for x in rng.integers(1, 9, size=3))
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = (rng.random((K, N)) * 4 - 2).astype(np.float32)
    C = oracle_mod.gemm_f64(A, B)
    exact, absum = exact_product(A, B)
    u = 2.0 ** -53
    for i in range(M):
        for j in range(N):
            bound = 1.01 * K * u * float(absum[i][j]) + 1e-300
            assert abs(C[i, j] - float(exact[i][j])) <= bound


@pytest.mark.parametrize("seed", range(6))
def test_f32_fma_seq_against_exact_rounding(oracle_mod, seed):
    rng = np.random.default_rng(100 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 7, size=3))
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    C = oracle_mod.gemm_f32_fma_seq(A, B)
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                acc = round_fraction_to_f32(Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                                            + Fraction(acc))
            assert C[i, j] == np.float32(acc), (i, j)


# --------------------------------------------------------------------------
# invariants with exact answers
# --------------------------------------------------------------------------


def strided(rows, cols, pad, fill=np.nan, seed=0, values=None):
    """A rows x cols float32 view inside a wider buffer whose padding is NaN."""
    buf = np.full((rows, cols + pad), fill, dtype=np.float32)
    if values is None:
        values = np.random.default_rng(seed).standard_normal((rows, cols)).astype(np.float32)
    buf[:, :cols] = values
    return buf[:, :cols]


@pytest.mark.parametrize("M,K,pad", [(1, 1, 0), (7, 5, 3), (33, 17, 1), (64, 64, 0)])
def test_identity_right_and_left(oracle_mod, M, K, pad):
    A = strided(M, K, pad, seed=M)
    I_K = strided(K, K, pad, values=np.eye(K, dtype=np.float32))
    assert np.array_equal(oracle_mod.gemm_f64(A, I_K), A.astype(np.float64))
    I_M = strided(M, M, pad, values=np.eye(M, dtype=np.float32))
    assert np.array_equal(oracle_mod.gemm_f64(I_M, A), A.astype(np.float64))


@pytest.mark.parametrize("n,cols", [(5, 3), (31, 9), (40, 40)])
def test_permutations_are_exact(oracle_mod, n, cols):
    rng = np.random.default_rng(n)
    perm = rng.permutation(n)
    P = np.zeros((n, n), dtype=np.float32)
    P[np.arange(n), perm] = 1.0            # (P X)[i] = X[perm[i]]
    X = rng.standard_normal((n, cols)).astype(np.float32)
    assert np.array_equal(oracle_mod.gemm_f64(P, X), X[perm].astype(np.float64))
    Y = rng.standard_normal((cols, n)).astype(np.float32)
    # (Y P)[:, j] = Y[:, i] where perm[i] = j
    inv = np.argsort(perm)
    assert np.array_equal(oracle_mod.gemm_f64(Y, P), Y[:, inv].astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(3, 4, 5), (37, 29, 300), (5, 70, 2000)])
def test_small_integers_match_integer_matmul(oracle_mod, M, N, K):
    rng = np.random.default_rng(M * N * K)
    A = rng.integers(-8, 9, (M, K)).astype(np.float32)
    B = rng.integers(-8, 9, (K, N)).astype(np.float32)
    want = A.astype(np.int64) @ B.astype(np.int64)
    assert np.array_equal(oracle_mod.gemm_f64(A, B), want.astype(np.float64))
    assert np.array_equal(oracle_mod.gemm_f32_fma_seq(A, B), want.astype(np.float32))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (9, 13, 1000), (4, 3, 4096)])
def test_ones_give_K(oracle_mod, M, N, K):
    A = np.ones((M, K), dtype=np.float32)
    B = np.ones((K, N), dtype=np.float32)
    assert np.all(oracle_mod.gemm_f64(A, B) == K)


def test_zero_K_is_zero(oracle_mod):
    A = np.zeros((3, 0), dtype=np.float32)
    B = np.zeros((0, 5), dtype=np.float32)
    C = oracle_mod.gemm_f64(A, B)
    assert C.shape == (3, 5) and np.all(C == 0)


def test_against_torch_float64_matmul(oracle_mod):
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(7)
    A = torch.randn(70, 130, generator=g, dtype=torch.float32)
    B = torch.randn(130, 45, generator=g, dtype=torch.float32)
    want = (A.double() @ B.double()).numpy()
    got = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    scale = (A.double().abs() @ B.double().abs()).numpy()
    assert np.all(np.abs(got - want) <= 1e-13 * scale)


def test_rows_and_elements_agree_with_full(oracle_mod):
    rng = np.random.default_rng(3)
    A = strided(50, 37, 5, seed=1)
    B = strided(37, 23, 2, seed=2)
    full = oracle_mod.gemm_f64(A, B)
    rows = np.array([0, 49, 17, 17, 3], dtype=np.int32)
    assert np.array_equal(oracle_mod.gemm_f64_rows(A, B, rows), full[rows])
    ii = rng.integers(0, 50, 40).astype(np.int32)
    jj = rng.integers(0, 23, 40).astype(np.int32)
    assert np.array_equal(oracle_mod.gemm_f64_elems(A, B, ii, jj), full[ii, jj])


def test_invalid_arguments_rejected(oracle_mod):
    import ctypes
    buf = (ctypes.c_float * 16)()
    out = (ctypes.c_double * 16)()
    fp = ctypes.cast(buf, ctypes.POINTER(ctypes.c_float))
    dp = ctypes.cast(out, ctypes.POINTER(ctypes.c_double))
    assert oracle_mod.raw_call_f64(-1, 2, 2, fp, 2, fp, 2, dp, 2) == -1
    assert oracle_mod.raw_call_f64(2, 2, 3, fp, 2, fp, 2, dp, 2) == -1   # lda < K
    assert oracle_mod.raw_call_f64(2, 2, 2, None, 2, fp, 2, dp, 2) == -1
    assert oracle_mod.raw_call_f64(2, 2, 2, fp, 2, fp, 2, dp, 2) == 0


def test_thread_count_does_not_change_results(oracle_mod):
    rng = np.random.default_rng(11)
    A = rng.standard_normal((61, 300)).astype(np.float32)
    B = rng.standard_normal((300, 47)).astype(np.float32)
    assert np.array_equal(oracle_mod.gemm_f64(A, B, nthreads=1),
                          oracle_mod.gemm_f64(A, B, nthreads=5))


def test_random_shapes_against_numpy_float64(oracle_mod):
    rnd = random.Random(5)
    for _ in range(10):
        M, N, K = rnd.randint(1, 40), rnd.randint(1, 40), rnd.randint(1, 200)
        rng = np.random.default_rng(rnd.randint(0, 1 << 30))
        A = rng.standard_normal((M, K)).astype(np.float32)
        B = rng.standard_normal((K, N)).astype(np.float32)
        want = A.astype(np.float64) @ B.astype(np.float64)
        scale = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
        assert np.all(np.abs(oracle_mod.gemm_f64(A, B) - want) <= 1e-13 * scale + 1e-300)


# --------------------------------------------------------------------------
# scaled form: alpha * A.B + beta * C0
# --------------------------------------------------------------------------


def test_ex_small_integers_exact(oracle_mod):
    rng = np.random.default_rng(21)
    A = rng.integers(-8, 9, (23, 301)).astype(np.float32)
    B = rng.integers(-8, 9, (301, 17)).astype(np.float32)
    C0 = rng.integers(-100, 101, (23, 17)).astype(np.float32)
    want = 2 * (A.astype(np.int64) @ B.astype(np.int64)) - 3 * C0.astype(np.int64)
    assert np.array_equal(oracle_mod.gemm_f64_ex(2.0, A, B, -3.0, C0), want.astype(np.float64))
    rows = np.array([22, 0, 5], dtype=np.int32)
    assert np.array_equal(oracle_mod.gemm_f64_ex(2.0, A, B, -3.0, C0, rows=rows),
                          want[rows].astype(np.float64))


def test_ex_beta_zero_does_not_read_C(oracle_mod):
    rng = np.random.default_rng(22)
    A = rng.integers(-4, 5, (9, 40)).astype(np.float32)
    B = rng.integers(-4, 5, (40, 11)).astype(np.float32)
    C0 = np.full((9, 11), np.nan, dtype=np.float32)
    want = 0.5 * (A.astype(np.int64) @ B.astype(np.int64))
    assert np.array_equal(oracle_mod.gemm_f64_ex(0.5, A, B, 0.0, C0), want)


def test_ex_alpha_zero_does_not_read_A_or_B(oracle_mod):
    A = np.full((6, 5), np.nan, dtype=np.float32)
    B = np.full((5, 7), np.inf, dtype=np.float32)
    C0 = np.arange(42, dtype=np.float32).reshape(6, 7)
    assert np.array_equal(oracle_mod.gemm_f64_ex(0.0, A, B, 0.25, C0), 0.25 * C0.astype(np.float64))


@pytest.mark.parametrize("seed", range(4))
def test_ex_against_exact_rationals(oracle_mod, seed):
    rng = np.random.default_rng(300 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 7, size=3))
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    alpha, beta = float(np.float32(0.1)), float(np.float32(-0.3))
    got = oracle_mod.gemm_f64_ex(alpha, A, B, beta, C0)
    exact, absum = exact_product(A, B)
    u = 2.0 ** -53
    for i in range(M):
        for j in range(N):
            want = Fraction(alpha) * exact[i][j] + Fraction(beta) * Fraction(float(C0[i, j]))
            bound = (K + 3) * u * (abs(alpha) * float(absum[i][j]) + abs(beta * float(C0[i, j])))
            assert abs(got[i, j] - float(want)) <= 1.01 * bound + 1e-300


# --------------------------------------------------------------------------
# transposed operands: op(A) . op(B)
# --------------------------------------------------------------------------


def stored(X, trans, pad=0):
    """X (the logical operand) as the oracle receives it: X itself or its
    transpose, optionally inside a NaN-padded row-major buffer (ld = width + pad)."""
    S = np.ascontiguousarray(X.T if trans else X)
    if pad == 0:
        return S
    buf = np.full((S.shape[0], S.shape[1] + pad), np.nan, dtype=np.float32)
    buf[:, :S.shape[1]] = S
    return buf[:, :S.shape[1]]


@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("seed", range(3))
def test_op_against_exact_rationals(oracle_mod, ta, tb, seed):
    """The logical product is formed by hand in exact arithmetic from the
    logical operands; the oracle gets them stored transposed where asked."""
    rng = np.random.default_rng(400 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 8, size=3))
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    alpha, beta = float(np.float32(1.5)), float(np.float32(0.25))
    got = oracle_mod.gemm_f64_op(ta, tb, stored(A, ta, 3), stored(B, tb, 2), alpha, beta, C0)
    exact, absum = exact_product(A, B)
    u = 2.0 ** -53
    for i in range(M):
        for j in range(N):
            want = Fraction(alpha) * exact[i][j] + Fraction(beta) * Fraction(float(C0[i, j]))
            bound = (K + 3) * u * (abs(alpha) * float(absum[i][j]) + abs(beta * float(C0[i, j])))
            assert abs(got[i, j] - float(want)) <= 1.01 * bound + 1e-300


@pytest.mark.parametrize("ta,tb", [(0, 1), (1, 0), (1, 1)])
def test_op_small_integers_exact(oracle_mod, ta, tb):
    rng = np.random.default_rng(7)
    M, N, K = 37, 29, 53
    A = rng.integers(-8, 9, (M, K)).astype(np.float32)
    B = rng.integers(-8, 9, (K, N)).astype(np.float32)
    want = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64)
    got = oracle_mod.gemm_f64_op(ta, tb, stored(A, ta, 5), stored(B, tb, 1))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("ta,tb", [(0, 1), (1, 0), (1, 1)])
def test_op_identity_and_permutation(oracle_mod, ta, tb):
    rng = np.random.default_rng(8)
    n = 23
    X = rng.standard_normal((n, n)).astype(np.float32)
    perm = rng.permutation(n)
    P = np.zeros((n, n), dtype=np.float32)
    P[np.arange(n), perm] = 1
    I = np.eye(n, dtype=np.float32)
    assert np.array_equal(oracle_mod.gemm_f64_op(ta, tb, stored(X, ta), stored(I, tb)),
                          X.astype(np.float64))
    assert np.array_equal(oracle_mod.gemm_f64_op(ta, tb, stored(P, ta), stored(X, tb)),
                          X[perm].astype(np.float64))


def test_op_rectangular_shapes_keep_their_roles(oracle_mod):
    """M, N and K all differ, so a swapped role would change the output shape
    or read the wrong extent."""
    rng = np.random.default_rng(9)
    M, N, K = 5, 3, 11
    A = rng.integers(-4, 5, (M, K)).astype(np.float32)
    B = rng.integers(-4, 5, (K, N)).astype(np.float32)
    want = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64)
    for ta in (0, 1):
        for tb in (0, 1):
            got = oracle_mod.gemm_f64_op(ta, tb, stored(A, ta), stored(B, tb))
            assert got.shape == (M, N) and np.array_equal(got, want)


def test_op_blas_conventions(oracle_mod):
    rng = np.random.default_rng(10)
    A = rng.standard_normal((6, 4)).astype(np.float32)    # stored K x M for transa
    B = rng.standard_normal((5, 6)).astype(np.float32)    # stored N x K for transb
    nan_c = np.full((4, 5), np.nan, dtype=np.float32)
    assert np.all(np.isfinite(oracle_mod.gemm_f64_op(1, 1, A, B, 1.0, 0.0, nan_c)))
    C0 = np.arange(20, dtype=np.float32).reshape(4, 5)
    nan_a = np.full_like(A, np.nan)
    nan_b = np.full_like(B, np.nan)
    assert np.array_equal(oracle_mod.gemm_f64_op(1, 1, nan_a, nan_b, 0.0, 2.0, C0),
                          2.0 * C0.astype(np.float64))


def test_op_invalid_arguments_rejected(oracle_mod):
    import ctypes
    lib = oracle_mod._load()
    f32p, f64p = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
    A = np.zeros((8, 8), dtype=np.float32)
    out = np.zeros(64, dtype=np.float64)
    pa = A.ctypes.data_as(f32p)
    po = out.ctypes.data_as(f64p)
    # transa == 1 with M = 8 needs lda >= 8; transb == 1 with K = 8 needs ldb >= 8
    assert lib.oracle_gemm_f64_op(1, 0, 8, 4, 4, 1.0, pa, 4, pa, 8, 0.0, None, 4, po, 1) == -1
    assert lib.oracle_gemm_f64_op(0, 1, 4, 4, 8, 1.0, pa, 8, pa, 4, 0.0, None, 4, po, 1) == -1
    assert lib.oracle_gemm_f64_op(2, 0, 4, 4, 4, 1.0, pa, 8, pa, 8, 0.0, None, 4, po, 1) == -1
    assert lib.oracle_gemm_f64_op(1, 1, 4, 4, 4, 1.0, pa, 8, pa, 8, 0.0, None, 4, po, 1) == 0
