"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a private copy of the oracle's C source (a
dropped term, a wrong sign, a transposed operand, an ignored leading dimension,
unfused accumulation), builds it with gcc and checks that at least one pin of
test_oracle.py's kind fails on it while the unmodified source passes them all.
Only square, in-bounds inputs are used so that no mutant reads outside its
buffers.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from conftest import REPO, read_golden

SRC = os.path.join(REPO, "oracle", "sgemm_oracle.c")

MUTATIONS = {
    "none": [],
    "drop_last_term": [("for (int k = 0; k < K; ++k) {\n        const double a",
                        "for (int k = 0; k < K - 1; ++k) {\n        const double a")],
    "wrong_sign": [("crow[j] += a * (double)brow[j];", "crow[j] -= a * (double)brow[j];")],
    "transposed_B": [("crow[j] += a * (double)brow[j];",
                      "crow[j] += a * (double)B[(int64_t)j * ldb + k];")],
    "ignores_lda": [("one_row_f64(N, K, A + (int64_t)i * lda,",
                     "one_row_f64(N, K, A + (int64_t)i * K,")],
    "drops_beta_term": [("o[j] += beta * (double)C0[(int64_t)i * ldc0 + j];",
                         "o[j] += 0.0 * (double)C0[(int64_t)i * ldc0 + j];")],
    "op_ignores_transb": [("const double b = transb ? (double)B[(int64_t)j * ldb + k]",
                           "const double b = transb ? (double)B[(int64_t)k * ldb + j]")],
    "op_ignores_transa": [("const double a = transa ? (double)A[(int64_t)k * lda + i]",
                           "const double a = transa ? (double)A[(int64_t)i * lda + k]")],
    "unfused_fp32": [("acc = fmaf(A[(int64_t)i * lda + k], B[(int64_t)k * ldb + j], acc);",
                      "acc = A[(int64_t)i * lda + k] * B[(int64_t)k * ldb + j] + acc;")],
}


def build_variant(tmp_path, name):
    src = open(SRC).read()
    for old, new in MUTATIONS[name]:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(so), str(c), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    f32p, f64p = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
    i, i64 = ctypes.c_int, ctypes.c_int64
    lib.oracle_gemm_f64.argtypes = [i, i, i, f32p, i64, f32p, i64, f64p, i64, i]
    lib.oracle_gemm_f32_fma_seq.argtypes = [i, i, i, f32p, i64, f32p, i64, f32p, i64]
    lib.oracle_gemm_f64_ex.argtypes = [i, i, i, ctypes.c_double, f32p, i64, f32p, i64,
                                       ctypes.c_double, f32p, i64, ctypes.c_void_p, i, f64p, i]
    lib.oracle_gemm_f64_op.argtypes = [i, i, i, i, i, ctypes.c_double, f32p, i64, f32p, i64,
                                       ctypes.c_double, f32p, i64, f64p, i]
    return lib


def call_f64(lib, A, lda, B, ldb, M, N, K):
    C = np.empty((M, N), dtype=np.float64)
    rc = lib.oracle_gemm_f64(M, N, K, A.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), lda,
                             B.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), ldb,
                             C.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), N, 1)
    assert rc == 0
    return C


def failing_pins(lib):
    """Names of the pins this build fails."""
    fails = []
    n = 31
    rng = np.random.default_rng(1)
    # identity with NaN padding between rows (square, ld = n + 3)
    buf = np.full((n, n + 3), np.nan, dtype=np.float32)
    X = rng.standard_normal((n, n)).astype(np.float32)
    buf[:, :n] = X
    ibuf = np.full((n, n + 3), np.nan, dtype=np.float32)
    ibuf[:, :n] = np.eye(n, dtype=np.float32)
    if not np.array_equal(call_f64(lib, buf, n + 3, ibuf, n + 3, n, n, n), X.astype(np.float64)):
        fails.append("identity")
    # permutation
    perm = rng.permutation(n)
    P = np.zeros((n, n), dtype=np.float32)
    P[np.arange(n), perm] = 1
    if not np.array_equal(call_f64(lib, P, n, X, n, n, n, n), X[perm].astype(np.float64)):
        fails.append("permutation")
    # small integers
    A = rng.integers(-8, 9, (n, n)).astype(np.float32)
    B = rng.integers(-8, 9, (n, n)).astype(np.float32)
    want = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64)
    if not np.array_equal(call_f64(lib, A, n, B, n, n, n, n), want):
        fails.append("small_integers")
    # scaled form: alpha * A.B + beta * C0 on small integers
    C0 = rng.integers(-50, 51, (n, n)).astype(np.float32)
    out = np.empty((n, n), dtype=np.float64)
    lib.oracle_gemm_f64_ex(n, n, n, 2.0, A.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), n,
                           B.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), n, -3.0,
                           C0.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), n, None, n,
                           out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), 1)
    if not np.array_equal(out, 2 * want - 3 * C0.astype(np.float64)):
        fails.append("scaled_small_integers")
    # transposed operands on small integers: op(A).op(B) with both stored transposed
    out = np.empty((n, n), dtype=np.float64)
    At, Bt = np.ascontiguousarray(A.T), np.ascontiguousarray(B.T)
    lib.oracle_gemm_f64_op(1, 1, n, n, n, 1.0, At.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                           n, Bt.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), n, 0.0, None,
                           n, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), 1)
    if not np.array_equal(out, want):
        fails.append("op_small_integers")
    # the pages' printed worked example (fp32 mode)
    rows = {r[0]: r[1:] for r in read_golden("p1_micro_gemm_4x4.txt")}
    K = int(rows["K"][0])
    A1 = ((np.arange(4 * K) % 7).astype(np.float32) * np.float32(0.1)).reshape(4, K)
    B1 = ((np.arange(4 * K) % 5).astype(np.float32) * np.float32(0.2)).reshape(K, 4)
    C1 = np.empty((4, 4), dtype=np.float32)
    lib.oracle_gemm_f32_fma_seq(4, 4, K, A1.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), K,
                                B1.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), 4,
                                C1.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), 4)
    if ["%f" % float(v) for v in C1[0]] != rows["C_row0_printed"]:
        fails.append("p1_printed")
    return fails


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    fails = failing_pins(build_variant(tmp_path, name))
    if name == "none":
        assert fails == []
    else:
        assert fails, f"no pin caught mutation {name}"
