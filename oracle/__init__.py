"""CPU oracle for the row-major FP32 product C = A . B.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference arm may import this package.  The CUDA
library never imports, links or calls it, and this package never imports the
CUDA library: the two share no code.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, fp64 accumulation, k
ascending); this module only compiles it with gcc and marshals numpy arrays
through ctypes.  See that file's header for the definition it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i, i64 = ctypes.c_int, ctypes.c_int64
        lib.oracle_gemm_f64.argtypes = [i, i, i, f32p, i64, f32p, i64, f64p, i64, i]
        lib.oracle_gemm_f64_rows.argtypes = [i, i, i, f32p, i64, f32p, i64, i32p, i, f64p, i]
        lib.oracle_gemm_f64_elems.argtypes = [i, i, i, f32p, i64, f32p, i64, i32p, i32p, i,
                                              f64p]
        lib.oracle_gemm_f32_fma_seq.argtypes = [i, i, i, f32p, i64, f32p, i64, f32p, i64]
        d = ctypes.c_double
        lib.oracle_gemm_f64_ex.argtypes = [i, i, i, d, f32p, i64, f32p, i64, d, f32p, i64,
                                           i32p, i, f64p, i]
        lib.oracle_gemm_f64_op.argtypes = [i, i, i, i, i, d, f32p, i64, f32p, i64, d, f32p,
                                           i64, f64p, i]
        for fn in (lib.oracle_gemm_f64, lib.oracle_gemm_f64_rows, lib.oracle_gemm_f64_ex,
                   lib.oracle_gemm_f64_op,
                   lib.oracle_gemm_f64_elems, lib.oracle_gemm_f32_fma_seq,
                   lib.oracle_max_threads):
            fn.restype = ctypes.c_int
        _lib = lib
        return lib


def _mat(x, name):
    """A 2-D float32 numpy view with unit column stride; returns (array, ld)."""
    x = np.asarray(x)
    if x.dtype != np.float32 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D float32 array")
    if x.strides[1] != 4 or x.strides[0] % 4 != 0 or x.strides[0] < 0:
        x = np.ascontiguousarray(x)
    ld = max(x.strides[0] // 4, x.shape[1], 1)
    return x, ld


def _ptr(x, ctype):
    return x.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return int(os.environ.get("ORACLE_THREADS", os.cpu_count() or 1))


def gemm_f64(A, B, nthreads: int | None = None) -> np.ndarray:
    """C = A.B summed in double with k ascending; returns an M x N float64 array.

    A and B may be strided row-major views (leading dimension > width); padding
    between rows is never read."""
    A, lda = _mat(A, "A")
    B, ldb = _mat(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    C = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_f64(M, N, K, _ptr(A, ctypes.c_float), lda,
                                 _ptr(B, ctypes.c_float), ldb,
                                 _ptr(C, ctypes.c_double), max(N, 1),
                                 nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm_f64 rejected its arguments")
    return C


def gemm_f64_rows(A, B, rows, nthreads: int | None = None) -> np.ndarray:
    """Rows ``rows`` of C = A.B in double: a len(rows) x N float64 array."""
    A, lda = _mat(A, "A")
    B, ldb = _mat(B, "B")
    M, K = A.shape
    N = B.shape[1]
    if B.shape[0] != K:
        raise ValueError("inner dimensions differ")
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    out = np.empty((rows.size, N), dtype=np.float64)
    rc = _load().oracle_gemm_f64_rows(M, N, K, _ptr(A, ctypes.c_float), lda,
                                      _ptr(B, ctypes.c_float), ldb,
                                      _ptr(rows, ctypes.c_int32), rows.size,
                                      _ptr(out, ctypes.c_double),
                                      nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm_f64_rows rejected its arguments")
    return out


def gemm_f64_elems(A, B, ii, jj) -> np.ndarray:
    """Elements C[ii[e], jj[e]] of C = A.B in double."""
    A, lda = _mat(A, "A")
    B, ldb = _mat(B, "B")
    M, K = A.shape
    N = B.shape[1]
    if B.shape[0] != K:
        raise ValueError("inner dimensions differ")
    ii = np.ascontiguousarray(ii, dtype=np.int32)
    jj = np.ascontiguousarray(jj, dtype=np.int32)
    if ii.shape != jj.shape:
        raise ValueError("ii and jj differ in length")
    out = np.empty(ii.size, dtype=np.float64)
    rc = _load().oracle_gemm_f64_elems(M, N, K, _ptr(A, ctypes.c_float), lda,
                                       _ptr(B, ctypes.c_float), ldb,
                                       _ptr(ii, ctypes.c_int32), _ptr(jj, ctypes.c_int32),
                                       ii.size, _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_gemm_f64_elems rejected its arguments")
    return out


def gemm_f64_ex(alpha, A, B, beta, C0, rows=None, nthreads: int | None = None) -> np.ndarray:
    """alpha * (A.B) + beta * C0 in double (BLAS conventions: beta == 0 does not
    read C0, alpha == 0 does not read A or B).  With `rows`, only those rows of the
    result are returned.  C0 may be None when beta == 0."""
    A, lda = _mat(A, "A")
    B, ldb = _mat(B, "B")
    M, K = A.shape
    N = B.shape[1]
    if B.shape[0] != K:
        raise ValueError("inner dimensions differ")
    if C0 is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C0")
        C0 = np.zeros((1, max(N, 1)), dtype=np.float32)
        ldc0 = max(N, 1)
    else:
        C0, ldc0 = _mat(C0, "C0")
        if C0.shape != (M, N):
            raise ValueError("C0 must be M x N")
    if rows is None:
        rp, nrows = None, M
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        rp, nrows = _ptr(rows, ctypes.c_int32), rows.size
    out = np.empty((nrows, N), dtype=np.float64)
    rc = _load().oracle_gemm_f64_ex(M, N, K, float(alpha), _ptr(A, ctypes.c_float), lda,
                                    _ptr(B, ctypes.c_float), ldb, float(beta),
                                    _ptr(C0, ctypes.c_float), ldc0, rp, nrows,
                                    _ptr(out, ctypes.c_double), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm_f64_ex rejected its arguments")
    return out


def gemm_f64_op(transa, transb, A, B, alpha=1.0, beta=0.0, C0=None,
                nthreads: int | None = None) -> np.ndarray:
    """alpha * op(A).op(B) + beta * C0 in double, op(X) = X^T where the flag is 1.

    A and B are passed as STORED (row-major, possibly strided): with transa == 1,
    A is K x M; with transb == 1, B is N x K."""
    A, lda = _mat(A, "A")
    B, ldb = _mat(B, "B")
    M, K = (A.shape[1], A.shape[0]) if transa else A.shape
    KB, N = (B.shape[1], B.shape[0]) if transb else B.shape
    if K != KB:
        raise ValueError(f"inner dimensions differ: {K} vs {KB}")
    if C0 is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C0")
        C0 = np.zeros((1, max(N, 1)), dtype=np.float32)
        ldc0 = max(N, 1)
    else:
        C0, ldc0 = _mat(C0, "C0")
        if C0.shape != (M, N):
            raise ValueError("C0 must be M x N")
    out = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_f64_op(int(transa), int(transb), M, N, K, float(alpha),
                                    _ptr(A, ctypes.c_float), lda, _ptr(B, ctypes.c_float), ldb,
                                    float(beta), _ptr(C0, ctypes.c_float), ldc0,
                                    _ptr(out, ctypes.c_double), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm_f64_op rejected its arguments")
    return out


def gemm_f32_fma_seq(A, B) -> np.ndarray:
    """C = A.B accumulated in fp32 with one fmaf per term, k ascending."""
    A, lda = _mat(A, "A")
    B, ldb = _mat(B, "B")
    M, K = A.shape
    N = B.shape[1]
    if B.shape[0] != K:
        raise ValueError("inner dimensions differ")
    C = np.empty((M, N), dtype=np.float32)
    rc = _load().oracle_gemm_f32_fma_seq(M, N, K, _ptr(A, ctypes.c_float), lda,
                                         _ptr(B, ctypes.c_float), ldb,
                                         _ptr(C, ctypes.c_float), max(N, 1))
    if rc != 0:
        raise ValueError("oracle_gemm_f32_fma_seq rejected its arguments")
    return C


def raw_call_f64(M, N, K, A, lda, B, ldb, C, ldc, nthreads=1) -> int:
    """Direct call with explicit sizes (used by tests of argument validation)."""
    return _load().oracle_gemm_f64(M, N, K, A, lda, B, ldb, C, ldc, nthreads)


def max_threads() -> int:
    return int(_load().oracle_max_threads())
