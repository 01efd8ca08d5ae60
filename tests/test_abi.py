"""The C-ABI library: it loads, exports every symbol include/sgemm.h declares,
and rejects bad arguments before touching the GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

from conftest import REPO

HEADER = os.path.join(REPO, "include", "sgemm.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SGEMM_API\s+[\w\s\*]+?\b(sgemm_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("sgemm_run", "sgemm_query_config", "sgemm_status_string", "sgemm_run_ws",
                 "sgemm_workspace_size", "sgemm_run_host"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    from dense_fp32_gemm_09_gb300 import _abi
    assert set(_abi.SIGNATURES) == set(declared_functions())


def test_config_struct_matches_header():
    from dense_fp32_gemm_09_gb300 import _abi
    text = open(HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} sgemm_config;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b(\w+)\s*[,;]", body)
    assert [f for f, _ in _abi.SgemmConfig._fields_] == fields


def test_status_strings(lib):
    assert lib.sgemm_status_string(0) == b"SGEMM_OK"
    assert lib.sgemm_status_string(-1) == b"SGEMM_ERR_INVALID_ARG"
    assert lib.sgemm_status_string(-6) == b"SGEMM_ERR_WORKSPACE"
    assert lib.sgemm_status_string(12345) == b"SGEMM_ERR_UNKNOWN"


def test_kernel_table_static_info(lib):
    from dense_fp32_gemm_09_gb300._abi import SgemmConfig
    n = lib.sgemm_num_kernels()
    assert n >= 3
    names = set()
    for i in range(n):
        cfg = SgemmConfig()
        assert lib.sgemm_kernel_info(i, ctypes.byref(cfg)) == 0
        assert cfg.bm % cfg.wm == 0 and cfg.bn % cfg.wn == 0
        assert cfg.threads == 32 * (cfg.bm // cfg.wm) * (cfg.bn // cfg.wn)
        assert cfg.wm * cfg.wn == 32 * cfg.tm * cfg.tn
        assert cfg.vec in (1, 4)
        names.add(lib.sgemm_kernel_name(i))
    assert len(names) == n
    assert lib.sgemm_kernel_info(n, ctypes.byref(SgemmConfig())) == -4
    assert lib.sgemm_kernel_name(n) == b""


P = 0x10000  # a 16-byte-aligned fake device address: these calls never launch


@pytest.mark.parametrize("args", [
    (-1, 4, 4, P, 4, P, 4, P * 8, 4),          # negative M
    (4, -1, 4, P, 4, P, 4, P * 8, 4),          # negative N
    (4, 4, -1, P, 4, P, 4, P * 8, 4),          # negative K
    (4, 4, 8, P, 7, P, 4, P * 8, 4),           # lda < K
    (4, 4, 4, P, 4, P, 3, P * 8, 4),           # ldb < N
    (4, 4, 4, P, 4, P, 4, P * 8, 3),           # ldc < N
    (4, 4, 4, 0, 4, P, 4, P * 8, 4),           # null A
    (4, 4, 4, P, 4, 0, 4, P * 8, 4),           # null B
    (4, 4, 4, P, 4, P * 4, 4, 0, 4),           # null C
    (4, 4, 4, P, 4, P * 4, 4, P + 8, 4),       # C overlaps A
    (4, 4, 4, P * 64, 4, P, 4, P + 16, 4),     # C overlaps B
])
def test_invalid_arguments_rejected_before_launch(lib, args):
    assert lib.sgemm_run(*args, None) == -1
    assert lib.sgemm_run_with(*args, -1, 0, None) == -1
    assert lib.sgemm_run_ws(*args, None, 0, None) == -1
    assert lib.sgemm_last_error() != b""


BIG = 2**30 + 1   # one past the largest dimension the kernels index in 32 bits


@pytest.mark.parametrize("M,N,K", [(BIG, 4, 4), (4, BIG, 4), (4, 4, BIG)])
def test_dimensions_above_2_30_are_refused_before_launch(lib, M, N, K):
    """A dimension above 2^30 is refused by every entry point (nothing is planned);
    the fake pointers are far enough apart that no overlap check fires first."""
    from dense_fp32_gemm_09_gb300._abi import SgemmConfig
    lda, ldb, ldc = max(K, 1), max(N, 1), max(N, 1)
    a, b, c = P, P + (1 << 44), P + (1 << 45)
    assert lib.sgemm_run(M, N, K, a, lda, b, ldb, c, ldc, None) == -4
    assert b"2^30" in lib.sgemm_last_error()
    assert lib.sgemm_run_ws(M, N, K, a, lda, b, ldb, c, ldc, None, 0, None) == -4
    assert lib.sgemm_run_ex(M, N, K, 1.0, a, lda, b, ldb, 0.0, c, ldc, -1, 0, None) == -4
    assert lib.sgemm_run_noalloc(M, N, K, a, lda, b, ldb, c, ldc, None) == -4
    assert lib.sgemm_tf32x3_run(M, N, K, a, lda, b, ldb, c, ldc, None) == -4
    out = ctypes.c_size_t(0)
    assert lib.sgemm_workspace_size(M, N, K, lda, ldb, ldc, None, None, None,
                                    ctypes.byref(out)) == -4
    assert lib.sgemm_tf32x3_workspace_size(M, N, K, ctypes.byref(out)) == -4
    cfg = SgemmConfig()
    assert lib.sgemm_query_config(M, N, K, lda, ldb, ldc, None, None, None,
                                  ctypes.byref(cfg)) == -4
    assert lib.sgemm_schedule_check(M, N, K, 0, 152, 1, 0, ctypes.byref(cfg)) == -4
    n = ctypes.c_int(0)
    assert lib.sgemm_host_plan_check(M, N, K, ctypes.byref(n), None, None) == -4


def test_largest_dimension_is_planned(lib):
    """2^30 itself is accepted: the host-side schedule walk plans it."""
    from dense_fp32_gemm_09_gb300._abi import SgemmConfig
    cfg = SgemmConfig()
    assert lib.sgemm_schedule_check(2**30, 64, 64, 0, 152, 1, 0, ctypes.byref(cfg)) == 0
    assert cfg.tiles > 0


def test_empty_output_is_a_noop(lib):
    assert lib.sgemm_run(0, 5, 3, P, 3, P * 4, 5, P * 8, 5, None) == 0
    assert lib.sgemm_run(5, 0, 3, P, 3, P * 4, 1, P * 8, 1, None) == 0
    assert lib.sgemm_run(0, 0, 0, 0, 1, 0, 1, 0, 1, None) == 0


def test_bad_kernel_or_schedule(lib):
    assert lib.sgemm_run_with(4, 4, 4, P, 4, P * 4, 4, P * 8, 4, -7, 0, None) == -4
    assert lib.sgemm_run_with(4, 4, 4, P, 4, P * 4, 4, P * 8, 4, 0, 9, None) == -1


def test_workspace_size_rejects_bad_sizes(lib):
    out = ctypes.c_size_t(99)
    assert lib.sgemm_workspace_size(-1, 4, 4, 4, 4, 4, None, None, None, ctypes.byref(out)) == -1
    assert lib.sgemm_workspace_size(4, 4, 0, 1, 4, 4, None, None, None, ctypes.byref(out)) == 0
    assert out.value == 0


def test_product_path_does_not_reference_the_oracle():
    """The library sources and the binding never name the oracle package."""
    pkg = os.path.join(REPO, "dense_fp32_gemm_09_gb300")
    for root, _, files in os.walk(pkg):
        if "_lib" in root:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(root, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text and "sgemm_oracle" not in text, f


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    from dense_fp32_gemm_09_gb300 import _abi
    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _abi.load()


def test_binding_layout_of_views():
    # Stride logic only (CPU tensors): what leading dimension each view maps to.
    import torch
    from dense_fp32_gemm_09_gb300 import _layout, _ld
    X = torch.zeros(6, 10)
    assert _layout(X, "X") == (0, 10)
    assert _layout(X[:, 2:7], "X") == (0, 10)            # column slice keeps the row step
    assert _layout(X.t(), "X") == (1, 10)                # transpose of a row-major view
    assert _layout(X[1:2], "X") == (0, 10)               # one row
    assert _layout(X[:, 3:4], "X") == (0, 10)            # one column
    assert _layout(torch.zeros(5, 0), "X")[0] == 0       # K = 0
    assert _ld(X[2:5, 1:9], "out") == 10


@pytest.mark.parametrize("make", [
    lambda t: t.zeros(1).expand(4, 1),                   # every row is the same element
    lambda t: t.zeros(8).as_strided((3, 4), (2, 1)),     # rows overlap by half
    lambda t: t.zeros(8).as_strided((4, 3), (1, 2)).t().t(),
    lambda t: t.zeros(16).as_strided((3, 4), (1, 2)),    # transposed view whose columns overlap
])
def test_binding_rejects_overlapping_rows(make):
    # The library would read (or, for `out`, write) past such a view's storage.
    import torch
    from dense_fp32_gemm_09_gb300 import _layout, _ld
    v = make(torch)
    with pytest.raises(ValueError, match="overlap"):
        _layout(v, "A")
    if v.shape[1] <= 1 or v.stride(1) == 1:
        with pytest.raises(ValueError, match="overlap"):
            _ld(v, "out")


def test_binding_rejects_values_beyond_32_bits():
    # ctypes would wrap 2**32 + 5 to 5 without a word.
    from dense_fp32_gemm_09_gb300 import _fits_int, _layout
    _fits_int("x", M=2**31 - 1)
    with pytest.raises(ValueError, match="32-bit"):
        _fits_int("x", K=2**31)

    class View:   # shape and strides of a view too large to allocate here
        shape = (2, 3)

        def dim(self):
            return 2

        def stride(self, i):
            return (2**31, 1)[i]

    with pytest.raises(ValueError, match="32-bit"):
        _layout(View(), "A")
