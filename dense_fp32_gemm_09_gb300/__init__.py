"""GB300-native FP32 SGEMM: C = A . B, row-major, on the CUDA cores of sm_103a.

Thin Python face of the C ABI in ``include/sgemm.h``.  PyTorch supplies device
memory and streams; every step of the product runs in the library's kernels.
The library is loaded on first use and its absence is an error.
"""
from __future__ import annotations

import ctypes

from ._abi import (SGEMM_ERR_INVALID_ARG, SGEMM_ERR_LAUNCH, SGEMM_ERR_UNSUPPORTED,  # noqa: F401
                   SGEMM_ERR_WORKSPACE, SGEMM_OK, SgemmConfig, SgemmError, check, load)

__all__ = ["sgemm", "sgemm_run", "sgemm_run_ws", "sgemm_run_with", "sgemm_run_host",
           "sgemm_run_noalloc", "sgemm_run_ex", "sgemm_run_op",
           "sgemm_query_config", "sgemm_workspace_size", "kernel_table", "launch_count",
           "SgemmError", "load"]


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


# The C ABI takes sizes and leading dimensions as 32-bit ints; ctypes would
# silently wrap a larger Python int, so the binding rejects it instead.
_INT_MAX = 2**31 - 1


def _fits_int(name: str, **values) -> None:
    for what, v in values.items():
        if v > _INT_MAX:
            raise ValueError(f"{name}: {what} = {v} does not fit the library's 32-bit ints")


def _stored_ld(step: int, lines: int, width: int, name: str) -> int:
    """Leading dimension of `lines` stored rows of `width` elements that start
    `step` elements apart.  Rows that overlap (step < width) would make the
    library read or write past the view, so they are rejected; a single row has
    no step to speak of."""
    if lines > 1 and step < width:
        raise ValueError(f"{name}: its rows overlap (row stride {step} < row width {width})")
    ld = max(step, width, 1)
    _fits_int(name, leading_dimension=ld)
    return ld


def _ld(t, name: str) -> int:
    """Leading dimension of a 2-D row-major tensor view (unit column stride)."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its columns")
    return _stored_ld(t.stride(0), t.shape[0], t.shape[1], name)


def _layout(t, name: str) -> tuple[int, int]:
    """(trans, ld) of a 2-D operand view: trans 0 for a row-major view (unit
    column stride), 1 for the transpose of one (unit row stride, e.g. ``X.t()``)."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    rows, cols = t.shape
    if cols <= 1 or t.stride(1) == 1:
        return 0, _stored_ld(t.stride(0), rows, cols, name)
    if rows <= 1 or t.stride(0) == 1:
        return 1, _stored_ld(t.stride(1), cols, rows, name)
    raise ValueError(f"{name} needs a unit stride along its rows or its columns")


def _check_operand(t, name: str):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def sgemm_run(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, stream=None) -> int:
    """Raw call of ``sgemm_run`` with integer device addresses; returns the status."""
    return load().sgemm_run(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc,
                            _stream_handle(stream))


def sgemm_run_ws(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, ws_ptr, ws_bytes,
                 stream=None) -> int:
    return load().sgemm_run_ws(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, ws_ptr, ws_bytes,
                               _stream_handle(stream))


def sgemm_run_noalloc(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, stream=None) -> int:
    """Raw call of ``sgemm_run_noalloc``: like ``sgemm_run`` but the library allocates
    no device memory (split-tile scratch comes from a fixed static array)."""
    return load().sgemm_run_noalloc(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc,
                                    _stream_handle(stream))


def sgemm_run_with(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, kernel_id, schedule=0,
                   stream=None) -> int:
    return load().sgemm_run_with(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, kernel_id,
                                 schedule, _stream_handle(stream))


def sgemm_run_host(M, N, K, hA, lda, hB, ldb, hC, ldc, dA, dB, dC, stream=None) -> int:
    return load().sgemm_run_host(M, N, K, hA, lda, hB, ldb, hC, ldc, dA, dB, dC,
                                 _stream_handle(stream))


def sgemm_workspace_size(M, N, K, lda, ldb, ldc, A_ptr=None, B_ptr=None, C_ptr=None) -> int:
    out = ctypes.c_size_t(0)
    check(load().sgemm_workspace_size(M, N, K, lda, ldb, ldc, A_ptr, B_ptr, C_ptr,
                                      ctypes.byref(out)), "sgemm_workspace_size")
    return int(out.value)


def sgemm_query_config(M, N, K, lda=None, ldb=None, ldc=None, A_ptr=None, B_ptr=None,
                       C_ptr=None) -> dict:
    cfg = SgemmConfig()
    check(load().sgemm_query_config(M, N, K, lda or K, ldb or N, ldc or N, A_ptr, B_ptr, C_ptr,
                                    ctypes.byref(cfg)), "sgemm_query_config")
    d = cfg.as_dict()
    d["name"] = load().sgemm_kernel_name(cfg.kernel_id).decode()
    return d


def kernel_table() -> list[dict]:
    lib = load()
    out = []
    for i in range(lib.sgemm_num_kernels()):
        cfg = SgemmConfig()
        check(lib.sgemm_kernel_info(i, ctypes.byref(cfg)), "sgemm_kernel_info")
        d = cfg.as_dict()
        d["name"] = lib.sgemm_kernel_name(i).decode()
        out.append(d)
    return out


def launch_count() -> int:
    return int(load().sgemm_launch_count())


def sgemm_run_ex(M, N, K, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, kernel_id=-1,
                 schedule=0, stream=None) -> int:
    """Raw call of ``sgemm_run_ex``: C = alpha * A.B + beta * C."""
    return load().sgemm_run_ex(M, N, K, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc,
                               kernel_id, schedule, _stream_handle(stream))


def sgemm_run_op(transa, transb, M, N, K, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc,
                 stream=None) -> int:
    """Raw call of ``sgemm_run_op``: C = alpha * op(A).op(B) + beta * C, op = transpose
    where the flag is 1 (A then stored K x M, B stored N x K)."""
    return load().sgemm_run_op(transa, transb, M, N, K, alpha, A_ptr, lda, B_ptr, ldb, beta,
                               C_ptr, ldc, _stream_handle(stream))


def sgemm(A, B, out=None, *, alpha: float = 1.0, beta: float = 0.0,
          kernel_id: int | None = None, schedule: int = 0, stream=None):
    """C = alpha * A @ B + beta * C for float32 CUDA tensors.  A and B may be
    row-major views (unit column stride) or transposes of them (``X.t()``, unit
    row stride); ``out`` is a row-major view.

    ``out`` may be a preallocated (M, N) float32 CUDA view; with beta == 0 it is
    only written, otherwise its contents are the C of the formula (beta != 0
    needs ``out``).  ``kernel_id``/``schedule`` force a tile-table entry."""
    import torch
    _check_operand(A, "A")
    _check_operand(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
    if out is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs `out` (the C that is scaled)")
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    else:
        _check_operand(out, "out")
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must be {(M, N)}, got {tuple(out.shape)}")
    if B.device != A.device or out.device != A.device:
        raise ValueError(f"A, B and out must be on one device: {A.device}, {B.device}, "
                         f"{out.device}")
    _fits_int("sgemm", M=M, N=N, K=K)
    if M == 0 or N == 0:
        return out
    (ta, lda), (tb, ldb), ldc = _layout(A, "A"), _layout(B, "B"), _ld(out, "out")
    args = (M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc)
    with torch.cuda.device(A.device):
        if ta or tb:
            if kernel_id is not None or schedule != 0:
                raise ValueError("kernel_id / schedule cannot be forced with transposed operands")
            st = sgemm_run_op(ta, tb, M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(),
                              ldb, float(beta), out.data_ptr(), ldc, stream=stream)
            check(st, "sgemm_run_op")
        elif alpha != 1.0 or beta != 0.0:
            st = sgemm_run_ex(M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb,
                              float(beta), out.data_ptr(), ldc,
                              -1 if kernel_id is None else kernel_id, schedule, stream=stream)
            check(st, "sgemm_run_ex")
        elif kernel_id is None and schedule == 0:
            st = sgemm_run(*args, stream=stream)
            check(st, "sgemm_run")
        else:
            st = sgemm_run_with(*args, -1 if kernel_id is None else kernel_id, schedule,
                                stream=stream)
            check(st, "sgemm_run_with")
    return out
