"""ctypes declarations of the C ABI in include/sgemm.h (argument marshalling only).

Every function here forwards to the same-named symbol of libsgemm_gb300.so.
Loading fails loudly if the library has not been built: there is no other
implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SGEMM_OK = 0
SGEMM_ERR_INVALID_ARG = -1
SGEMM_ERR_ALIGNMENT = -2
SGEMM_ERR_LAUNCH = -3
SGEMM_ERR_UNSUPPORTED = -4
SGEMM_ERR_TIMEOUT = -5
SGEMM_ERR_WORKSPACE = -6


class SgemmConfig(ctypes.Structure):
    """Mirror of ``sgemm_config``."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "bm", "bn", "bk", "wm", "wn", "tm", "tn", "stages", "threads", "smem_bytes",
        "split_k", "kernel_id", "vec", "grid", "tiles", "sk_tiles", "ctas_per_sm", "fma2",
        "packed", "sk_gap", "cluster")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


# name -> (restype, argtypes)
_i, _sz, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
_RUN = [_i, _i, _i, _vp, _i, _vp, _i, _vp, _i]
SIGNATURES = {
    "sgemm_run": (_i, _RUN + [_vp]),
    "sgemm_run_ws": (_i, _RUN + [_vp, _sz, _vp]),
    "sgemm_run_ex": (_i, [_i, _i, _i, ctypes.c_float, _vp, _i, _vp, _i, ctypes.c_float, _vp, _i,
                          _i, _i, _vp]),
    "sgemm_run_op": (_i, [_i, _i, _i, _i, _i, ctypes.c_float, _vp, _i, _vp, _i, ctypes.c_float,
                          _vp, _i, _vp]),
    "sgemm_run_noalloc": (_i, _RUN + [_vp]),
    "sgemm_workspace_size": (_i, [_i, _i, _i, _i, _i, _i, _vp, _vp, _vp,
                                  ctypes.POINTER(_sz)]),
    "sgemm_run_with": (_i, _RUN + [_i, _i, _vp]),
    "sgemm_query_config": (_i, [_i, _i, _i, _i, _i, _i, _vp, _vp, _vp,
                                ctypes.POINTER(SgemmConfig)]),
    "sgemm_run_host": (_i, _RUN + [_vp, _vp, _vp, _vp]),
    "sgemm_tf32x3_query_config": (_i, [_i, _i, _i, ctypes.POINTER(SgemmConfig)]),
    "sgemm_tf32x3_run": (_i, _RUN + [_vp]),
    "sgemm_tf32x3_run_ex": (_i, [_i, _i, _i, ctypes.c_float, _vp, _i, _vp, _i, ctypes.c_float,
                                 _vp, _i, _vp, _sz, _vp]),
    "sgemm_tf32x3_workspace_size": (_i, [_i, _i, _i, ctypes.POINTER(_sz)]),
    "sgemm_tf32x3_prepare": (_i, _RUN[:7] + [_vp, _sz, _vp]),
    "sgemm_tf32x3_multiply": (_i, [_i, _i, _i, ctypes.c_float, ctypes.c_float, _vp, _i, _vp, _sz,
                                   _vp]),
    "sgemm_device_status": (_i, []),
    "sgemm_selftest_bounded_wait": (_i, [_i]),
    "sgemm_schedule_check": (_i, [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(SgemmConfig)]),
    "sgemm_choose_check": (_i, [_i] * 8 + [ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "sgemm_host_plan_check": (_i, [_i, _i, _i] + [ctypes.POINTER(_i)] * 3),
    "sgemm_num_kernels": (_i, []),
    "sgemm_kernel_info": (_i, [_i, ctypes.POINTER(SgemmConfig)]),
    "sgemm_kernel_name": (ctypes.c_char_p, [_i]),
    "sgemm_status_string": (ctypes.c_char_p, [_i]),
    "sgemm_last_error": (ctypes.c_char_p, []),
    "sgemm_launch_count": (ctypes.c_uint64, []),
    "sgemm_shutdown": (_i, []),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """The loaded library.  Raises if it is absent (no silent fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"{path} is missing: build the CUDA library first "
                    "(python -m dense_fp32_gemm_09_gb300.build or __graft_entry__.build())")
            _build.build()
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class SgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        self.status = status
        msg = lib.sgemm_status_string(status).decode()
        detail = lib.sgemm_last_error().decode()
        super().__init__(f"{where}: {msg}" + (f" ({detail})" if detail else ""))


def check(status: int, where: str) -> None:
    if status != SGEMM_OK:
        raise SgemmError(status, where)
