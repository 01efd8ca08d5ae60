"""The host-buffer entry's plan as host logic (no GPU).

sgemm_run_host splits C into row panels and computes the first panel in
k-chunks as its inputs arrive; it keeps one event per panel and per chunk in
arrays of SGEMM_HOST_MAX_PANELS.  sgemm_host_plan_check returns that plan, so
the split and the bound on both counts are checked here for default sizes and
for every tuning override, including nonsense ones."""
import ctypes
import itertools

import pytest

MAX_PANELS = 16   # SGEMM_HOST_MAX_PANELS in include/sgemm.h


def _plan(lib, M, N, K):
    n = ctypes.c_int(-1)
    rows = (ctypes.c_int * MAX_PANELS)(*([-1] * MAX_PANELS))
    kc = ctypes.c_int(-1)
    assert lib.sgemm_host_plan_check(M, N, K, ctypes.byref(n), rows, ctypes.byref(kc)) == 0
    return list(rows[:n.value]), kc.value


def _check_plan(M, K, rows, kc):
    assert 1 <= len(rows) <= MAX_PANELS
    assert sum(rows) == M and all(r > 0 for r in rows)
    assert all(r % 256 == 0 for r in rows[:-1]), rows
    if K == 0:
        assert kc == 0
    else:
        assert 1 <= kc <= K
        assert -(-K // kc) <= MAX_PANELS, (K, kc)


@pytest.mark.parametrize("shape,rows,kc", [
    # >= 4e9 multiply-adds: a quarter of C in 4 k-chunks, then 65 %, then the last 10 %.
    ((4096, 4096, 4096), [1024, 2560, 512], 1024),
    ((8192, 8192, 8192), [2048, 5376, 768], 2048),
    # >= 5e8: two halves, the first in 2 k-chunks.
    ((1024, 1024, 1024), [512, 512], 512),
    # smaller: one panel, not chunked.
    ((256, 256, 256), [256], 256),
    ((100, 300, 7), [100], 7),
    ((3000, 40, 0), [3000], 0),
])
def test_default_plans(lib, shape, rows, kc):
    assert _plan(lib, *shape) == (rows, kc)


def test_plans_cover_C_for_many_shapes(lib):
    Ms = [1, 2, 255, 256, 257, 1000, 3001, 4096, 16384, 100000]
    NKs = [(1, 1), (64, 4096), (2047, 1999), (4096, 4096), (8192, 1), (33, 100000)]
    for M, (N, K) in itertools.product(Ms, NKs):
        _check_plan(M, K, *_plan(lib, M, N, K))


@pytest.mark.parametrize("env", [
    {"SGEMM_HOST_PANELS": "100"},
    {"SGEMM_HOST_PANELS": "7"},
    {"SGEMM_HOST_PANELS": "-3"},
    {"SGEMM_HOST_SPLIT": ",".join(["1"] * 40)},
    {"SGEMM_HOST_SPLIT": "2000000000,2000000000,5"},   # the percentages' sum exceeds an int
    {"SGEMM_HOST_SPLIT": "0,,x,-4"},                     # nothing usable: the default split
    {"SGEMM_HOST_KCHUNKS": "1000"},
    {"SGEMM_HOST_KCHUNKS": "0"},
    {"SGEMM_HOST_KCHUNKS": "-9"},
])
def test_overrides_stay_within_the_event_arrays(lib, monkeypatch, env):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    for M, N, K in [(4096, 4096, 4096), (100000, 64, 70000), (300, 5, 3), (16384, 64, 4096)]:
        _check_plan(M, K, *_plan(lib, M, N, K))


def test_override_values(lib, monkeypatch):
    monkeypatch.setenv("SGEMM_HOST_PANELS", "4")
    monkeypatch.setenv("SGEMM_HOST_KCHUNKS", "8")
    assert _plan(lib, 4096, 4096, 4096) == ([1024, 1024, 1024, 1024], 512)
    monkeypatch.setenv("SGEMM_HOST_SPLIT", "50,50")          # takes precedence over PANELS
    assert _plan(lib, 4096, 512, 512)[0] == [2048, 2048]


def test_invalid_arguments(lib):
    n = ctypes.c_int()
    for args in [(0, 4, 4), (4, 0, 4), (4, 4, -1)]:
        assert lib.sgemm_host_plan_check(*args, ctypes.byref(n), None, None) == -1, args
    assert lib.sgemm_host_plan_check(4, 4, 4, None, None, None) == -1
    assert lib.sgemm_host_plan_check(4, 4, 4, ctypes.byref(n), None, None) == 0 and n.value == 1
