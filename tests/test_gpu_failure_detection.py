"""Failure detection without a GPU fault: a bounded mbarrier wait that nothing
completes must give up by itself, report SGEMM_ERR_TIMEOUT through the device
status word, and leave the context usable."""
import time

import pytest

from dense_fp32_gemm_09_gb300 import load, sgemm

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports(cuda):
    torch = cuda
    lib = load()
    assert lib.sgemm_device_status() == 0            # nothing pending
    t0 = time.perf_counter()
    assert lib.sgemm_selftest_bounded_wait(100) == -5   # SGEMM_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert lib.sgemm_device_status() == 0            # read-and-clear
    A = torch.ones(300, 200, device="cuda")
    B = torch.ones(200, 100, device="cuda")
    assert torch.all(sgemm(A, B) == 200)             # the context still works


def test_selftest_rejects_bad_limits(cuda):
    lib = load()
    assert lib.sgemm_selftest_bounded_wait(0) == -1
    assert lib.sgemm_selftest_bounded_wait(100000) == -1
