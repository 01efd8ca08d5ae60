"""Host-side checks of the persistent / stream-K schedule (no GPU).

sgemm_schedule_check plans a problem for a given SM count and residency and
walks every CTA's k-slice list with the same code the kernel runs."""
import ctypes
import itertools

import pytest

SHAPES = [(1, 1, 1), (3, 5, 7), (64, 64, 16), (65, 63, 17), (129, 127, 300), (256, 256, 256),
          (1, 1, 100000), (64, 64, 300000), (300, 1, 65536),
          (1024, 1024, 1024), (3001, 2047, 1999), (4096, 4096, 4096), (16384, 64, 4096),
          (8192, 8192, 8192), (5000, 300, 33), (128, 128, 100000)]
MACHINES = [(152, 1), (152, 2), (152, 3), (148, 2), (7, 1), (1, 1), (13, 4)]


def _cfg():
    from dense_fp32_gemm_09_gb300._abi import SgemmConfig
    return SgemmConfig()


@pytest.mark.parametrize("schedule", [0, 1, 2])
def test_schedule_covers_each_slice_once(lib, schedule):
    n = lib.sgemm_num_kernels()
    for kid, (M, N, K), (sms, occ) in itertools.product(range(n), SHAPES, MACHINES):
        cfg = _cfg()
        rc = lib.sgemm_schedule_check(M, N, K, kid, sms, occ, schedule, ctypes.byref(cfg))
        assert rc == 0, (kid, M, N, K, sms, occ, schedule, lib.sgemm_last_error())
        assert cfg.grid <= sms * occ
        assert cfg.tiles == -(-M // cfg.bm) * -(-N // cfg.bn)
        if schedule == 1:
            assert cfg.sk_tiles == 0 and cfg.split_k == 1


def test_stream_k_balances_a_partial_last_wave(lib):
    # 4096^3 with 128x256 tiles: 512 tiles on 152 resident CTAs -> 3 full waves
    # plus 56 tiles shared out by k-slices.
    table = [lib.sgemm_kernel_name(i).decode() for i in range(lib.sgemm_num_kernels())]
    kid = table.index("128x256x64_t8x16_s2_f2_v4")
    cfg = _cfg()
    assert lib.sgemm_schedule_check(4096, 4096, 4096, kid, 152, 1, 0, ctypes.byref(cfg)) == 0
    assert (cfg.tiles, cfg.grid, cfg.sk_tiles) == (512, 152, 512 - 3 * 152)
    assert cfg.split_k >= 2
    cfg = _cfg()
    assert lib.sgemm_schedule_check(4096, 4096, 4096, kid, 152, 1, 1, ctypes.byref(cfg)) == 0
    assert cfg.sk_tiles == 0 and cfg.grid == 152


def test_small_problem_splits_k(lib):
    table = [lib.sgemm_kernel_name(i).decode() for i in range(lib.sgemm_num_kernels())]
    kid = table.index("128x256x32_t8x16_s4_f2_v4")
    cfg = _cfg()
    assert lib.sgemm_schedule_check(1024, 1024, 1024, kid, 152, 1, 0, ctypes.byref(cfg)) == 0
    assert cfg.tiles == 32 and cfg.sk_tiles == 32 and cfg.grid == 152


def test_rejects_bad_arguments(lib):
    assert lib.sgemm_schedule_check(0, 4, 4, 0, 152, 2, 0, None) == -1
    assert lib.sgemm_schedule_check(4, 4, 4, 0, 0, 2, 0, None) == -1
    assert lib.sgemm_schedule_check(4, 4, 4, 999, 152, 2, 0, None) == -1


@pytest.mark.parametrize("M,N,K", [(67000, 64, 32768), (50000, 45000, 8)])
def test_schedule_of_operands_past_2_31_elements(lib, M, N, K):
    """The shapes of the GPU tests whose A or C hold more than 2**31 elements."""
    for kid in range(lib.sgemm_num_kernels()):
        for sms, occ in [(152, 1), (152, 4)]:
            cfg = _cfg()
            rc = lib.sgemm_schedule_check(M, N, K, kid, sms, occ, 0, ctypes.byref(cfg))
            assert rc == 0, (kid, sms, occ, lib.sgemm_last_error())
