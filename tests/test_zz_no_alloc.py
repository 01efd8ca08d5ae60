"""sgemm_run_noalloc: the entry point for callers that cannot let the library
allocate device memory (cudaMalloc may synchronise the device and take
unbounded time, and some processes fix their device memory budget up front).

It runs the same kernels as sgemm_run but takes the stream-K partial tiles from
a static array compiled into the library.  Checked here through the C ABI:
two calls in a row (the second one finds the array dirty from the first) must
agree with sgemm_run within the parity tolerance of the other GPU tests, and
must not change the device's free memory.  This file is collected last so that
a failure here comes after every other test has run.
"""
import numpy as np
import pytest

from dense_fp32_gemm_09_gb300 import load, sgemm, sgemm_workspace_size
from dense_fp32_gemm_09_gb300.workloads import make_inputs, random_pair

pytestmark = pytest.mark.gpu


def tolerance(A, B):
    return 1e-6 * A.shape[1] * float(A.abs().max()) * float(B.abs().max())


@pytest.mark.parametrize("case", ["sgemm_1024", "sgemm_ragged_3001x2047x1999", "small_dp"])
def test_noalloc_matches_sgemm_run_twice(cuda, case):
    torch = cuda
    lib = load()
    if case == "small_dp":
        A, B = random_pair(64, 64, 64, seed=5)      # one tile: no scratch needed
    else:
        A, B = make_inputs(case)
    M, K = A.shape
    N = B.shape[1]
    dA, dB = A.cuda(), B.cuda()
    ref = sgemm(dA, dB)                                  # the existing entry point
    torch.cuda.synchronize()
    need = sgemm_workspace_size(M, N, K, K, N, N, dA.data_ptr(), dB.data_ptr(), ref.data_ptr())
    if case != "small_dp":
        assert 0 < need <= 40 * 2**20   # fits the static scratch (SGEMM_NOALLOC_SCRATCH_BYTES)
    stream = torch.cuda.current_stream().cuda_stream
    outs = [torch.full((M, N), float("nan"), device="cuda") for _ in range(2)]
    # first call: sets up the scratch address for this device
    assert lib.sgemm_run_noalloc(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N,
                                 outs[0].data_ptr(), N, stream) == 0, lib.sgemm_last_error()
    torch.cuda.synchronize()
    for out in outs:
        out.fill_(float("nan"))
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for out in outs:   # two calls in a row on the same stream
        rc = lib.sgemm_run_noalloc(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N,
                                   out.data_ptr(), N, stream)
        assert rc == 0, lib.sgemm_last_error()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before, "device memory changed"
    for out in outs:
        err = float((out - ref).abs().max())
        assert np.isfinite(err) and err <= tolerance(A, B), (case, err)


def test_noalloc_rejects_bad_arguments_like_sgemm_run(cuda):
    lib = load()
    P = 0x10000
    assert lib.sgemm_run_noalloc(-1, 4, 4, P, 4, P, 4, P * 8, 4, None) == -1
    assert lib.sgemm_run_noalloc(4, 4, 8, P, 7, P, 4, P * 8, 4, None) == -1
