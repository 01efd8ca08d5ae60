"""Several host threads calling the library at once.

Calls on one stream share that stream's library-owned workspace.  The shapes here
need workspaces of different sizes (stream-K partial tiles, staged misaligned
operands, the 3xTF32 split operands), so calls grow the workspace (free and
re-allocate it) while other threads are between their workspace lookup and
their launch.  Every product must match the oracle and equal, bit for bit, the
same call made alone (the kernels are deterministic); the second case gives each
thread its own stream, so the products also run concurrently on the GPU."""
import ctypes
import threading

import numpy as np
import pytest

from dense_fp32_gemm_09_gb300 import check, load, sgemm_query_config, sgemm_run, \
    sgemm_workspace_size
from dense_fp32_gemm_09_gb300.workloads import random_pair

pytestmark = pytest.mark.gpu

# (M, N, K, path): stream-K plans of several sizes, a misaligned large problem that
# stages its operands in the workspace, and two 3xTF32 calls (split operands).
CALLS = [
    (1024, 1024, 1024, "fp32"),
    (2048, 1536, 4096, "fp32"),
    (4096, 512, 2048, "fp32"),
    (3001, 2047, 1999, "fp32"),
    (1536, 1536, 2048, "tf32x3"),
    (2048, 1024, 1024, "tf32x3"),
]
THREADS, ROUNDS = 4, 3


def tol(A, B, path):
    scale = 1e-6 if path == "fp32" else 1e-5
    return scale * A.shape[1] * float(A.abs().max()) * float(B.abs().max())


def _launch(lib, path, M, N, K, dA, dB, dC, stream):
    if path == "fp32":
        return sgemm_run(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N,
                         stream=stream)
    return lib.sgemm_tf32x3_run(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N,
                                stream)


@pytest.mark.parametrize("shared_stream", [True, False])
def test_threads_growing_one_workspace(cuda, oracle_mod, shared_stream):
    torch = cuda
    lib = load()
    inputs = []
    for i, (M, N, K, path) in enumerate(CALLS):
        A, B = random_pair(M, N, K, seed=60 + i)
        inputs.append((A, B, A.cuda(), B.cuda()))
    # Workspace needs: partial tiles take one sized by the grid (the same for every
    # stream-K plan here), 3xTF32 its split operands, the staged ragged problem its
    # aligned copies as well.  Every thread starts with the call that needs least,
    # so the fresh stream's workspace is grown by the calls that follow.
    needs = []
    for M, N, K, p in CALLS:
        if p == "fp32":
            needs.append(sgemm_workspace_size(M, N, K, K, N, N))
        else:
            out = ctypes.c_size_t(0)
            check(lib.sgemm_tf32x3_workspace_size(M, N, K, ctypes.byref(out)), "ws")
            needs.append(out.value)
    first = int(np.argmin([n if n > 0 else 1 << 62 for n in needs]))
    assert len(set(needs) - {0}) >= 3 and needs[first] < max(needs)
    assert sgemm_query_config(1024, 1024, 1024)["sk_tiles"] > 0

    # Each call alone, on a stream of its own, checked against the oracle.
    solo = []
    s0 = torch.cuda.Stream()
    for (M, N, K, path), (A, B, dA, dB) in zip(CALLS, inputs):
        dC = torch.full((M, N), float("nan"), device="cuda")
        torch.cuda.synchronize()
        check(_launch(lib, path, M, N, K, dA, dB, dC, s0.cuda_stream), path)
        s0.synchronize()
        C = dC.cpu()
        ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
        assert np.max(np.abs(C.numpy() - ref)) <= tol(A, B, path), (M, N, K, path)
        solo.append(C)

    streams = [torch.cuda.Stream() for _ in range(1 if shared_stream else THREADS)]
    outs = {}
    for t in range(THREADS):
        for r in range(ROUNDS):
            for j, (M, N, K, _) in enumerate(CALLS):
                outs[t, r, j] = torch.full((M, N), float("nan"), device="cuda")
    torch.cuda.synchronize()
    errors = []
    barrier = threading.Barrier(THREADS)

    def worker(t):
        try:
            stream = streams[0 if shared_stream else t].cuda_stream
            rest = [j for j in range(len(CALLS)) if j != first]
            order = [first] + [rest[i] for i in np.random.default_rng(t).permutation(len(rest))]
            barrier.wait()
            for r in range(ROUNDS):
                for j in order:
                    M, N, K, path = CALLS[j]
                    _, _, dA, dB = inputs[j]
                    st = _launch(lib, path, M, N, K, dA, dB, outs[t, r, j], stream)
                    if st != 0:
                        errors.append((t, r, j, st))
        except Exception as e:   # surfaced below, in the test's own thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for (t, r, j), dC in outs.items():
        assert torch.equal(dC.cpu(), solo[j]), (t, r, CALLS[j])
