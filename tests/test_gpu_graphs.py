"""The product inside a captured CUDA graph: replays recompute C from whatever
the captured input buffers hold.  Captured launches include the stream-K
reduction (a programmatic dependent launch), cluster-split launches (a cluster
dimension launch attribute) and, for the TMA entry, tensor maps passed by value;
the library's workspace for the capturing stream is allocated by a warm-up call
before capture, as the header asks."""
import numpy as np
import pytest

from dense_fp32_gemm_09_gb300 import check, load, sgemm, sgemm_query_config, sgemm_run_noalloc
from dense_fp32_gemm_09_gb300.workloads import random_pair

pytestmark = pytest.mark.gpu


def tol(A, B):
    return 1e-6 * A.shape[1] * float(A.abs().max()) * float(B.abs().max())


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (2048, 1536, 4096), (3001, 2047, 1999),
                                   (256, 256, 256), (768, 768, 768)])
def test_graph_replay_recomputes(cuda, oracle_mod, M, N, K):
    """1024^3 and up take stream-K (reduction launch); 256^3 and 768^3 a cluster split
    (cluster launch attribute, one launch)."""
    torch = cuda
    A1, B = random_pair(M, N, K, seed=30)
    A2, _ = random_pair(M, N, K, seed=31)
    dA, dB = A1.cuda(), B.cuda()
    dC = torch.empty(M, N, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sgemm(dA, dB, out=dC)                      # warm-up: workspace for stream s
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sgemm(dA, dB, out=dC)
    for A in (A2, A1):
        dA.copy_(A)
        dC.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
        assert np.max(np.abs(dC.cpu().numpy() - ref)) <= tol(A, B)
    cfg = sgemm_query_config(M, N, K)
    assert cfg["grid"] > 0


def test_graph_of_noalloc_entry(cuda, oracle_mod):
    torch = cuda
    M, N, K = 1000, 700, 900
    A, B = random_pair(M, N, K, seed=32)
    dA, dB = A.cuda(), B.cuda()
    dC = torch.empty(M, N, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                     # first call looks up the scratch address
        check(sgemm_run_noalloc(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N,
                                stream=s), "noalloc")
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        check(sgemm_run_noalloc(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N,
                                stream=s), "noalloc")
    dC.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    assert np.max(np.abs(dC.cpu().numpy() - ref)) <= tol(A, B)
    assert load().sgemm_device_status() == 0
