"""Cluster split on the GPU: the CTAs that share one tile's K range form a
thread-block cluster and sum their partial tiles through distributed shared
memory, in rank (= k) order, inside the product launch.

Every cp.async tile-table entry runs with clusters of 2, 4 and 8 CTAs on ragged
shapes against the fp64 oracle (max |C - C_ref| <= 1e-6 K max|A| max|B|), with a
canary around C; exact cases (small integers) must match bit for bit; and the
result must not change from run to run.
"""
import ctypes

import numpy as np
import pytest

from dense_fp32_gemm_09_gb300 import kernel_table, load, sgemm, sgemm_query_config
from dense_fp32_gemm_09_gb300.workloads import random_pair, small_int_pair

from test_gpu_parity import canaried, check_canary, padded, tolerance
from test_gpu_scaled import tol

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1, 64), (3, 5, 70), (31, 33, 129), (65, 63, 257), (127, 129, 300),
          (257, 383, 1000), (300, 260, 129), (1000, 70, 517)]


def _cluster_entries():
    try:
        return [k["name"] for k in kernel_table() if not k["name"].endswith("_tma")]
    except Exception:   # library not built: the fixture reports it
        return []


def _planned_cluster(M, N, K, kid, schedule):
    from dense_fp32_gemm_09_gb300._abi import SgemmConfig
    cfg = SgemmConfig()
    assert load().sgemm_schedule_check(M, N, K, kid, 152, 1, schedule, ctypes.byref(cfg)) == 0
    return cfg.cluster


@pytest.mark.parametrize("kname", _cluster_entries())
@pytest.mark.parametrize("S", [2, 4, 8])
def test_cluster_split_each_kernel(cuda, oracle_mod, monkeypatch, kname, S):
    torch = cuda
    monkeypatch.setenv("SGEMM_CLUSTER", str(S))
    kid = {k["name"]: k for k in kernel_table()}[kname]["kernel_id"]
    v1 = kname.endswith("_v1")
    used = 0
    for (M, N, K) in SHAPES:
        A, B = random_pair(M, N, K, seed=M * 5 + N * 11 + K + S)
        if v1:   # odd leading dimensions, bases off 16 bytes
            dA = padded(torch, A, 1, offset=1)
            dB = padded(torch, B, 3, offset=3)
            buf, C = canaried(torch, M, N, ldc_pad=1)
        else:
            dA = padded(torch, A, (-K) % 4 + 4)
            dB = padded(torch, B, (-N) % 4 + 4)
            buf, C = canaried(torch, M, N, ldc_pad=(-N) % 4 + 4)
        sgemm(dA, dB, out=C, kernel_id=kid, schedule=3)
        torch.cuda.synchronize()
        check_canary(buf, M, N)
        ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
        err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
        assert err <= tolerance(A, B), (kname, S, (M, N, K), err)
        # the plan: clusters of the largest power of two up to S with a slice per CTA
        KT = -(-K // kernel_table()[kid]["bk"])
        cap = 1
        while 2 * cap <= min(S, KT):
            cap *= 2
        planned = _planned_cluster(M, N, K, kid, 3)
        assert planned == (cap if cap >= 2 else 0), (kname, S, (M, N, K), planned)
        used += planned == S
    assert used >= 1, (kname, S)


@pytest.mark.parametrize("S", [2, 4, 8])
def test_cluster_split_exact_and_deterministic(cuda, oracle_mod, monkeypatch, S):
    """Small-integer operands: every partial sum is exact in fp32, so the cluster
    sum must equal the oracle bit for bit; two runs must agree bit for bit."""
    torch = cuda
    monkeypatch.setenv("SGEMM_CLUSTER", str(S))
    for (M, N, K) in [(256, 256, 256), (301, 205, 999), (64, 64, 4096)]:
        A, B = small_int_pair(M, N, K, seed=S + K)
        dA, dB = A.cuda(), B.cuda()
        C1 = sgemm(dA, dB, schedule=3)
        C2 = sgemm(dA, dB, schedule=3)
        torch.cuda.synchronize()
        ref = oracle_mod.gemm_f64(A.numpy(), B.numpy()).astype(np.float32)
        assert np.array_equal(C1.cpu().numpy(), ref), (S, M, N, K)
        assert torch.equal(C1, C2)


@pytest.mark.parametrize("alpha,beta", [(1.5, 0.0), (-0.5, 2.0), (1.0, 1.0)])
def test_cluster_split_scaled(cuda, oracle_mod, monkeypatch, alpha, beta):
    """C = alpha A.B + beta C through the cluster sum's epilogue."""
    torch = cuda
    monkeypatch.setenv("SGEMM_CLUSTER", "4")
    M, N, K = 200, 300, 777
    A, B = random_pair(M, N, K, seed=7)
    C0 = torch.rand(M, N, generator=torch.Generator().manual_seed(3)) - 0.5
    dC = C0.cuda()
    sgemm(A.cuda(), B.cuda(), out=dC, alpha=alpha, beta=beta, schedule=3)
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64_ex(alpha, A.numpy(), B.numpy(), beta, C0.numpy())
    assert np.max(np.abs(dC.cpu().numpy().astype(np.float64) - ref)) <= tol(alpha, beta, A, B,
                                                                             C0)


def test_small_cube_takes_one_launch(cuda, oracle_mod):
    """256^3 (the bench's smallest workload): the library splits its 32 x 32 tiles
    over clusters and needs neither a workspace nor a second launch."""
    torch = cuda
    from dense_fp32_gemm_09_gb300 import sgemm_workspace_size
    cfg = sgemm_query_config(256, 256, 256)
    assert cfg["cluster"] >= 2 and cfg["grid"] == cfg["tiles"] * cfg["cluster"]
    assert sgemm_workspace_size(256, 256, 256, 256, 256, 256) == 0
    lib = load()
    A, B = random_pair(256, 256, 256, seed=0)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(256, 256, device="cuda")
    torch.cuda.synchronize()
    n0 = lib.sgemm_launch_count()
    sgemm(dA, dB, out=C)
    assert lib.sgemm_launch_count() - n0 == 1
    torch.cuda.synchronize()
    ref = oracle_mod.gemm_f64(A.numpy(), B.numpy())
    assert np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref)) <= tolerance(A, B)


def test_chained_cluster_products_see_their_inputs_complete(cuda, oracle_mod):
    """Products on one stream, each reading the C of the one before, alternating
    cluster splits (one launch, programmatic dependent of the previous kernel) with
    a stream-K product (main kernel + reduction): every stage must see its inputs
    complete."""
    torch = cuda
    g = torch.Generator().manual_seed(22)

    def u(r, c):
        return ((torch.rand(r, c, generator=g) - 0.5) * 0.2).cuda()

    X0, B1, B2, B3, B4 = u(256, 256), u(256, 256), u(256, 768), u(768, 4096), u(4096, 1024)
    shapes = [(256, 256, 256), (256, 768, 256), (256, 4096, 768)]
    plans = [sgemm_query_config(*s) for s in shapes]
    assert all(plans[i]["cluster"] >= 2 for i in (0, 1)), plans
    assert plans[2]["cluster"] == 0 and plans[2]["sk_tiles"] > 0, plans[2]
    lib = load()
    C1 = sgemm(X0, B1)
    C2 = sgemm(C1, B2)
    C3 = sgemm(C2, B3)
    n0 = lib.sgemm_launch_count()
    C4 = sgemm(C3, B4, schedule=3)   # a cluster split (one launch) right after stream-K
    assert lib.sgemm_launch_count() - n0 == 1
    torch.cuda.synchronize()
    for A, B, C in ((X0, B1, C1), (C1, B2, C2), (C2, B3, C3), (C3, B4, C4)):
        a, b = A.cpu(), B.cpu()
        ref = oracle_mod.gemm_f64(a.numpy(), b.numpy())
        err = np.max(np.abs(C.cpu().numpy().astype(np.float64) - ref))
        assert err <= tolerance(a, b), (tuple(A.shape), tuple(B.shape), err)
