"""sgemm_shutdown, then the library again, in a fresh process.

Shutdown frees the library-owned workspaces, destroys the host-buffer entry's
streams and events and forgets the per-device state (kernel attributes set in the
device's context, the allocation-free entry's scratch addresses).  Every entry
point that uses one of those is run, the library is shut down (twice: it must be
idempotent), and everything is run again: the second results must equal the
first bit for bit, and both must match the fp64 oracle."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

# (name, M, N, K): stream-K with the library workspace, a cluster split, the
# 3xTF32 path (its own workspace and kernel attributes), the host-buffer entry
# (library streams and events) and the allocation-free entry (static scratch).
CASES = [("run", 1024, 1024, 1024), ("cluster", 256, 256, 256), ("tf32x3", 512, 384, 640),
         ("host", 768, 640, 512), ("noalloc", 1024, 1024, 1024)]

_CHILD = r"""
import sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch
from dense_fp32_gemm_09_gb300 import check, load, sgemm_query_config
from dense_fp32_gemm_09_gb300.workloads import random_pair
lib = load()
cases = eval(sys.argv[3])
stream = torch.cuda.current_stream().cuda_stream

def run_all():
    outs = []
    for i, (name, M, N, K) in enumerate(cases):
        A, B = random_pair(M, N, K, seed=70 + i)
        dA, dB = A.cuda(), B.cuda()
        dC = torch.full((M, N), float("nan"), device="cuda")
        args = (M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N)
        if name in ("run", "cluster"):
            st = lib.sgemm_run(*args, stream)
        elif name == "tf32x3":
            st = lib.sgemm_tf32x3_run(*args, stream)
        elif name == "noalloc":
            st = lib.sgemm_run_noalloc(*args, stream)
        else:
            hA, hB = A.pin_memory(), B.pin_memory()
            hC = torch.full((M, N), float("nan")).pin_memory()
            st = lib.sgemm_run_host(M, N, K, hA.data_ptr(), K, hB.data_ptr(), N, hC.data_ptr(),
                                    N, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), stream)
            torch.cuda.synchronize()
            dC.copy_(hC)
        check(st, name)
        torch.cuda.synchronize()
        outs.append(dC.cpu().numpy())
    return outs

assert sgemm_query_config(1024, 1024, 1024)["sk_tiles"] > 0
assert sgemm_query_config(256, 256, 256)["cluster"] > 1
first = run_all()
check(lib.sgemm_shutdown(), "shutdown")
check(lib.sgemm_shutdown(), "second shutdown")
second = run_all()
np.savez(sys.argv[2], **{f"first{i}": a for i, a in enumerate(first)},
         **{f"second{i}": a for i, a in enumerate(second)})
print("ok")
"""


def test_library_works_again_after_shutdown(cuda, oracle_mod, tmp_path):
    from dense_fp32_gemm_09_gb300.workloads import random_pair
    repo = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    path = str(tmp_path / "out.npz")
    out = subprocess.run([sys.executable, "-c", _CHILD, repo, path, repr(CASES)],
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    res = np.load(path)
    for i, (name, M, N, K) in enumerate(CASES):
        A, B = random_pair(M, N, K, seed=70 + i)
        exact = oracle_mod.gemm_f64(A.numpy(), B.numpy())
        scale = 1e-5 if name == "tf32x3" else 1e-6
        tol = scale * K * float(A.abs().max()) * float(B.abs().max())
        first, second = res[f"first{i}"], res[f"second{i}"]
        assert np.array_equal(first, second), name
        err = float(np.max(np.abs(first.astype(np.float64) - exact)))
        assert np.isfinite(err) and err <= tol, (name, err, tol)
