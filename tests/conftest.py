import os
import sys

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if REPO not in sys.path:
    sys.path.insert(0, REPO)

GOLDEN = os.path.join(REPO, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Key -> list of whitespace-separated fields, '#' lines skipped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def lib():
    """The CUDA library (built here with nvcc if needed).  Loading needs no GPU."""
    from dense_fp32_gemm_09_gb300 import build, load
    build.build()
    return load()


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_09_gb300 import build
    build.build()
    return torch


def padded_device(torch, X, pad, offset=0):
    """X copied into a device buffer with leading dimension cols + pad, starting
    `offset` elements into the buffer (offset 1 breaks 16-byte alignment)."""
    rows, cols = X.shape
    ld = cols + pad
    flat = torch.full((offset + rows * ld + 8,), float("nan"), dtype=torch.float32,
                      device="cuda")
    view = flat[offset:offset + rows * ld].view(rows, ld)[:, :cols]
    view.copy_(X)
    return view
