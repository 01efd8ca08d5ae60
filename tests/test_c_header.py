"""The boundary as a C user sees it (no GPU): a C99 program and the same source as
C++17 include include/sgemm.h, link libsgemm_gb300.so and call the entry points
that need no device (tile table, tile choice, schedule check, argument rejection)."""
import os
import shutil
import subprocess

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "sgemm.h"
int main(void) {
    sgemm_config c;
    int n = sgemm_num_kernels();
    if (n <= 0) return 1;
    if (sgemm_kernel_info(0, &c) != SGEMM_OK || c.threads <= 0) return 2;
    if (sgemm_schedule_check(1024, 1024, 1024, 0, 152, 1, 0, &c) != SGEMM_OK) return 3;
    if (sgemm_run(-1, 4, 4, 0, 4, 0, 4, 0, 4, 0) != SGEMM_ERR_INVALID_ARG) return 4;
    if (sgemm_kernel_info(n, &c) != SGEMM_ERR_UNSUPPORTED) return 5;
    int kid = -1, packed = -1;
    if (sgemm_choose_check(4096, 4096, 4096, 4096, 4096, 0, 0, 152, &kid, &packed) != SGEMM_OK ||
        kid < 0 || kid >= n || packed != 0) return 6;
    printf("%s %d\n", sgemm_status_string(SGEMM_OK), n);
    return 0;
}
"""


@pytest.mark.parametrize("compiler,flags", [("gcc", ["-std=c99"]), ("g++", ["-std=c++17", "-x", "c++"])])
def test_header_compiles_links_and_runs(lib, tmp_path, compiler, flags):
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not found")
    from dense_fp32_gemm_09_gb300._abi import library_path
    libdir = os.path.dirname(library_path())
    src = tmp_path / "use.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use"
    r = subprocess.run([compiler, *flags, "-Wall", "-Wextra", "-Werror",
                        "-I", os.path.join(REPO, "include"), str(src), "-L", libdir,
                        "-lsgemm_gb300", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("SGEMM_OK ")
