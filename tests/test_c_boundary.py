"""The boundary is plain C: a C99 program includes include/fp8w.h under
-Wall -Werror -pedantic, links libfp8w.so and calls entry points that need
no GPU (version, status strings, argument checks that fail on the host)."""
import os
import shutil
import subprocess

import pytest

import fp8_weight_only_gb300 as fw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fp8w.h"

int main(void) {
    float scales[4];
    unsigned char codes[64];
    int fails = 0;
    if (fp8w_abi_version() != FP8W_ABI_VERSION) { puts("abi version"); ++fails; }
    if (strcmp(fp8w_status_string(99), "unknown status") != 0) { puts("status string"); ++fails; }
    /* a NULL weight is refused before any CUDA call */
    if (fp8w_quantize(NULL, 4, 16, codes, scales, NULL) != FP8W_ERR_NULL) { puts("null check"); ++fails; }
    /* k % 16 != 0 is refused before any CUDA call (host pointers never reach a kernel) */
    if (fp8w_linear(codes, FP8W_BF16, 1, 24, codes, scales, NULL, 4, codes, NULL) != FP8W_ERR_SHAPE) {
        puts("shape check"); ++fails;
    }
    /* an activation dtype other than bf16 / fp16: refused on the host */
    if (fp8w_linear_mx(codes, FP8W_F32, 2, 128, codes, codes, NULL, 4, codes, NULL) != FP8W_ERR_DTYPE) {
        puts("mx check"); ++fails;
    }
    printf("%s\n", fails ? "FAIL" : "ok");
    return fails;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_header_is_c99_and_the_library_links(tmp_path):
    lib = fw.LIB_PATH
    if not os.path.exists(lib):
        pytest.skip("libfp8w.so not built")
    src = tmp_path / "boundary.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "boundary"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", libdir, "-l:libfp8w.so", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), (r.stdout, r.stderr)
