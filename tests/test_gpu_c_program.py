"""The boundary from plain C on the GPU: a C99 program built against
include/fp8w.h allocates device memory with cudaMalloc, quantises a weight
and runs the linear layer at M = 1 (the GEMV), 8 (the tensor-core kernel,
a cluster-shared shape) and 96 (the prefill GEMM) through the library, and
compares the codes and scales byte for byte with the oracle's, which the test
writes to a file beforehand; the outputs it writes back are held to the
oracle's within the stated tolerance.  No Python object touches the device
data on the way."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import synthetic
from tests.parity import assert_parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import fp8_weight_only_gb300 as fw  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime.h>
#include "fp8w.h"

static void *slurp(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    void *p = malloc(bytes);
    FILE *f;
    snprintf(path, sizeof path, "%s/%s", dir, name);
    f = fopen(path, "rb");
    if (!f || !p || fread(p, 1, bytes, f) != bytes) { fprintf(stderr, "read %s\n", path); exit(2); }
    fclose(f);
    return p;
}

static void spill(const char *dir, const char *name, const void *p, size_t bytes) {
    char path[4096];
    FILE *f;
    snprintf(path, sizeof path, "%s/%s", dir, name);
    f = fopen(path, "wb");
    if (!f || fwrite(p, 1, bytes, f) != bytes) { fprintf(stderr, "write %s\n", path); exit(2); }
    fclose(f);
}

#define CK(call) do { cudaError_t e_ = (call); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_)); return 3; } } while (0)
#define FW(call) do { fp8w_status s_ = (call); if (s_ != FP8W_OK) { \
    fprintf(stderr, "%s: %s %s\n", #call, fp8w_status_string(s_), fp8w_last_cuda_error()); return 4; } } while (0)

int main(int argc, char **argv) {
    if (argc != 5) { fputs("usage: run DIR N K MMAX\n", stderr); return 2; }
    const char *dir = argv[1];
    const long long n = atoll(argv[2]), k = atoll(argv[3]), mmax = atoll(argv[4]);
    static const long long ms[3] = {1, 8, 96};
    float *w = slurp(dir, "w.bin", (size_t)(n * k) * 4);
    unsigned short *x = slurp(dir, "x.bin", (size_t)(mmax * k) * 2);
    float *bias = slurp(dir, "bias.bin", (size_t)n * 4);
    unsigned char *ref_codes = slurp(dir, "codes_ref.bin", (size_t)(n * k));
    float *ref_scales = slurp(dir, "scales_ref.bin", (size_t)n * 4);
    unsigned char *codes = malloc((size_t)(n * k));
    float *scales = malloc((size_t)n * 4);
    unsigned short *y = malloc((size_t)(mmax * n) * 2);
    float *d_w, *d_scales, *d_bias;
    unsigned char *d_codes;
    unsigned short *d_x, *d_y;
    cudaStream_t st;
    int i;
    if (fp8w_abi_version() != FP8W_ABI_VERSION) { puts("abi version"); return 1; }
    CK(cudaStreamCreate(&st));
    CK(cudaMalloc((void **)&d_w, (size_t)(n * k) * 4));
    CK(cudaMalloc((void **)&d_codes, (size_t)(n * k)));
    CK(cudaMalloc((void **)&d_scales, (size_t)n * 4));
    CK(cudaMalloc((void **)&d_bias, (size_t)n * 4));
    CK(cudaMalloc((void **)&d_x, (size_t)(mmax * k) * 2));
    CK(cudaMalloc((void **)&d_y, (size_t)(mmax * n) * 2));
    CK(cudaMemcpy(d_w, w, (size_t)(n * k) * 4, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_bias, bias, (size_t)n * 4, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_x, x, (size_t)(mmax * k) * 2, cudaMemcpyHostToDevice));
    FW(fp8w_quantize(d_w, n, k, d_codes, d_scales, st));
    CK(cudaStreamSynchronize(st));
    CK(cudaMemcpy(codes, d_codes, (size_t)(n * k), cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(scales, d_scales, (size_t)n * 4, cudaMemcpyDeviceToHost));
    if (memcmp(codes, ref_codes, (size_t)(n * k)) != 0) { puts("codes differ from the oracle"); return 5; }
    if (memcmp(scales, ref_scales, (size_t)n * 4) != 0) { puts("scales differ from the oracle"); return 5; }
    for (i = 0; i < 3; ++i) {
        char name[32];
        FW(fp8w_linear(d_x, FP8W_BF16, ms[i], k, d_codes, d_scales, d_bias, n, d_y, st));
        CK(cudaStreamSynchronize(st));
        CK(cudaMemcpy(y, d_y, (size_t)(ms[i] * n) * 2, cudaMemcpyDeviceToHost));
        snprintf(name, sizeof name, "y%lld.bin", ms[i]);
        spill(dir, name, y, (size_t)(ms[i] * n) * 2);
    }
    if (fp8w_device_error() != 0) { puts("device error"); return 6; }
    printf("ok\n");
    return 0;
}
"""


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_program_quantises_and_runs_the_layer_through_the_header(tmp_path):
    home = _cuda_home()
    libdirs = [d for d in (os.path.join(home, "lib64"), os.path.join(home, "lib")) if os.path.isdir(d)]
    src = tmp_path / "run.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "run"
    libdir = os.path.dirname(fw.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           "-isystem", os.path.join(home, "include"), str(src), "-o", str(exe), "-L", libdir, "-l:libfp8w.so",
           "-Wl,-rpath," + libdir]
    for d in libdirs:
        cmd += ["-L", d, "-Wl,-rpath," + d]
    cmd += ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    c = synthetic.random_case(4242, 96, 1000, 1040)
    codes, scales = oracle.quantize(c["w"])
    for name, arr in (("w.bin", c["w"]), ("x.bin", c["x"]), ("bias.bin", c["bias"]), ("codes_ref.bin", codes),
                      ("scales_ref.bin", scales)):
        np.ascontiguousarray(arr).tofile(str(tmp_path / name))
    r = subprocess.run([str(exe), str(tmp_path), "1000", "1040", "96"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), (r.stdout, r.stderr)
    for m in (1, 8, 96):
        y = np.fromfile(str(tmp_path / ("y%d.bin" % m)), dtype=np.uint16).reshape(m, 1000)
        ref = oracle.linear(c["x"][:m], oracle.ACT_BF16, codes, scales, c["bias"], threads=oracle.host_cores())
        assert_parity(y, ref, oracle.ACT_BF16, "C program m=%d" % m)
