"""GPU: the C ABI used from a plain C program, as the README's quick start does: handles, device
buffers from the CUDA runtime, gemm_run in three modes, gemm_query_status, gemm_destroy.

The check needs no oracle: small integer operands (|a|, |b| <= 3, exact in bf16) give integer
products whose fp32 sums are exact at K = 320, so C = A.B + 2.C_in must match the program's own
integer arithmetic bit for bit.
"""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime.h>
#include "densegemm.h"

static uint16_t bf16_of_int(int v) {            /* small integers are exact in bf16 */
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static int run(int mode_id, int M, int N, int K) {
    gemm_options_t o;
    gemm_options_default(&o);                    /* A row-major, B column-major, C row-major */
    o.out_type = GEMM_OUT_F32;
    if (mode_id == 1) { o.mode = GEMM_MODE_MCAST; o.mcast_b = 1; o.cluster_m = 2; }
    if (mode_id == 2) { o.cta_group = 0; o.cluster_m = 2; }
    uint16_t *A = malloc((size_t)M * K * 2), *B = malloc((size_t)N * K * 2);
    float *C = malloc((size_t)M * N * 4), *R = malloc((size_t)M * N * 4);
    int *Ai = malloc((size_t)M * K * sizeof(int)), *Bi = malloc((size_t)N * K * sizeof(int));
    for (int i = 0; i < M * K; ++i) { Ai[i] = (int)((i * 37 + 11) % 7) - 3; A[i] = bf16_of_int(Ai[i]); }
    for (int i = 0; i < N * K; ++i) { Bi[i] = (int)((i * 53 + 5) % 7) - 3; B[i] = bf16_of_int(Bi[i]); }
    for (int i = 0; i < M * N; ++i) C[i] = (float)((i % 5) - 2);
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            long s = 0;
            for (int k = 0; k < K; ++k) s += (long)Ai[(size_t)m * K + k] * Bi[(size_t)n * K + k];  /* B col-major */
            R[(size_t)m * N + n] = (float)s + 2.0f * C[(size_t)m * N + n];
        }
    void *dA, *dB, *dC;
    if (cudaMalloc(&dA, (size_t)M * K * 2) || cudaMalloc(&dB, (size_t)N * K * 2) || cudaMalloc(&dC, (size_t)M * N * 4))
        return 10;
    cudaMemcpy(dA, A, (size_t)M * K * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(dB, B, (size_t)N * K * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(dC, C, (size_t)M * N * 4, cudaMemcpyHostToDevice);
    gemm_handle_t h;
    gemm_status_t s = gemm_create(&h, &o, 0);
    if (s != GEMM_OK) { printf("create: %s\n", gemm_last_error(NULL)); return 11; }
    s = gemm_run(h, M, N, K, dA, K, dB, K, dC, N, 1.0f, 2.0f, NULL);
    if (s == GEMM_OK) s = gemm_query_status(h, NULL);
    if (s != GEMM_OK) { printf("run: %s\n", gemm_last_error(h)); return 12; }
    cudaMemcpy(C, dC, (size_t)M * N * 4, cudaMemcpyDeviceToHost);
    int bad = 0;
    for (int i = 0; i < M * N; ++i) bad += (memcmp(&C[i], &R[i], 4) != 0);
    gemm_destroy(h);
    cudaFree(dA); cudaFree(dB); cudaFree(dC);
    free(A); free(B); free(C); free(R); free(Ai); free(Bi);
    printf("mode %d: %d of %d outputs differ\n", mode_id, bad, M * N);
    return bad ? 13 : 0;
}

int main(void) {
    int rc = 0;
    for (int mode_id = 0; mode_id < 3 && !rc; ++mode_id) rc = run(mode_id, 300, 520, 320);
    return rc;
}
"""


def test_c_program_runs_gemm_through_the_abi(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from dense_gemm_cluster_gb300 import build
    build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    src, exe = tmp_path / "abi_gpu.c", tmp_path / "abi_gpu"
    src.write_text(C_PROGRAM)
    r = subprocess.run([cc, "-std=c99", "-O1", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                        str(src), "-L", build.BUILD_DIR, "-ldensegemm", f"-Wl,-rpath,{build.BUILD_DIR}",
                        "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}",
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.count("0 of 156000 outputs differ") == 3, out.stdout
