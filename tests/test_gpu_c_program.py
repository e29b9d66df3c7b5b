"""The C ABI from a plain C program on the GPU: a C11 program that includes
cuda_runtime.h and sar.h allocates 4 ranks of fp32 with the CUDA runtime, runs
the fused rsag allreduce, the LL allreduce with caller packet buffers and
sar_allreduce with SAR_ALGO_LL_ALLPAIR through libsar, and checks every
output element against the in-order binary32 sum it computes itself (exact:
the inputs are multiples of 1/64 below 16 in magnitude)."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "sar.h"

#define N 4
#define COUNT 100003

static int check(float* const* d_out, float* const* h, const char* what) {
    float* got = (float*)malloc(COUNT * sizeof(float));
    int bad = 0;
    for (int j = 0; j < N && !bad; ++j) {
        if (cudaMemcpy(got, d_out[j], COUNT * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
        for (int i = 0; i < COUNT; ++i) {
            float want = h[0][i];
            for (int r = 1; r < N; ++r) want = want + h[r][i];
            if (memcmp(&got[i], &want, sizeof(float)) != 0) {
                printf("%s: out[%d][%d] = %a, want %a\n", what, j, i, got[i], want);
                bad = 1;
                break;
            }
        }
    }
    free(got);
    return bad;
}

int main(void) {
    float* h[N];
    float* d_in[N];
    float* d_out[N];
    void* d_pkt[N];
    const size_t pkt_bytes = sar_ll_packet_bytes(COUNT, SAR_FP32);
    for (int r = 0; r < N; ++r) {
        h[r] = (float*)malloc(COUNT * sizeof(float));
        for (int i = 0; i < COUNT; ++i) h[r][i] = (float)((i * 7 + r * 13) % 1000) / 64.0f - 7.5f;
        if (cudaMalloc((void**)&d_in[r], COUNT * sizeof(float)) != cudaSuccess) return 2;
        if (cudaMalloc((void**)&d_out[r], COUNT * sizeof(float)) != cudaSuccess) return 2;
        if (cudaMalloc(&d_pkt[r], pkt_bytes) != cudaSuccess) return 2;
        if (cudaMemset(d_pkt[r], 0, pkt_bytes) != cudaSuccess) return 2;
        if (cudaMemcpy(d_in[r], h[r], COUNT * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess) return 2;
    }
    const void* in[N];
    void* out[N];
    for (int r = 0; r < N; ++r) {
        in[r] = d_in[r];
        out[r] = d_out[r];
    }
    sar_status st = sar_allreduce(in, out, N, COUNT, SAR_FP32, SAR_ALGO_RSAG, NULL);
    if (st != SAR_OK) {
        printf("sar_allreduce: %s\n", sar_status_string(st));
        return 3;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return 3;
    if (check(d_out, h, "rsag")) return 4;

    int32_t* d_status;
    if (cudaMalloc((void**)&d_status, sizeof(int32_t)) != cudaSuccess) return 2;
    if (cudaMemset(d_status, 0, sizeof(int32_t)) != cudaSuccess) return 2;
    for (int r = 0; r < N; ++r)
        if (cudaMemset(d_out[r], 0, COUNT * sizeof(float)) != cudaSuccess) return 2;
    st = sar_allreduce_ll(in, out, (void* const*)d_pkt, N, COUNT, SAR_FP32, 1, 1u << 20, d_status, NULL);
    if (st != SAR_OK) {
        printf("sar_allreduce_ll: %s\n", sar_status_string(st));
        return 5;
    }
    st = sar_read_device_status(d_status, NULL);
    if (st != SAR_OK) {
        printf("device status: %s\n", sar_status_string(st));
        return 5;
    }
    if (check(d_out, h, "ll")) return 6;

    for (int r = 0; r < N; ++r)
        if (cudaMemset(d_out[r], 0, COUNT * sizeof(float)) != cudaSuccess) return 2;
    st = sar_allreduce(in, out, N, COUNT, SAR_FP32, SAR_ALGO_LL_ALLPAIR, NULL);
    if (st != SAR_OK) {
        printf("sar_allreduce (LL all-pair): %s\n", sar_status_string(st));
        return 7;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return 7;
    if (check(d_out, h, "ll_allpair")) return 8;

    for (int r = 0; r < N; ++r) {
        cudaFree(d_in[r]);
        cudaFree(d_out[r]);
        cudaFree(d_pkt[r]);
        free(h[r]);
    }
    cudaFree(d_status);
    printf("OK\n");
    return 0;
}
"""


def test_c_program_allreduces_on_the_gpu(tmp_path):
    import allreduce_reduction_rank_gb300 as sar
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cuda_lib = next((os.path.join(cuda, d) for d in ("lib64", "lib", "targets/sbsa-linux/lib",
                                                       "targets/x86_64-linux/lib")
                     if os.path.exists(os.path.join(cuda, d, "libcudart.so"))), None)
    if cuda_lib is None:
        pytest.skip("libcudart.so not found")
    src, exe = tmp_path / "c_allreduce.c", tmp_path / "c_allreduce"
    src.write_text(C_PROGRAM)
    libdir = os.path.dirname(sar.LIB_PATH)
    build = subprocess.run([cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
                            "-I", os.path.join(cuda, "include"), "-I", os.path.join(ROOT, "include"), str(src),
                            "-L", libdir, "-lsar", "-L", cuda_lib, "-lcudart",
                            f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cuda_lib}", "-o", str(exe)],
                           capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0 and run.stdout.strip().endswith("OK"), (run.returncode, run.stdout, run.stderr)
