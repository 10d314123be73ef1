"""The C ABI driven by a plain C11 program, with no Python or torch in the
loop: device buffers from cudaMalloc, a stream from cudaStreamCreate, every
schedule x protocol through ar_allreduce, and AUTO through ar_allreduce_n
captured in a CUDA graph and replayed, then ar_allreduce_host on buffers
from cudaMallocHost.  The program reads its inputs from a file (drawn here by
the seeded generator) and writes every path's outputs to a file, which this
test compares with the oracle bit for bit."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from all_reduce_reduction_gb300 import build as cuda_build
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include "ar.h"
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>

#define CHECK_CUDA(x)                                                        \
    do {                                                                     \
        cudaError_t e_ = (x);                                                \
        if (e_ != cudaSuccess) {                                             \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));         \
            return 2;                                                        \
        }                                                                    \
    } while (0)
#define CHECK_AR(x)                                                          \
    do {                                                                     \
        int c_ = (x);                                                        \
        if (c_ != AR_OK) {                                                   \
            fprintf(stderr, "%s: %s\n", #x, ar_strerror(c_));                \
            return 3;                                                        \
        }                                                                    \
    } while (0)

/* usage: prog R n dtype inputs.bin outputs.bin */
int main(int argc, char **argv) {
    if (argc != 6)
        return 1;
    const int R = atoi(argv[1]);
    const size_t n = (size_t)strtoull(argv[2], NULL, 10);
    const int dtype = atoi(argv[3]);
    const size_t bytes = n * (dtype == AR_FP32 ? 4u : 2u);
    unsigned char *host = malloc((size_t)R * bytes);
    FILE *f = fopen(argv[4], "rb");
    if (!host || !f || fread(host, 1, (size_t)R * bytes, f) != (size_t)R * bytes)
        return 1;
    fclose(f);

    void *inw[AR_MAX_RANKS] = {0};
    const void *in[AR_MAX_RANKS] = {0};
    void *out[AR_MAX_RANKS] = {0};
    for (int r = 0; r < R; ++r) {
        CHECK_CUDA(cudaMalloc(&inw[r], bytes));
        CHECK_CUDA(cudaMalloc(&out[r], bytes));
        CHECK_CUDA(cudaMemcpy(inw[r], host + (size_t)r * bytes, bytes, cudaMemcpyHostToDevice));
        in[r] = inw[r];
    }
    ar_handle_t h = NULL;
    cudaStream_t s;
    CHECK_AR(ar_create(R, n, dtype, &h));
    CHECK_CUDA(cudaStreamCreate(&s));
    FILE *fo = fopen(argv[5], "wb");
    if (!fo)
        return 1;

    const int paths[4][2] = {{AR_ONE_SHOT, AR_HB}, {AR_TWO_SHOT, AR_HB},
                             {AR_ONE_SHOT, AR_LL}, {AR_TWO_SHOT, AR_LL}};
    for (int p = 0; p < 5; ++p) {
        for (int r = 0; r < R; ++r)
            CHECK_CUDA(cudaMemsetAsync(out[r], 0xFF, bytes, s));
        if (p < 4) {
            CHECK_AR(ar_allreduce(h, in, out, paths[p][0], paths[p][1], s));
        } else {
            /* AUTO, captured once and replayed twice */
            cudaGraph_t g;
            cudaGraphExec_t ge;
            CHECK_CUDA(cudaStreamBeginCapture(s, cudaStreamCaptureModeGlobal));
            CHECK_AR(ar_allreduce_n(h, in, out, n, AR_ALGO_AUTO, AR_PROTO_AUTO, s));
            CHECK_CUDA(cudaStreamEndCapture(s, &g));
            CHECK_CUDA(cudaGraphInstantiate(&ge, g, 0));
            CHECK_CUDA(cudaGraphLaunch(ge, s));
            CHECK_CUDA(cudaGraphLaunch(ge, s));
            CHECK_CUDA(cudaStreamSynchronize(s));
            CHECK_CUDA(cudaGraphExecDestroy(ge));
            CHECK_CUDA(cudaGraphDestroy(g));
        }
        CHECK_AR(ar_status(h, s));
        for (int r = 0; r < R; ++r)
            CHECK_CUDA(cudaMemcpy(host + (size_t)r * bytes, out[r], bytes, cudaMemcpyDeviceToHost));
        if (fwrite(host, 1, (size_t)R * bytes, fo) != (size_t)R * bytes)
            return 1;
    }
    /* page-locked host buffers, read and written by the kernels in place */
    void *hin[AR_MAX_RANKS] = {0};
    void *hout[AR_MAX_RANKS] = {0};
    FILE *fi = fopen(argv[4], "rb");
    if (!fi)
        return 1;
    for (int r = 0; r < R; ++r) {
        CHECK_CUDA(cudaMallocHost(&hin[r], bytes));
        CHECK_CUDA(cudaMallocHost(&hout[r], bytes));
        if (fread(hin[r], 1, bytes, fi) != bytes)
            return 1;
        in[r] = hin[r];
    }
    fclose(fi);
    CHECK_AR(ar_allreduce_host(h, in, hout, n, AR_ALGO_AUTO, AR_PROTO_AUTO, s));
    CHECK_AR(ar_status(h, s));
    for (int r = 0; r < R; ++r) {
        if (fwrite(hout[r], 1, bytes, fo) != bytes)
            return 1;
        CHECK_CUDA(cudaFreeHost(hin[r]));
        CHECK_CUDA(cudaFreeHost(hout[r]));
    }
    fclose(fo);
    CHECK_AR(ar_destroy(h));
    CHECK_CUDA(cudaStreamDestroy(s));
    for (int r = 0; r < R; ++r) {
        CHECK_CUDA(cudaFree(inw[r]));
        CHECK_CUDA(cudaFree(out[r]));
    }
    free(host);
    return 0;
}
"""


def _cuda_home() -> str:
    nv = cuda_build.nvcc()
    if os.path.isabs(nv):
        return os.path.dirname(os.path.dirname(nv))
    found = shutil.which(nv)
    return os.path.dirname(os.path.dirname(found)) if found else "/usr/local/cuda"


@pytest.fixture(scope="module")
def c_program(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    lib = cuda_build.build()
    d = tmp_path_factory.mktemp("cprog")
    src = d / "allreduce.c"
    src.write_text(C_PROGRAM)
    exe = d / "allreduce"
    cuda = _cuda_home()
    libdirs = [os.path.dirname(lib), os.path.join(cuda, "lib64")]
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(cuda, "include"),
           str(src), "-o", str(exe)]
    for ld in libdirs:
        cmd += ["-L" + ld, "-Wl,-rpath," + ld]
    cmd += ["-lar_gb300", "-lcudart"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("R,n", [(5, 4099), (8, 70001)])
def test_c_program_every_path_bit_exact(c_program, tmp_path, dtype, R, n):
    need_gpu()
    cpu = wl.make_inputs(95, R, n, dtype, "loguniform")
    bits = [wl.bits(t) for t in cpu]
    inp = tmp_path / "in.bin"
    outp = tmp_path / "out.bin"
    np.concatenate(bits).tofile(inp)
    res = subprocess.run([str(c_program), str(R), str(n), str(wl.DTYPE_CODE[dtype]), str(inp),
                          str(outp)], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    want = oracle.allreduce(bits, wl.DTYPE_CODE[dtype])[0]
    u = np.uint32 if dtype == "fp32" else np.uint16
    got = np.fromfile(outp, dtype=u).reshape(6, R, n)
    names = ["one_shot_hb", "two_shot_hb", "one_shot_ll", "two_shot_ll", "auto_graph",
             "host_buffers"]
    for p in range(6):
        for r in range(R):
            bad = np.nonzero(got[p, r] != np.ascontiguousarray(want).view(u))[0]
            assert bad.size == 0, "%s rank %d: %d elements differ, first at %d" % (
                names[p], r, bad.size, bad[0])
