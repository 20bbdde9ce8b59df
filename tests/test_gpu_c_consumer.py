"""The C ABI from a plain C program on the GPU: no Python between the caller
and the library.  The program (C99, built here with the host C compiler
against include/zero1.h, libzero1.so and the CUDA runtime) allocates device
buffers with cudaMalloc, runs two fused steps through
zero1_reduce_scatter_adamw_allgather on its own stream, checks an error path,
and writes the outputs to a file; the test compares them with the oracle bit
for bit."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from zero_sharded_mixed_zero1_gb300 import build as zbuild
from gpu_helpers import assert_bf16_bits, assert_f32_bits

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime.h>
#include "zero1.h"

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 2; } } while (0)

static int rd(FILE *f, void *p, size_t n) { return fread(p, 1, n, f) == n ? 0 : 1; }

int main(int argc, char **argv)
{
    if (argc != 3) return 1;
    FILE *in = fopen(argv[1], "rb");
    if (!in) return 1;
    int64_t hdr[3];
    if (rd(in, hdr, sizeof hdr)) return 1;
    const int64_t n = hdr[0];
    const int32_t M = (int32_t)hdr[1], align = (int32_t)hdr[2];
    zero1_plan_t plan;
    if (zero1_plan(n, M, align, NULL, 0, &plan) != ZERO1_OK) return 3;
    const int64_t P = plan.padded_n;
    uint16_t *g = malloc(sizeof(uint16_t) * (size_t)(2 * M * n));
    float *state = malloc(sizeof(float) * (size_t)(3 * P));
    uint16_t *params = malloc(sizeof(uint16_t) * (size_t)n);
    if (!g || !state || !params) return 1;
    if (rd(in, g, sizeof(uint16_t) * (size_t)(2 * M * n)) || rd(in, state, sizeof(float) * (size_t)(3 * P))) return 1;
    fclose(in);

    uint16_t *dg; float *ds; uint16_t *dp; uint32_t *dflag;
    CK(cudaMalloc((void **)&dg, sizeof(uint16_t) * (size_t)(2 * M * n)));
    CK(cudaMalloc((void **)&ds, sizeof(float) * (size_t)(3 * P)));
    CK(cudaMalloc((void **)&dp, sizeof(uint16_t) * (size_t)n));
    CK(cudaMalloc((void **)&dflag, sizeof(uint32_t)));
    CK(cudaMemcpy(dg, g, sizeof(uint16_t) * (size_t)(2 * M * n), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(ds, state, sizeof(float) * (size_t)(3 * P), cudaMemcpyHostToDevice));
    CK(cudaMemset(dflag, 0, sizeof(uint32_t)));
    cudaStream_t st;
    CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));

    const void *grads[64];
    for (int step = 1; step <= 2; ++step) {
        for (int r = 0; r < M; ++r) grads[r] = dg + (size_t)((step - 1) * M + r) * (size_t)n;
        zero1_adamw_t hp = {1e-3f, 0.9f, 0.95f, 1e-8f, 0.1f, 1.0f, 64, step};
        int rc = zero1_reduce_scatter_adamw_allgather(&plan, 0, M, grads, ds, ds + P, ds + 2 * P, dp, &hp, dflag, 0,
                                                      (zero1_stream_t)st);
        if (rc != ZERO1_OK) { fprintf(stderr, "step %d: %s\n", step, zero1_last_error()); return 4; }
    }
    /* an error path: a misaligned master pointer is refused before any launch */
    zero1_adamw_t hp = {1e-3f, 0.9f, 0.95f, 1e-8f, 0.1f, 1.0f, 64, 3};
    int bad = zero1_reduce_scatter_adamw_allgather(&plan, 0, M, grads, (float *)((char *)ds + 2), ds + P, ds + 2 * P,
                                                   dp, &hp, dflag, 0, (zero1_stream_t)st);
    if (bad != ZERO1_EALIGN || strstr(zero1_last_error(), "aligned") == NULL) return 5;
    CK(cudaStreamSynchronize(st));
    uint32_t flag = 7;
    CK(cudaMemcpy(state, ds, sizeof(float) * (size_t)(3 * P), cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(params, dp, sizeof(uint16_t) * (size_t)n, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&flag, dflag, sizeof flag, cudaMemcpyDeviceToHost));
    FILE *out = fopen(argv[2], "wb");
    if (!out) return 1;
    fwrite(state, sizeof(float), (size_t)(3 * P), out);
    fwrite(params, sizeof(uint16_t), (size_t)n, out);
    fwrite(&flag, sizeof flag, 1, out);
    fclose(out);
    cudaFree(dg); cudaFree(ds); cudaFree(dp); cudaFree(dflag);
    cudaStreamDestroy(st);
    free(g); free(state); free(params);
    return 0;
}
"""


@pytest.mark.parametrize("n,M,align", [(100_003, 8, 128), (40_961, 3, 1)])
def test_c_program_runs_the_step_through_the_abi(cuda_device, tmp_path, n, M, align):
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(zbuild.LIB)
    subprocess.run(["gcc", "-std=c99", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda_home, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-l:libzero1.so", f"-Wl,-rpath,{libdir}",
                    "-L", os.path.join(cuda_home, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(cuda_home, 'lib64')}"],
                   check=True)
    P, s = oracle.plan(n, M, align)
    rng = np.random.default_rng(n + M)
    grads = [[oracle.f32_to_bf16((rng.standard_normal(n) * 1e-2).astype(np.float32)) for _ in range(M)]
             for _ in range(2)]
    master = np.zeros(P, np.float32)
    master[:n] = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = np.zeros(P, np.float32)
    v = np.zeros(P, np.float32)
    inp = tmp_path / "in.bin"
    with open(inp, "wb") as f:
        f.write(np.array([n, M, align], np.int64).tobytes())
        for step in grads:
            for g in step:
                f.write(g.tobytes())
        for a in (master, m, v):
            f.write(a.tobytes())
    out = tmp_path / "out.bin"
    r = subprocess.run([str(exe), str(inp), str(out)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stderr)
    raw = open(out, "rb").read()
    got_state = np.frombuffer(raw[:12 * P], np.float32).reshape(3, P)
    got_params = np.frombuffer(raw[12 * P:12 * P + 2 * n], np.uint16)
    got_flag = int(np.frombuffer(raw[12 * P + 2 * n:], np.uint32)[0])
    # the oracle, shard by shard, two steps
    params = np.zeros(n, np.uint16)
    for t, step in enumerate(grads, start=1):
        hp = oracle.AdamW(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, loss_scale=1.0,
                          global_batch=64, step=t)
        for i in range(M):
            lo, hi = i * s, (i + 1) * s
            nv = max(0, min(hi, n) - lo)
            w_, m_, v_ = master[lo:hi].copy(), m[lo:hi].copy(), v[lo:hi].copy()
            p_ = np.zeros(nv, np.uint16)
            oracle.zero1_step([np.ascontiguousarray(g[lo:lo + nv]) for g in step], nv, w_, m_, v_, p_, hp)
            master[lo:hi], m[lo:hi], v[lo:hi] = w_, m_, v_
            params[lo:lo + nv] = p_
    for got, want, what in zip(got_state, (master, m, v), ("master", "m", "v")):
        assert_f32_bits(got, want, f"C program: {what}")
    assert_bf16_bits(got_params, params, "C program: params")
    assert got_flag == 0
