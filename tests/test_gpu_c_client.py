"""A plain C program drives the whole path through the C ABI: it reads a
batch from files, allocates a device workspace with the CUDA runtime and its
result buffer with ep_host_alloc, runs the host-buffer pipeline
(ep_host_pipeline_*) for three steps and writes every step's combined result.
Each must match the CPU oracle's combine of the same batch (within the
whole-path bound, each side with its own gate weights) and equal, bit for
bit, the same batch run through the Python binding."""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import combine_ep_route_topk_gb300 as ep
from combine_ep_route_topk_gb300 import workloads as wl

from _util import bits, np_

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime.h>
#include "ep.h"

static void* read_file(const char* dir, const char* name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    void* h = NULL;
    if (!f || cudaMallocHost(&h, bytes) != cudaSuccess || fread(h, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot read %s\n", path);
        exit(10);
    }
    fclose(f);
    return h;
}

int main(int argc, char** argv) {
    if (argc != 8) return 2;
    const char* dir = argv[1];
    int N = atoi(argv[2]), E = atoi(argv[3]), K = atoi(argv[4]), H = atoi(argv[5]);
    int R = atoi(argv[6]), steps = atoi(argv[7]);
    size_t rows = (size_t)N * K;
    float* logits = (float*)read_file(dir, "logits.bin", (size_t)N * E * 4);
    int* ro = (int*)read_file(dir, "ro.bin", (size_t)(R + 1) * 4);
    void* x = read_file(dir, "x.bin", (size_t)N * H * 2);
    void* y = read_file(dir, "y.bin", rows * H * 2);
    void* out = NULL;  /* the library's huge-page-backed page-locked host memory */
    if (ep_host_alloc((size_t)steps * N * H * 2, &out) != EP_OK) return 11;
    size_t ws_bytes = ep_host_pipeline_workspace_size(N, E, K, H, R, 0, EP_DTYPE_BF16, 2);
    void* ws = NULL;
    if (ws_bytes == 0 || cudaMalloc(&ws, ws_bytes) != cudaSuccess) return 12;
    cudaStream_t s;
    if (cudaStreamCreate(&s) != cudaSuccess) return 13;
    ep_host_pipeline_t* p = NULL;
    ep_status_t st = ep_host_pipeline_create(N, E, K, H, R, 0, EP_DTYPE_BF16, 2, NULL, ws,
                                             ws_bytes, &p);
    if (st != EP_OK) { fprintf(stderr, "create: %s\n", ep_status_string(st)); return 14; }
    for (int i = 0; i < steps; ++i) {
        st = ep_host_pipeline_step(p, logits, ro, x, y, (char*)out + (size_t)i * N * H * 2, s);
        if (st != EP_OK) { fprintf(stderr, "step: %s\n", ep_status_string(st)); return 15; }
    }
    if (ep_host_pipeline_join(p, s) != EP_OK || cudaStreamSynchronize(s) != cudaSuccess)
        return 16;
    if (ep_host_pipeline_destroy(p) != EP_OK) return 17;
    char path[4096];
    snprintf(path, sizeof path, "%s/out.bin", dir);
    FILE* f = fopen(path, "wb");
    if (!f || fwrite(out, 1, (size_t)steps * N * H * 2, f) != (size_t)steps * N * H * 2)
        return 18;
    fclose(f);
    cudaFree(ws);
    if (ep_host_free(out) != EP_OK) return 19;
    printf("ok %llu kernels\n", (unsigned long long)ep_kernel_launch_count());
    return 0;
}
"""


def test_c_program_runs_the_path_through_the_c_abi(tmp_path):
    w = wl.WORKLOADS["lumpy"]
    inp = wl.make_inputs(w, seed=4)
    N, E, K, H, R = inp["N"], w.E, w.K, w.H, w.R
    inp["logits"].numpy().astype(np.float32).tofile(tmp_path / "logits.bin")
    inp["rank_offsets"].numpy().astype(np.int32).tofile(tmp_path / "ro.bin")
    bits(inp["x"]).tofile(tmp_path / "x.bin")
    bits(inp["y"]).tofile(tmp_path / "y.bin")
    src = tmp_path / "client.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "client"
    libdir = os.path.dirname(ep.ep.LIB_PATH)
    subprocess.run(["nvcc", "-cudart", "shared", "-x", "c", str(src), "-o", str(exe),
                    "-I", os.path.join(ROOT, "include"), "-L", libdir, "-lep_gb300",
                    "-Xlinker", f"-rpath={libdir}"], check=True)
    steps = 3
    r = subprocess.run([str(exe), str(tmp_path), str(N), str(E), str(K), str(H), str(R),
                        str(steps)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok")
    got = np.fromfile(tmp_path / "out.bin", np.uint16).reshape(steps, N, H)

    # the same batch through the Python binding (same kernels: bit for bit)
    idx, wt = ep.ep_route_topk(inp["logits"].cuda(), K)
    lay = ep.ep_dispatch_layout(idx, inp["rank_offsets"].cuda(), E)
    comb = ep.ep_combine(inp["y"].cuda(), idx, wt, lay.pos, lay.expert_offsets, E)
    ref = bits(comb)
    for i in range(steps):
        np.testing.assert_array_equal(got[i], ref)
    oidx, ow = oracle.route_topk(inp["logits"].numpy(), K)
    np.testing.assert_array_equal(np_(idx), oidx)
    olay = oracle.layout(oidx, inp["rank_offsets"].numpy(), E)
    o = dict(idx=oidx, w=ow, lay=olay, y=bits(inp["y"]),
             comb=oracle.combine(bits(inp["y"]), oidx, ow, olay["pos"], olay["expert_offsets"],
                                 E))
    from test_gpu_pipeline import _assert_matches_oracle
    for i in range(steps):
        _assert_matches_oracle(torch.from_numpy(got[i].view(np.int16)).view(torch.bfloat16),
                               o, K, E)
