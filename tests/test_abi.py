"""The C ABI library: it loads, exports every function include/ep.h declares,
and its host-side argument checks return the documented status codes without
launching anything (these calls never reach the GPU, so they run on CPU)."""
import ctypes
import os
import re

import pytest

from combine_ep_route_topk_gb300 import build as ep_build
from combine_ep_route_topk_gb300 import ep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, WORKSPACE, CUDA, UNSUPPORTED = 0, 1, 2, 3, 4
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def L():
    ep_build.build()
    return ep.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "ep.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "ep_route_topk" in names and "ep_combine" in names and len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_static_queries(L):
    launches0 = L.ep_kernel_launch_count()  # other tests of the process may have launched
    assert L.ep_abi_version() == 1
    assert L.ep_status_string(0) == b"EP_OK"
    assert L.ep_status_string(2) == b"EP_ERR_WORKSPACE"
    assert L.ep_kernel_launch_count() == launches0
    a = ep.ep_dispatch_layout_workspace_size(32768, 256, 8, 8)
    b = ep.ep_dispatch_layout_workspace_size(65536, 256, 8, 8)
    assert a % 256 == 0 and b % 256 == 0 and 0 < a <= b


def p(v=4096):
    return P(v)


def test_route_argument_checks(L):
    launches0 = L.ep_kernel_launch_count()
    f = L.ep_route_topk
    assert f(p(), 10, 16, 17, None, p(), p(), None) == INVALID       # K > E
    assert f(p(), 10, 16, 0, None, p(), p(), None) == INVALID        # K < 1
    assert f(p(), -1, 16, 2, None, p(), p(), None) == INVALID        # N < 0
    assert f(p(), 10, 2048, 2, None, p(), p(), None) == UNSUPPORTED  # E > 1024
    assert f(p(), 10, 64, 33, None, p(), p(), None) == UNSUPPORTED   # K > 32
    assert f(p(), 1 << 30, 16, 4, None, p(), p(), None) == UNSUPPORTED  # N*K overflow
    assert f(None, 10, 16, 2, None, p(), p(), None) == INVALID       # null logits
    assert f(p(4098), 10, 16, 2, None, p(), p(), None) == INVALID    # misaligned
    assert L.ep_kernel_launch_count() == launches0


def test_layout_argument_checks(L):
    launches0 = L.ep_kernel_launch_count()
    f = L.ep_dispatch_layout
    need = ep.ep_dispatch_layout_workspace_size(100, 16, 2, 4)

    def call(R=4, N=100, E=16, K=2, cap=0, mm=None, ov=None, ws=p(), wsb=need):
        return f(p(), p(), R, N, E, K, cap, p(), p(), p(), p(), p(), mm, ov, ws, wsb, None)
    assert call(wsb=need - 1) == WORKSPACE
    assert call(ws=None) == WORKSPACE
    assert call(ws=p(4104)) == WORKSPACE  # workspace not 16-byte aligned
    assert call(R=0) == INVALID
    assert call(R=2000) == UNSUPPORTED
    assert call(cap=-1) == INVALID
    assert call(cap=0, mm=p()) == INVALID  # masked outputs need a capacity
    assert call(K=20) == INVALID
    assert L.ep_kernel_launch_count() == launches0


def test_dispatch_and_combine_argument_checks(L):
    launches0 = L.ep_kernel_launch_count()
    d = L.ep_dispatch
    c = L.ep_combine

    def disp(x=p(), H=1024, layout=0, cap=0, dtype=0, scales=None, out=p()):
        return d(x, 100, H, 16, 2, p(), p(), p(), layout, cap, dtype, out, scales, None)
    assert disp(H=100) == INVALID                 # H % 8
    assert disp(H=0) == INVALID
    assert disp(x=p(4104)) == INVALID             # x not 16-byte aligned
    assert disp(out=p(4100)) == INVALID           # out not 16-byte aligned
    assert disp(layout=1, cap=0) == INVALID       # masked needs cap > 0
    assert disp(layout=7) == INVALID
    assert disp(dtype=9) == INVALID
    assert disp(dtype=1, H=520, scales=p()) == INVALID  # FP8 needs H % 128
    assert disp(dtype=1, scales=None) == INVALID        # FP8 needs scales
    assert c(p(), 100, 1024, 16, 2, p(), None, p(), p(), 0, 0, p(), None) == INVALID  # no weights
    assert c(p(), 100, 1024, 16, 20, p(), p(), p(), p(), 0, 0, p(), None) == INVALID  # K > E
    assert L.ep_expert_balance_map(p(), 3, 16, p(), None) == INVALID  # E % R != 0
    assert L.ep_expert_balance_map(p(), 0, 16, p(), None) == INVALID
    assert L.ep_kernel_launch_count() == launches0


def test_selftest_argument_checks(L):
    launches0 = L.ep_kernel_launch_count()
    f = L.ep_selftest_wait_timeout
    assert f(None, p(), 256, None) == INVALID
    assert f(p(), None, 256, None) == INVALID
    assert f(p(), p(), 3, None) == INVALID        # room for the counter
    assert f(p(4098), p(), 256, None) == INVALID  # status not 4-byte aligned
    assert L.ep_kernel_launch_count() == launches0


def test_binding_refuses_cpu_tensors(L):
    import torch
    with pytest.raises(ep.EPError):
        ep.ep_route_topk(torch.zeros(4, 16), 2, topk_idx=torch.zeros(4, 2, dtype=torch.int32),
                         topk_w=torch.zeros(4, 2))


def test_host_pipeline_argument_checks(L):
    launches0 = L.ep_kernel_launch_count()
    size = L.ep_host_pipeline_workspace_size
    assert size(1024, 256, 8, 7168, 8, 128, 0, 2) > 0
    assert size(1024, 256, 8, 7168, 8, 128, 0, 2) < size(1024, 256, 8, 7168, 8, 128, 0, 3)
    assert size(0, 256, 8, 7168, 8, 0, 0, 2) == 0          # N >= 1
    assert size(10, 16, 2, 100, 4, 0, 0, 2) == 0           # H % 8
    assert size(10, 16, 2, 200, 4, 0, 1, 2) == 0           # FP8 needs H % 128
    assert size(10, 16, 2, 128, 4, 0, 0, 5) == 0           # depth 1..4
    create = L.ep_host_pipeline_create
    need = size(10, 16, 2, 128, 4, 0, 0, 2)
    out = P()
    assert create(10, 16, 2, 128, 4, 0, 0, 2, None, p(4096), need, None) == INVALID  # no out
    assert create(10, 16, 17, 128, 4, 0, 0, 2, None, p(4096), need,
                  ctypes.byref(out)) == INVALID                                  # K > E
    assert create(10, 2048, 2, 128, 4, 0, 0, 2, None, p(4096), need,
                  ctypes.byref(out)) == UNSUPPORTED                              # E > 1024
    assert create(10, 16, 2, 128, 4, 0, 0, 2, None, p(4096), need - 1,
                  ctypes.byref(out)) == WORKSPACE
    assert create(10, 16, 2, 128, 4, 0, 0, 2, None, p(4096 + 16), need,
                  ctypes.byref(out)) == WORKSPACE                                # 256-byte aligned
    assert create(10, 16, 2, 128, 4, 0, 0, 2, p(4098), p(4096), need,
                  ctypes.byref(out)) == INVALID                                  # expert_map align
    assert out.value is None
    assert L.ep_host_pipeline_step(None, p(), p(), p(), p(), p(), None) == INVALID
    assert L.ep_host_pipeline_join(None, None) == INVALID
    ptr, nb = P(), ctypes.c_size_t()
    assert L.ep_host_pipeline_buffer(None, 0, ctypes.byref(ptr), ctypes.byref(nb)) == INVALID
    assert L.ep_host_pipeline_destroy(None) == OK
    assert L.ep_kernel_launch_count() == launches0


C_CLIENT = r"""
#include <stdio.h>
#include "ep.h"

int main(void) {
    /* argument checks only: nothing here reaches a GPU */
    ep_status_t st = ep_route_topk((const float*)0, 10, 16, 17, 0, 0, 0, 0);  /* K > E */
    if (st != EP_ERR_INVALID_ARG) return 1;
    st = ep_dispatch((const void*)0, 4, 100, 16, 2, 0, 0, 0, EP_LAYOUT_CONTIG, 0,
                     EP_DTYPE_BF16, 0, 0, 0);  /* H % 8 != 0 */
    if (st != EP_ERR_INVALID_ARG) return 2;
    if (ep_abi_version() != 1) return 3;
    if (ep_dispatch_layout_workspace_size(32768, 256, 8, 8) == 0) return 4;
    if (ep_kernel_launch_count() != 0) return 5;
    printf("%s\n", ep_status_string(EP_ERR_UNSUPPORTED));
    return 0;
}
"""


def test_header_is_plain_c_and_the_library_links_from_c(L, tmp_path):
    """include/ep.h compiles as C11 with warnings as errors, and a C program
    links against libep_gb300.so and gets the documented status codes."""
    import subprocess
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(ep.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lep_gb300", f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.strip() == "EP_ERR_UNSUPPORTED"


def test_host_memory_argument_checks(L):
    """ep_host_alloc / ep_host_free / ep_host_pipeline_copy_ms refuse bad
    arguments on the host, before any mapping or CUDA call."""
    out = P(1234)
    assert L.ep_host_alloc(0, ctypes.byref(out)) == INVALID
    assert out.value is None  # cleared on failure
    assert L.ep_host_alloc(4096, None) == INVALID
    assert L.ep_host_free(None) == OK
    assert L.ep_host_free(p(4096)) == INVALID  # not from ep_host_alloc
    a, b = ctypes.c_float(), ctypes.c_float()
    assert L.ep_host_pipeline_copy_ms(None, ctypes.byref(a), ctypes.byref(b)) == INVALID



def test_route_dispatch_argument_checks(L):
    launches0 = L.ep_kernel_launch_count()
    f = L.ep_route_dispatch
    need = L.ep_route_dispatch_workspace_size(100, 16, 2, 4)
    assert need > 0 and need % 256 == 0

    def call(N=100, H=256, E=16, K=2, R=4, layout=0, cap=0, dtype=0, x=p(), out=p(), sc=p(),
             mm=None, ov=None, ws=p(), wsb=need):
        return f(p(), p(), x, R, N, H, E, K, None, layout, cap, dtype, p(), p(), p(), p(), p(),
                 p(), p(), mm, ov, out, sc, ws, wsb, None)
    assert call(K=20) == INVALID                 # K > E
    assert call(layout=1, cap=0) == INVALID      # masked needs a capacity
    assert call(cap=0, ov=p()) == INVALID        # masked outputs need a capacity
    assert call(H=100) == INVALID                # H % 8
    assert call(dtype=1, H=200) == INVALID       # FP8 needs H % 128
    assert call(dtype=1, sc=None) == INVALID     # FP8 needs scales
    assert call(x=p(4104)) == INVALID            # x not 16-byte aligned
    assert call(R=0) == INVALID
    assert call(R=2000) == UNSUPPORTED
    assert call(ws=None) == WORKSPACE
    assert call(wsb=need - 1) == WORKSPACE
    # past 2048 tokens the layout workspace is needed instead of the histograms
    big = L.ep_route_dispatch_workspace_size(4096, 16, 2, 4)
    assert big >= ep.ep_dispatch_layout_workspace_size(4096, 16, 2, 4)
    assert L.ep_kernel_launch_count() == launches0
