"""ep_dispatch_layout_static: the layout entry point that allocates nothing.

It exists for callers that cannot allocate device memory (an embedder whose
device memory is reserved up front by another allocator, a plain C host
without a device allocator, code running where cudaMalloc is not permitted):
its scratch is a fixed array inside the library instead of a caller-provided
workspace.  These tests call it through the C ABI and compare every output
with the workspace entry point, ep_dispatch_layout, on two calls in a row
(the array keeps the previous call's contents, which must not leak into the
next result).  Integer outputs, so the comparison is bit-exact.

This file is collected last on purpose: a failure here stops a -x run only
after every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

from combine_ep_route_topk_gb300 import build as ep_build
from combine_ep_route_topk_gb300 import ep
from combine_ep_route_topk_gb300 import workloads as wl

SCRATCH_BYTES = 4 * 1024 * 1024
P = ctypes.c_void_p


def _static_fn():
    L = ep.lib()
    f = L.ep_dispatch_layout_static
    i32 = ctypes.c_int32
    f.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P]
    f.restype = ctypes.c_int
    return f


def _ptr(t):
    return None if t is None else P(t.data_ptr())


def test_static_layout_refuses_oversized_problems_without_launching():
    ep_build.build()
    f = _static_fn()
    before = ep.lib().ep_kernel_launch_count()
    # 1024 ranks x 1024 experts need more than 4 MiB of chunk histograms
    assert ep.ep_dispatch_layout_workspace_size(1 << 20, 1024, 8, 1024) > SCRATCH_BYTES
    fake = P(4096)
    st = f(fake, fake, 1024, 1 << 20, 1024, 8, 0, fake, fake, fake, fake, fake, None, None,
           None)
    assert st == 4  # EP_ERR_UNSUPPORTED
    assert f(fake, fake, 8, 100, 16, 20, 0, fake, fake, fake, fake, fake, None, None,
             None) == 1  # K > E: EP_ERR_INVALID_ARG
    assert ep.lib().ep_kernel_launch_count() == before


def _run_static(idx, ro, E, cap):
    N, K = idx.shape
    R = ro.shape[0] - 1
    out = ep.alloc_layout(N, E, K, R, cap, idx.device)
    st = _static_fn()(_ptr(idx), _ptr(ro), R, N, E, K, cap, _ptr(out.counts),
                      _ptr(out.expert_offsets), _ptr(out.rank_expert_offsets), _ptr(out.pos),
                      _ptr(out.row_src), _ptr(out.masked_m), _ptr(out.overflow_count),
                      P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return out


def _same(a, b, cap):
    for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    if cap > 0:
        assert torch.equal(a.masked_m, b.masked_m)
        assert torch.equal(a.overflow_count, b.overflow_count)


@pytest.mark.gpu
def test_static_layout_matches_workspace_layout_on_two_calls_in_a_row():
    cases = [(wl.WORKLOADS["prefill"], 0, 0),    # 32768 tokens, E=256, K=8
             (wl.WORKLOADS["lumpy"], 3, 400)]    # ragged ranks, masked capacity
    for w, seed, cap in cases:
        inp = wl.make_inputs(w, seed=seed, with_y=False)
        N, E, K, R = inp["N"], w.E, w.K, w.R
        assert ep.ep_dispatch_layout_workspace_size(N, E, K, R) <= SCRATCH_BYTES
        logits = inp["logits"].cuda()
        ro = inp["rank_offsets"].cuda()
        idx, _ = ep.ep_route_topk(logits, K)
        ref = ep.ep_dispatch_layout(idx, ro, E, cap)
        got = _run_static(idx, ro, E, cap)
        torch.cuda.synchronize()
        _same(got, ref, cap)
    # a second pair of calls right after, on different routing: the scratch
    # still holds the previous call's histograms
    w = wl.WORKLOADS["decode"]
    for seed in (5, 6):
        inp = wl.make_inputs(w, seed=seed, with_y=False)
        idx, _ = ep.ep_route_topk(inp["logits"].cuda(), w.K)
        ro = inp["rank_offsets"].cuda()
        got = _run_static(idx, ro, w.E, w.cap)
        ref = ep.ep_dispatch_layout(idx, ro, w.E, w.cap)
        torch.cuda.synchronize()
        _same(got, ref, w.cap)
