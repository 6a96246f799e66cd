"""ep_dispatch_layout_static: the layout entry point that allocates nothing.

It exists for callers that cannot allocate device memory (an embedder whose
device memory is reserved up front by another allocator, a plain C host
without a device allocator, code running where cudaMalloc is not permitted):
its scratch is a fixed 4 MiB array inside the library instead of a
caller-provided workspace.  These tests call it through the C ABI, several
times in a row on different routing and sizes, and compare every output with
the CPU oracle's layout and with the workspace entry point,
ep_dispatch_layout (integer outputs, so both comparisons are bit-exact).  The
array keeps the previous call's contents, which must never leak into the next
result, so the calls that are compared all take the three-kernel path, the
one that uses the array (EP_LAYOUT_CLUSTER=0 for the small problems, which
would otherwise run as one launch without scratch).  One case
needs exactly the whole array, so its expert totals end on its last bytes.

This file is collected last on purpose: a failure here stops a -x run only
after every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_ep_route_topk_gb300 import build as ep_build
from combine_ep_route_topk_gb300 import ep
from combine_ep_route_topk_gb300 import workloads as wl

from _util import np_

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
    """Host-side checks only (no device call): runs wherever the library
    loads, with or without a GPU."""
    ep_build.build()
    f = _static_fn()
    before = ep.lib().ep_kernel_launch_count()
    # 1024 ranks x 1024 experts need more than 4 MiB of chunk histograms
    assert ep.ep_dispatch_layout_workspace_size(1 << 20, 1024, 8, 1024) > SCRATCH_BYTES
    fake = P(4096)
    st = f(fake, fake, 1024, 1 << 20, 1024, 8, 0, fake, fake, fake, fake, fake, None, None,
           None)
    assert st == 4  # EP_ERR_UNSUPPORTED
    # the largest accepted size and the next one: 2048 tokens of 1024 experts
    # over 767 ranks need exactly the array; one rank more needs one more
    # histogram row (4 E bytes) and is refused
    assert ep.ep_dispatch_layout_workspace_size(2048, 1024, 8, 767) == SCRATCH_BYTES
    over = ep.ep_dispatch_layout_workspace_size(2048, 1024, 8, 768)
    assert over == SCRATCH_BYTES + 4 * 1024
    assert f(fake, fake, 768, 2048, 1024, 8, 0, fake, fake, fake, fake, fake, None, None,
             None) == 4
    assert f(fake, fake, 8, 100, 16, 20, 0, fake, fake, fake, fake, fake, None, None,
             None) == 1  # K > E: EP_ERR_INVALID_ARG
    assert ep.lib().ep_kernel_launch_count() == before


def _run_static(idx, ro, E, cap):
    N, K = idx.shape
    R = ro.shape[0] - 1
    out = ep.alloc_layout(N, E, K, R, cap, idx.device)
    before = ep.lib().ep_kernel_launch_count()
    st = _static_fn()(_ptr(idx), _ptr(ro), R, N, E, K, cap, _ptr(out.counts),
                      _ptr(out.expert_offsets), _ptr(out.rank_expert_offsets), _ptr(out.pos),
                      _ptr(out.row_src), _ptr(out.masked_m), _ptr(out.overflow_count),
                      P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    # three launches: the path that keeps its histograms in the static array
    assert ep.lib().ep_kernel_launch_count() - before == 3
    return out


def _same(a, b, cap):
    for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    if cap > 0:
        assert torch.equal(a.masked_m, b.masked_m)
        assert torch.equal(a.overflow_count, b.overflow_count)


def _against_oracle(got, idx_np, ro_np, E, cap):
    ref = oracle.layout(idx_np, ro_np, E, cap)
    for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
        np.testing.assert_array_equal(np_(getattr(got, name)), ref[name], err_msg=name)
    if cap > 0:
        np.testing.assert_array_equal(np_(got.masked_m), ref["masked_m"])
        assert int(got.overflow_count.item()) == ref["overflow"]


def _workload_case(name, seed, cap=None):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, seed=seed, with_y=False)
    idx, _ = oracle.route_topk(inp["logits"].numpy(), w.K)
    return idx, inp["rank_offsets"].numpy(), w.E, w.cap if cap is None else cap


def _full_array_case(seed):
    """2048 tokens, E = 1024, K = 8 over 767 ranks of random sizes (some
    empty): the workspace is exactly the static array."""
    rng = np.random.default_rng(seed)
    B = rng.multinomial(2048, np.full(767, 1.0 / 767))
    ro = np.concatenate([[0], np.cumsum(B)]).astype(np.int32)
    idx = np.argsort(rng.random((2048, 1024)), axis=1)[:, :8].astype(np.int32)
    return idx, ro, 1024, 0


@pytest.mark.gpu
def test_static_layout_matches_oracle_and_workspace_layout_on_calls_in_a_row(monkeypatch):
    monkeypatch.setenv("EP_LAYOUT_CLUSTER", "0")  # small problems use the array too
    cases = [_workload_case("prefill", 0, 0),        # 32768 tokens, E=256, K=8
             _workload_case("prefill", 1, 0),        # the same size, other routing
             _workload_case("lumpy", 3, 400),        # ragged ranks, masked capacity
             _full_array_case(0),                    # the whole array, E = 1024
             _workload_case("decode", 5),            # masked, cap 128, after a larger E
             _workload_case("decode", 6),
             _full_array_case(1)]
    for idx_np, ro_np, E, cap in cases:
        N, K = idx_np.shape
        R = ro_np.shape[0] - 1
        assert ep.ep_dispatch_layout_workspace_size(N, E, K, R) <= SCRATCH_BYTES
        idx = torch.from_numpy(idx_np).cuda()
        ro = torch.from_numpy(ro_np).cuda()
        got = _run_static(idx, ro, E, cap)
        ref = ep.ep_dispatch_layout(idx, ro, E, cap)
        torch.cuda.synchronize()
        _same(got, ref, cap)
        _against_oracle(got, idx_np, ro_np, E, cap)


@pytest.mark.gpu
def test_static_layout_two_calls_in_a_row_without_a_sync():
    """Two calls queued back to back on one stream (the second overwrites the
    array while nothing has been read back yet), each checked afterwards."""
    a = _workload_case("prefill", 2, 0)
    b = _workload_case("prefill", 3, 0)
    outs = []
    for idx_np, ro_np, E, cap in (a, b):
        outs.append(_run_static(torch.from_numpy(idx_np).cuda(),
                                torch.from_numpy(ro_np).cuda(), E, cap))
    torch.cuda.synchronize()
    for got, (idx_np, ro_np, E, cap) in zip(outs, (a, b)):
        _against_oracle(got, idx_np, ro_np, E, cap)
