"""ep_route_layout (route + layout in one cooperative persistent kernel)
against the CPU oracle: ids bit-exact, weights within the float tolerance,
every layout output bit-exact, status 0; on every workload and on the sizes
that exercise each compiled instance and the two-kernel fallback."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_route_topk_gb300 as ep
from combine_ep_route_topk_gb300 import workloads as wl

from _util import np_, weight_rtol

pytestmark = pytest.mark.gpu


def _check(logits, offs, K, cap, emap=None):
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    idx, w, lay = ep.ep_route_layout(torch.as_tensor(logits).cuda(),
                                     torch.as_tensor(offs).cuda(), K, cap,
                                     expert_map=None if emap is None else
                                     torch.as_tensor(emap).cuda(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    logits = np.asarray(logits)
    ridx, rw = oracle.route_topk(logits, K, expert_map=emap) if logits.shape[0] else \
        (np.zeros((0, K), np.int32), np.zeros((0, K), np.float32))
    np.testing.assert_array_equal(np_(idx), ridx)
    np.testing.assert_allclose(np_(w), rw, rtol=weight_rtol())
    ref = oracle.layout(ridx, np.asarray(offs), logits.shape[1], cap)
    for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
        np.testing.assert_array_equal(np_(getattr(lay, name)), ref[name], err_msg=name)
    if cap > 0:
        np.testing.assert_array_equal(np_(lay.masked_m), ref["masked_m"])
        assert int(lay.overflow_count.item()) == ref["overflow"]


@pytest.mark.parametrize("name,seed", [("toy", 0), ("lumpy", 0), ("lumpy", 3), ("decode", 0),
                                       ("prefill", 0), ("skew", 0)])
def test_route_layout_workloads(name, seed):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, seed=seed, with_y=False)
    cap = w.cap if w.cap else wl.masked_cap_overflow(inp["N"], w.K, w.E)
    _check(inp["logits"].numpy(), inp["rank_offsets"].numpy(), w.K, cap)
    _check(inp["logits"].numpy(), inp["rank_offsets"].numpy(), w.K, 0)


def test_route_layout_with_renumbering():
    w = wl.WORKLOADS["skew"]
    inp = wl.make_inputs(w, seed=2, with_y=False)
    emap = np.random.default_rng(0).permutation(w.E).astype(np.int32)
    _check(inp["logits"].numpy(), inp["rank_offsets"].numpy(), w.K, 0, emap)


@pytest.mark.parametrize("B,E,K,cap", [
    ([50, 0, 70, 3], 384, 8, 0),          # no fused instance: two-kernel fallback
    ([300, 200], 1024, 8, 16),            # E = 1024 (16-byte loads, runtime K)
    ([64] * 8, 100, 7, 9),                # scalar loads, runtime K
    ([0, 0, 0], 16, 2, 1),                # N = 0
    ([1] * 1024, 64, 4, 0),               # R = 1024
    ([9000, 1, 5000], 256, 8, 0),         # ragged chunks
    ([40] * 8, 512, 2, 0),
])
def test_route_layout_sizes(B, E, K, cap):
    g = torch.Generator().manual_seed(E + K + len(B))
    N = sum(B)
    offs = np.concatenate([[0], np.cumsum(B)]).astype(np.int32)
    _check(torch.randn(N, E, generator=g).numpy(), offs, K, cap)


def test_route_layout_graph_capture():
    w = wl.WORKLOADS["decode"]
    inp = wl.make_inputs(w, seed=0, with_y=False)
    N, E, K, R, cap = inp["N"], w.E, w.K, w.R, w.cap
    logits = inp["logits"].cuda()
    ro = inp["rank_offsets"].cuda()
    idx = torch.empty(N, K, dtype=torch.int32, device="cuda")
    wt = torch.empty(N, K, device="cuda")
    lay = ep.alloc_layout(N, E, K, R, cap, "cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(ep.ep_route_layout_workspace_size(N, E, K, R), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ep.ep_route_layout(logits, ro, K, cap, topk_idx=idx, topk_w=wt, out=lay, status=st,
                           workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ep.ep_route_layout(logits, ro, K, cap, topk_idx=idx, topk_w=wt, out=lay, status=st,
                           workspace=ws)
    new = wl.make_inputs(w, seed=9, with_y=False)["logits"]
    logits.copy_(new.cuda())
    graph.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ridx, _ = oracle.route_topk(new.numpy(), K)
    ref = oracle.layout(ridx, inp["rank_offsets"].numpy(), E, cap)
    np.testing.assert_array_equal(np_(idx), ridx)
    np.testing.assert_array_equal(np_(lay.pos), ref["pos"])
    np.testing.assert_array_equal(np_(lay.masked_m), ref["masked_m"])


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """The fused kernel's grid barrier bounds its wait.  A barrier that waits
    for a block that never comes must give up, set the status word and let
    every block return; the next library call then works as usual."""
    import time
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    status = ep.ep_selftest_wait_timeout()
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert time.perf_counter() - t0 < 30.0
    g = torch.Generator().manual_seed(1)
    logits = torch.randn(300, 64, generator=g)
    idx, w = ep.ep_route_topk(logits.cuda(), 4)
    ref_idx, _ = oracle.route_topk(logits.numpy(), 4)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)


@pytest.mark.parametrize("E", [256, 384])  # a fused instance; the two-kernel fallback
def test_status_word_left_at_one_is_cleared_by_the_next_call(E):
    """The status word is written on every call: a 1 left in it (here by the
    bounded-wait self-test, which records a timeout into the same word) reads
    0 after a normal call, on the fused kernel and on the two-kernel fallback
    (E = 384 has no fused instance), and the results match the oracle."""
    status = ep.ep_selftest_wait_timeout()
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    g = torch.Generator().manual_seed(E)
    B = [120, 0, 77, 300]
    N, K = sum(B), 8
    offs = np.concatenate([[0], np.cumsum(B)]).astype(np.int32)
    logits = torch.randn(N, E, generator=g)
    idx, w, lay = ep.ep_route_layout(logits.cuda(), torch.from_numpy(offs).cuda(), K, 0,
                                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ridx, _ = oracle.route_topk(logits.numpy(), K)
    ref = oracle.layout(ridx, offs, E)
    np.testing.assert_array_equal(np_(idx), ridx)
    for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
        np.testing.assert_array_equal(np_(getattr(lay, name)), ref[name], err_msg=name)
