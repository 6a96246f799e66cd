"""ep_route_dispatch (route, layout and dispatch in one call; two launches up
to 2048 tokens and 16384 picks) against the CPU oracle: top-K ids bit-exact,
weights within the float tolerance, every layout output bit-exact, every
dispatched row (bf16 copies, FP8 codes and scales) bit-exact.  Covers the
workloads that fit, the layout's edge cases (empty batch and ranks, rank
bounds inside a routing block of 8 tokens, 1024 ranks, one expert, scalar
and vector routing, expert maps with out-of-range entries), the sizes just
past the limits (where the call runs the route, layout and dispatch kernels),
and the decode step captured in a CUDA graph.  Output buffers start filled
with a sentinel on both sides, so rows that receive no pick must be left
alone."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_route_topk_gb300 as ep
from combine_ep_route_topk_gb300 import workloads as wl

from _util import bits, np_, weight_rtol

pytestmark = pytest.mark.gpu

BF16, FP8 = ep.EP_DTYPE_BF16, ep.EP_DTYPE_FP8_E4M3_B128
CONTIG, MASKED = ep.EP_LAYOUT_CONTIG, ep.EP_LAYOUT_MASKED


def _run_both(logits, x, offs, K, layout, cap, dtype, emap=None, expect_launches=None):
    N, E = logits.shape
    H = x.shape[1]
    rows = N * K if layout == CONTIG else E * cap
    if dtype == BF16:
        ref_out = np.full((rows, H), 0xFFFF, np.uint16)
        gpu_out = torch.full((rows, H), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        ref_s, gpu_s = None, None
    else:
        ref_out = np.full((rows, H), 0xFF, np.uint8)
        gpu_out = torch.full((rows, H), 0xFF, dtype=torch.uint8, device="cuda")
        ref_s = np.full((rows, H // 128), -1.0, np.float32)
        gpu_s = torch.full((rows, H // 128), -1.0, device="cuda")
    ridx, rw = oracle.route_topk(logits, K, expert_map=emap) if N else \
        (np.zeros((0, K), np.int32), np.zeros((0, K), np.float32))
    ref = oracle.layout(ridx, offs, E, cap)
    oracle.dispatch(bits(x), ridx, ref["pos"], ref["expert_offsets"], E, layout=layout,
                    cap=cap, dtype=dtype, out=ref_out, out_scales=ref_s)
    R = offs.shape[0] - 1
    lay = ep.alloc_layout(N, E, K, R, cap, "cuda")
    if cap > 0:
        lay.overflow_count.fill_(12345)  # the call must reset it
    before = ep.ep_kernel_launch_count()
    idx, w, lay, _, _ = ep.ep_route_dispatch(
        torch.from_numpy(logits).cuda(), torch.from_numpy(offs).cuda(), x.cuda(), K, layout, cap,
        dtype, expert_map=None if emap is None else torch.from_numpy(emap).cuda(), lay=lay,
        out=gpu_out, out_scales=gpu_s)
    launched = ep.ep_kernel_launch_count() - before
    torch.cuda.synchronize()
    if expect_launches is not None:
        assert launched == expect_launches
    np.testing.assert_array_equal(np_(idx), ridx)
    np.testing.assert_allclose(np_(w), rw, rtol=weight_rtol())
    for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
        np.testing.assert_array_equal(np_(getattr(lay, name)), ref[name], err_msg=name)
    if cap > 0:
        np.testing.assert_array_equal(np_(lay.masked_m), ref["masked_m"])
        assert int(lay.overflow_count.item()) == ref["overflow"]
    if dtype == BF16:
        np.testing.assert_array_equal(bits(gpu_out), ref_out)
    else:
        np.testing.assert_array_equal(np_(gpu_out), ref_out)
        np.testing.assert_array_equal(np_(gpu_s).view(np.uint32), ref_s.view(np.uint32))


@pytest.mark.parametrize("name,layout,dtype,scaled", [
    ("toy", CONTIG, BF16, {}),
    ("toy", MASKED, FP8, {}),
    ("lumpy", CONTIG, BF16, {}),
    ("lumpy", MASKED, BF16, {}),                                  # capacity with overflow
    ("decode", MASKED, BF16, {}),                                 # the decode step
    ("decode", MASKED, FP8, {}),
    ("decode", CONTIG, FP8, {}),
    ("prefill", CONTIG, FP8, {"batch": ("uniform", 150, 250)}),  # ragged, < 2048 tokens
    ("skew", CONTIG, BF16, {"batch": ("uniform_to_total", 1024, 3072, 2000)}),
])
def test_route_dispatch_workloads(name, layout, dtype, scaled):
    w = wl.WORKLOADS[name]
    if scaled:
        w = w.scaled(**scaled)
    inp = wl.make_inputs(w, seed=2, with_y=False)
    N = inp["N"]
    assert N <= 2048 and N * w.K <= 16384
    cap = 0
    if layout == MASKED:
        cap = w.cap if w.cap > 0 else wl.masked_cap_overflow(N, w.K, w.E)
    emap = None
    if w.relabel:  # the balanced renumbering of the same batch, by the oracle
        i0, _ = oracle.route_topk(inp["logits"].numpy(), w.K)
        emap = oracle.balance_map(oracle.layout(i0, inp["rank_offsets"].numpy(), w.E)["counts"])
    _run_both(inp["logits"].numpy(), inp["x"], inp["rank_offsets"].numpy(), w.K, layout, cap,
              dtype, emap=emap, expect_launches=2)


def _case(seed, B, E, H):
    g = np.random.default_rng(seed)
    N = int(sum(B))
    offs = np.concatenate([[0], np.cumsum(B)]).astype(np.int32)
    logits = g.standard_normal((N, E)).astype(np.float32)
    x = torch.from_numpy(g.standard_normal((N, H)).astype(np.float32)).to(torch.bfloat16)
    return logits, x, offs


@pytest.mark.parametrize("B,E,K,H,layout,cap,dtype", [
    ([0, 0, 0], 16, 2, 128, CONTIG, 0, BF16),           # N = 0
    ([0, 0, 0], 16, 2, 128, MASKED, 3, BF16),
    ([5, 0, 0, 9, 0, 3], 32, 4, 256, CONTIG, 2, FP8),   # empty ranks, bounds inside blocks
    ([13, 3, 77, 1, 0, 30], 100, 7, 1024, MASKED, 2, BF16),  # scalar routing, runtime K
    ([1] * 1024, 64, 4, 128, CONTIG, 0, BF16),          # R = 1024
    ([300, 211], 1, 1, 136, MASKED, 100, BF16),          # one expert, overflow
    ([1000, 1048], 1024, 8, 128, CONTIG, 0, BF16),       # 2048 tokens, 16384 picks: the limit
    ([7, 9, 11], 384, 8, 128, MASKED, 1, FP8),           # E = 384: scalar routing of 12 per lane
    ([64] * 8, 512, 32, 8, CONTIG, 0, BF16),             # K = 32, one vector per row
])
def test_route_dispatch_edge_cases(B, E, K, H, layout, cap, dtype):
    logits, x, offs = _case(len(B) * 31 + E + K, B, E, H)
    _run_both(logits, x, offs, K, layout, cap, dtype, expect_launches=2 if sum(B) else 1)


def test_route_dispatch_expert_map_with_out_of_range_entries():
    """Map entries outside [0, E) make the pick "no pick": not counted, pos
    -1, no row moved (the oracle's reading)."""
    logits, x, offs = _case(7, [40, 0, 57], 64, 256)
    emap = np.random.default_rng(3).permutation(64).astype(np.int32)
    emap[[3, 17, 40]] = [-1, 64, 1000]
    _run_both(logits, x, offs, 8, MASKED, 4, BF16, emap=emap)
    _run_both(logits, x, offs, 8, CONTIG, 0, FP8, emap=emap)


@pytest.mark.parametrize("B,K", [([1000, 1049], 8),     # 2049 tokens
                                 ([500, 500, 600], 16),   # 1600 tokens but 25600 picks
                                 ([2000, 2100], 4)])      # 4100 tokens: bulk-copy dispatch
def test_route_dispatch_past_the_limits(B, K):
    """Past 2048 tokens or 16384 picks the call runs the route kernel, the
    layout kernels and the dispatch kernel, with the same results."""
    logits, x, offs = _case(11, B, 256, 256)
    _run_both(logits, x, offs, K, CONTIG, 0, FP8, expect_launches=5)
    _run_both(logits, x, offs, K, MASKED, 2 * sum(B) * K // 256, BF16, expect_launches=5)


def test_route_dispatch_matches_the_separate_calls():
    w = wl.WORKLOADS["decode"]
    inp = wl.make_inputs(w, seed=8, with_y=False)
    logits, ro, x = inp["logits"].cuda(), inp["rank_offsets"].cuda(), inp["x"].cuda()
    idx_a, w_a = ep.ep_route_topk(logits, w.K)
    lay_a = ep.ep_dispatch_layout(idx_a, ro, w.E, w.cap)
    out_a, _ = ep.ep_dispatch(x, idx_a, lay_a.pos, lay_a.expert_offsets, w.E, MASKED, w.cap)
    idx_b, w_b, lay_b, out_b, _ = ep.ep_route_dispatch(logits, ro, x, w.K, MASKED, w.cap)
    torch.cuda.synchronize()
    assert torch.equal(idx_a, idx_b) and torch.equal(w_a, w_b)
    for name in lay_a._fields:
        assert torch.equal(getattr(lay_a, name), getattr(lay_b, name)), name
    m = lay_a.masked_m.cpu()
    a = out_a.view(w.E, w.cap, w.H)
    b = out_b.view(w.E, w.cap, w.H)
    for e in range(w.E):
        assert torch.equal(a[e, :m[e]], b[e, :m[e]])


def test_decode_step_in_a_cuda_graph():
    """route+layout+dispatch, then combine, captured once and replayed on new
    logits; every output against the oracle (combine fed the oracle's
    weights, so it is bit-exact)."""
    w = wl.WORKLOADS["decode"]
    inp = wl.make_inputs(w, seed=0)
    N, E, K, H, R, cap = inp["N"], w.E, w.K, w.H, w.R, w.cap
    logits, ro = inp["logits"].cuda(), inp["rank_offsets"].cuda()
    x, y = inp["x"].cuda(), inp["y"].cuda()
    idx = torch.empty(N, K, dtype=torch.int32, device="cuda")
    wt = torch.empty(N, K, device="cuda")
    lay = ep.alloc_layout(N, E, K, R, cap, "cuda")
    out = torch.empty(E * cap, H, dtype=torch.bfloat16, device="cuda")
    comb = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(ep.ep_route_dispatch_workspace_size(N, E, K, R), dtype=torch.uint8,
                     device="cuda")

    def step():
        ep.ep_route_dispatch(logits, ro, x, K, MASKED, cap, topk_idx=idx, topk_w=wt, lay=lay,
                             out=out, workspace=ws)
        ep.ep_combine(y, idx, wt, lay.pos, lay.expert_offsets, E, MASKED, cap, out=comb)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    new = wl.make_inputs(w, seed=13, with_y=False)["logits"]
    logits.copy_(new.cuda())
    graph.replay()
    torch.cuda.synchronize()
    oidx, ow = oracle.route_topk(new.numpy(), K)
    olay = oracle.layout(oidx, inp["rank_offsets"].numpy(), E, cap)
    np.testing.assert_array_equal(np_(idx), oidx)
    np.testing.assert_allclose(np_(wt), ow, rtol=weight_rtol())
    for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src",
                 "masked_m"):
        np.testing.assert_array_equal(np_(getattr(lay, name)), olay[name], err_msg=name)
    assert int(lay.overflow_count.item()) == olay["overflow"]
    oout, _ = oracle.dispatch(bits(inp["x"]), oidx, olay["pos"], olay["expert_offsets"], E,
                              layout=oracle.LAYOUT_MASKED, cap=cap)
    got = bits(out).reshape(E, cap, H)
    ref = oout.reshape(E, cap, H)
    for e in range(E):
        m = olay["masked_m"][e]
        np.testing.assert_array_equal(got[e, :m], ref[e, :m])
    ocomb = oracle.combine(bits(inp["y"]), oidx, ow, olay["pos"], olay["expert_offsets"], E,
                           layout=oracle.LAYOUT_MASKED, cap=cap)
    gcomb = ep.ep_combine(y, idx, torch.from_numpy(ow).cuda(), lay.pos, lay.expert_offsets, E,
                          MASKED, cap)
    np.testing.assert_array_equal(bits(gcomb), ocomb)
