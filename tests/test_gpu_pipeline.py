"""Schedules built from the entry points (combine_ep_route_topk_gb300.pipeline):
two-micro-batch overlap on two streams and chunked ("ant-moving") rounds with
a bounded dispatch buffer.  Each must give the same combined output as the
single-batch path (per-token work is unchanged: same routing, same FMA chain)
and every micro-batch / round layout must match the CPU oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_route_topk_gb300 as ep
from combine_ep_route_topk_gb300 import pipeline as pl
from combine_ep_route_topk_gb300 import workloads as wl

from _util import np_

pytestmark = pytest.mark.gpu


def _row_experts(lay, E):
    counts = lay.expert_offsets[1:] - lay.expert_offsets[:-1]
    return torch.repeat_interleave(torch.arange(E, device=counts.device), counts.long())


def _scaled(out, scales, lay, E, n_rows):
    """Expert stand-in: row of expert e times 2^(e % 3) (exact in bf16), after
    dequantising FP8 rows (code * block scale)."""
    if scales is None:
        rows = out[:n_rows].float()
    else:
        H = out.shape[1]
        codes = out[:n_rows].view(torch.float8_e4m3fn).float().view(n_rows, H // 128, 128)
        rows = (codes * scales[:n_rows, :, None]).view(n_rows, H)
    e = _row_experts(lay, E)
    assert e.numel() == n_rows
    return (rows * torch.exp2((e % 3).float())[:, None]).to(torch.bfloat16)


def _single_batch(inp, w, dtype):
    N, E, K, H = inp["N"], w.E, w.K, w.H
    idx, wt = ep.ep_route_topk(inp["logits"].cuda(), K)
    lay = ep.ep_dispatch_layout(idx, inp["rank_offsets"].cuda(), E)
    out, sc = ep.ep_dispatch(inp["x"].cuda(), idx, lay.pos, lay.expert_offsets, E,
                             ep.EP_LAYOUT_CONTIG, 0, dtype)
    y = _scaled(out, sc, lay, E, N * K)
    return ep.ep_combine(y, idx, wt, lay.pos, lay.expert_offsets, E)


@pytest.mark.parametrize("name,dtype", [("lumpy", ep.EP_DTYPE_BF16),
                                        ("prefill", ep.EP_DTYPE_FP8_E4M3_B128)])
@pytest.mark.parametrize("groups", [None, [(0, 1), (1, 8)], [(0, 1), (1, 3), (3, 8)]])
def test_two_batch_overlap_matches_single_batch(name, dtype, groups):
    w = wl.WORKLOADS[name]
    if name == "prefill":
        w = w.scaled(batch=("uniform", 200, 300))
    inp = wl.make_inputs(w, seed=5, with_y=False)
    N, E, K, H = inp["N"], w.E, w.K, w.H
    logits, x, ro = inp["logits"].cuda(), inp["x"].cuda(), inp["rank_offsets"].cuda()
    comb = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    mbs = pl.make_micro_batches(logits, x, ro, K, dtype, comb, rank_groups=groups)
    assert len(mbs) == (2 if groups is None else len(groups))
    assert mbs[0].t0 == 0 and mbs[-1].t1 == N
    assert all(a.t1 == b.t0 for a, b in zip(mbs, mbs[1:]))
    pl.two_batch_overlap(mbs, K, dtype,
                         lambda mb: _scaled(mb.out, mb.scales, mb.lay, E, (mb.t1 - mb.t0) * K))
    torch.cuda.synchronize()
    ref = _single_batch(inp, w, dtype)
    torch.cuda.synchronize()
    assert torch.equal(comb.view(torch.int16), ref.view(torch.int16))
    for mb in mbs:
        idx, _ = oracle.route_topk(inp["logits"].numpy()[mb.t0:mb.t1], K)
        olay = oracle.layout(idx, np_(mb.ro), E)
        np.testing.assert_array_equal(np_(mb.lay.pos), olay["pos"])
        np.testing.assert_array_equal(np_(mb.lay.counts), olay["counts"])


@pytest.mark.parametrize("name,dtype,T", [("lumpy", ep.EP_DTYPE_BF16, 300),
                                          ("skew", ep.EP_DTYPE_BF16, 4096),
                                          ("prefill", ep.EP_DTYPE_FP8_E4M3_B128, 640)])
@pytest.mark.parametrize("sets", [1, 2, 3])
def test_chunked_rounds_match_single_batch(name, dtype, T, sets):
    w = wl.WORKLOADS[name]
    if name == "prefill":
        w = w.scaled(batch=("uniform", 200, 300))
    inp = wl.make_inputs(w, seed=6, with_y=False)
    N, E, K, H, R = inp["N"], w.E, w.K, w.H, w.R
    offs = inp["rank_offsets"].tolist()
    logits, x = inp["logits"].cuda(), inp["x"].cuda()
    comb = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    bufs = pl.make_chunk_buffers(T, E, K, H, R, dtype, "cuda", sets=sets)
    rounds = pl.chunked(logits, x, offs, K, dtype, bufs,
                        lambda t0, n, out, sc, lay: _scaled(out, sc, lay, E, n * K), comb)
    torch.cuda.synchronize()
    assert len(rounds) == (N + T - 1) // T > 1
    for b in (bufs if sets > 1 else [bufs]):
        assert b.out.shape[0] == T * K  # each dispatch buffer is bounded by the round
    ref = _single_batch(inp, w, dtype)
    torch.cuda.synchronize()
    assert torch.equal(comb.view(torch.int16), ref.view(torch.int16))
    idx_all, _ = oracle.route_topk(inp["logits"].numpy(), K)
    for t0, t1, lay in rounds:
        olay = oracle.layout(idx_all[t0:t1], np.array(pl.round_rank_offsets(offs, t0, t1),
                                                      np.int32), E)
        for nm in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
            np.testing.assert_array_equal(np_(getattr(lay, nm)), olay[nm], err_msg=nm)


def test_chunked_identity_experts_return_x():
    w = wl.WORKLOADS["lumpy"]
    inp = wl.make_inputs(w, seed=7, with_y=False)
    N, E, K, H, R = inp["N"], w.E, w.K, w.H, w.R
    x = inp["x"].cuda()
    comb = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    bufs = pl.make_chunk_buffers(512, E, K, H, R, ep.EP_DTYPE_BF16, "cuda")
    pl.chunked(inp["logits"].cuda(), x, inp["rank_offsets"].tolist(), K, ep.EP_DTYPE_BF16, bufs,
               lambda t0, n, out, sc, lay: out, comb)
    torch.cuda.synchronize()
    assert torch.equal(comb.view(torch.int16), x.view(torch.int16))


def _pinned(t):
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


@pytest.mark.parametrize("name,dtype", [("lumpy", ep.EP_DTYPE_BF16),
                                        ("prefill", ep.EP_DTYPE_FP8_E4M3_B128)])
def test_host_pipeline_matches_single_batch(name, dtype):
    """Steps over pinned host buffers, copies overlapped across steps: every
    step's result and the last step's dispatched rows equal the single-batch
    path's on the same inputs, bit for bit (including a reused buffer set)."""
    w = wl.WORKLOADS[name]
    if name == "prefill":
        w = w.scaled(batch=("uniform", 200, 300))
    E, K, H = w.E, w.K, w.H
    cases = []
    for seed in (21, 22):
        inp = wl.make_inputs(w, seed=seed, with_y=False)
        N = inp["N"]
        idx, wt = ep.ep_route_topk(inp["logits"].cuda(), K)
        lay = ep.ep_dispatch_layout(idx, inp["rank_offsets"].cuda(), E)
        out, sc = ep.ep_dispatch(inp["x"].cuda(), idx, lay.pos, lay.expert_offsets, E,
                                 ep.EP_LAYOUT_CONTIG, 0, dtype)
        y = _scaled(out, sc, lay, E, N * K)
        comb = ep.ep_combine(y, idx, wt, lay.pos, lay.expert_offsets, E)
        cases.append(dict(N=N, x=_pinned(inp["x"]), logits=_pinned(inp["logits"]),
                          ro=_pinned(inp["rank_offsets"]), y=_pinned(y.cpu()),
                          comb=comb.cpu(), out=out.cpu(), sc=None if sc is None else sc.cpu()))
    # the seeds draw different batch sizes, so each gets its own pipeline
    for c in cases:
        hp = pl.HostPipeline(c["N"], E, K, H, w.R, dtype)
        outs = [torch.empty(c["N"], H, dtype=torch.bfloat16, pin_memory=True) for _ in range(3)]
        for o in outs:
            hp.step(c["x"], c["logits"], c["ro"], c["y"], o)
        hp.synchronize()
        for o in outs:
            assert torch.equal(o, c["comb"])
        assert torch.equal(hp.out.cpu(), c["out"])
        if c["sc"] is not None:
            assert torch.equal(hp.scales.cpu(), c["sc"])


def test_host_pipeline_alternating_inputs():
    """Alternating two input sets of one size through a depth-2 pipeline: each
    step's result is its own inputs' (no buffer set is overwritten early)."""
    w = wl.WORKLOADS["lumpy"]
    E, K, H = w.E, w.K, w.H
    g = torch.Generator().manual_seed(3)
    N, R = 700, 4
    ro = torch.tensor([0, 100, 350, 351, 700], dtype=torch.int32)
    sets = []
    for _ in range(2):
        logits = torch.randn(N, E, generator=g)
        x = torch.randn(N, H, generator=g).to(torch.bfloat16)
        y = torch.randn(N * K, H, generator=g).to(torch.bfloat16)
        idx, wt = ep.ep_route_topk(logits.cuda(), K)
        lay = ep.ep_dispatch_layout(idx, ro.cuda(), E)
        comb = ep.ep_combine(y.cuda(), idx, wt, lay.pos, lay.expert_offsets, E)
        sets.append((_pinned(x), _pinned(logits), _pinned(ro), _pinned(y), comb.cpu()))
    hp = pl.HostPipeline(N, E, K, H, R, ep.EP_DTYPE_BF16)
    order = [0, 1, 0, 1, 1, 0]
    outs = [torch.empty(N, H, dtype=torch.bfloat16, pin_memory=True) for _ in order]
    for i, o in zip(order, outs):
        x, lg, r, y, _ = sets[i]
        hp.step(x, lg, r, y, o)
    hp.synchronize()
    for i, o in zip(order, outs):
        assert torch.equal(o, sets[i][4])


def test_host_pipeline_masked_with_expert_map():
    """The decode shape (masked capacity, overflow dropped) with a balanced
    renumbering map: each step's result equals the single-batch path's."""
    w = wl.WORKLOADS["decode"].scaled(batch=("uniform", 20, 60))
    E, K, H, cap = w.E, w.K, w.H, 4  # small capacity: some picks overflow
    inp = wl.make_inputs(w, seed=9, with_y=False)
    N = inp["N"]
    logits, ro, x = inp["logits"].cuda(), inp["rank_offsets"].cuda(), inp["x"].cuda()
    i0, _ = ep.ep_route_topk(logits, K)
    emap = ep.ep_expert_balance_map(ep.ep_dispatch_layout(i0, ro, E).counts)
    idx, wt = ep.ep_route_topk(logits, K, expert_map=emap)
    lay = ep.ep_dispatch_layout(idx, ro, E, cap)
    assert int(lay.overflow_count.item()) > 0
    g = torch.Generator().manual_seed(4)
    y = torch.randn(E, cap, H, generator=g).to(torch.bfloat16)
    comb = ep.ep_combine(y.cuda(), idx, wt, lay.pos, lay.expert_offsets, E,
                         ep.EP_LAYOUT_MASKED, cap).cpu()
    out, _ = ep.ep_dispatch(x, idx, lay.pos, lay.expert_offsets, E, ep.EP_LAYOUT_MASKED, cap,
                            ep.EP_DTYPE_BF16)
    hp = pl.HostPipeline(N, E, K, H, w.R, ep.EP_DTYPE_BF16, cap=cap, expert_map=emap)
    outs = [torch.empty(N, H, dtype=torch.bfloat16, pin_memory=True) for _ in range(3)]
    args = [_pinned(t) for t in (inp["x"], inp["logits"], inp["rank_offsets"], y)]
    for o in outs:
        hp.step(*args, o)
    hp.synchronize()
    for o in outs:
        assert torch.equal(o, comb)
    # only the delivered slots of the masked buffer are defined
    m = hp.layout.masked_m.cpu()
    ref = out.cpu().view(E, cap, H)
    got = hp.out.cpu().view(E, cap, H)
    for e in range(E):
        assert torch.equal(got[e, :m[e]], ref[e, :m[e]])
