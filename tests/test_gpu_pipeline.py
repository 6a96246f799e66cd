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
def test_two_batch_overlap_matches_single_batch(name, dtype):
    w = wl.WORKLOADS[name]
    if name == "prefill":
        w = w.scaled(batch=("uniform", 200, 300))
    inp = wl.make_inputs(w, seed=5, with_y=False)
    N, E, K, H = inp["N"], w.E, w.K, w.H
    logits, x, ro = inp["logits"].cuda(), inp["x"].cuda(), inp["rank_offsets"].cuda()
    comb = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    mbs = pl.make_micro_batches(logits, x, ro, K, dtype, comb)
    assert len(mbs) == 2 and mbs[0].t1 == mbs[1].t0
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
def test_chunked_rounds_match_single_batch(name, dtype, T):
    w = wl.WORKLOADS[name]
    if name == "prefill":
        w = w.scaled(batch=("uniform", 200, 300))
    inp = wl.make_inputs(w, seed=6, with_y=False)
    N, E, K, H, R = inp["N"], w.E, w.K, w.H, w.R
    offs = inp["rank_offsets"].tolist()
    logits, x = inp["logits"].cuda(), inp["x"].cuda()
    comb = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    bufs = pl.make_chunk_buffers(T, E, K, H, R, dtype, "cuda")
    rounds = pl.chunked(logits, x, offs, K, dtype, bufs,
                        lambda t0, n, out, sc, lay: _scaled(out, sc, lay, E, n * K), comb)
    torch.cuda.synchronize()
    assert len(rounds) == (N + T - 1) // T > 1
    assert bufs.out.shape[0] == T * K  # the dispatch buffer is bounded by the round
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
