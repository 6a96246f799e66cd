"""The prefill workload at full size (8 ranks x 4096 tokens, E=256, K=8,
H=7168), run exactly as bench.py runs it (same entry points, same launch
configuration, inputs drawn on the device), checked against the oracle:
routing and layout on every token (the oracle finishes those in about a
second), FP8 dispatch rows and combine outputs on a sample of tokens that
the oracle recomputes one by one (random tokens plus the first and last
token of every rank).  The end-to-end schedule over host buffers must give
the device path's results bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_route_topk_gb300 as ep
from combine_ep_route_topk_gb300 import workloads as wl

from _util import bf16_ulp, bits, combine_rel_err, np_, weight_rtol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prefill():
    w = wl.WORKLOADS["prefill"]
    inp = wl.make_inputs(w, seed=0, device="cuda")
    N, E, K, H, R = inp["N"], w.E, w.K, w.H, w.R
    idx = torch.empty(N, K, dtype=torch.int32, device="cuda")
    wt = torch.empty(N, K, device="cuda")
    lay = ep.alloc_layout(N, E, K, R, 0, "cuda")
    ws = torch.empty(ep.ep_dispatch_layout_workspace_size(N, E, K, R), dtype=torch.uint8,
                     device="cuda")
    q = torch.empty(N * K, H, dtype=torch.uint8, device="cuda")
    qs = torch.empty(N * K, H // 128, device="cuda")
    comb = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    ep.ep_route_topk(inp["logits"], K, topk_idx=idx, topk_w=wt)
    ep.ep_dispatch_layout(idx, inp["rank_offsets"], E, 0, out=lay, workspace=ws)
    ep.ep_dispatch(inp["x"], idx, lay.pos, lay.expert_offsets, E, ep.EP_LAYOUT_CONTIG, 0,
                   ep.EP_DTYPE_FP8_E4M3_B128, out=q, out_scales=qs)
    ep.ep_combine(inp["y"], idx, wt, lay.pos, lay.expert_offsets, E, ep.EP_LAYOUT_CONTIG, 0,
                  out=comb)
    torch.cuda.synchronize()
    oidx, ow = oracle.route_topk(np_(inp["logits"]), K)
    olay = oracle.layout(oidx, np_(inp["rank_offsets"]), E)
    rng = np.random.default_rng(0)
    offs = np_(inp["rank_offsets"])
    sample = np.unique(np.concatenate([rng.choice(N, 384, replace=False), offs[:-1],
                                       offs[1:] - 1]))
    return dict(w=w, inp=inp, idx=idx, wt=wt, lay=lay, q=q, qs=qs, comb=comb, oidx=oidx, ow=ow,
                olay=olay, sample=sample)


def test_fullsize_route_and_layout_every_token(prefill):
    p = prefill
    np.testing.assert_array_equal(np_(p["idx"]), p["oidx"])
    np.testing.assert_allclose(np_(p["wt"]), p["ow"], rtol=weight_rtol())
    for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
        np.testing.assert_array_equal(np_(getattr(p["lay"], name)), p["olay"][name], err_msg=name)


def test_fullsize_fp8_dispatch_sampled_rows(prefill):
    p = prefill
    s = p["sample"]
    K, E, H = p["w"].K, p["w"].E, p["w"].H
    xs = bits(p["inp"]["x"][torch.from_numpy(s).cuda()])
    S = len(s)
    local_pos = np.arange(S * K, dtype=np.int32).reshape(S, K)
    ref_q, ref_s = oracle.dispatch(xs, p["oidx"][s], local_pos, p["olay"]["expert_offsets"], E,
                                   dtype=oracle.DTYPE_FP8)
    rows = torch.from_numpy(p["olay"]["pos"][s].reshape(-1).astype(np.int64)).cuda()
    np.testing.assert_array_equal(np_(p["q"][rows]), ref_q)
    np.testing.assert_array_equal(np_(p["qs"][rows]).view(np.uint32), ref_s.view(np.uint32))


def test_fullsize_combine_sampled_tokens(prefill):
    p = prefill
    s = p["sample"]
    K, E, H = p["w"].K, p["w"].E, p["w"].H
    S = len(s)
    rows = torch.from_numpy(p["olay"]["pos"][s].reshape(-1).astype(np.int64)).cuda()
    ys = bits(p["inp"]["y"][rows])                      # the rows these tokens read
    local_pos = np.arange(S * K, dtype=np.int32).reshape(S, K)
    eoff = p["olay"]["expert_offsets"]
    # same inputs on both sides (the oracle's weights): bit-exact, within 1e-3
    ow_dev = torch.from_numpy(p["ow"]).cuda()
    got = ep.ep_combine(p["inp"]["y"], p["idx"], ow_dev, p["lay"].pos, p["lay"].expert_offsets, E)
    torch.cuda.synchronize()
    ref = oracle.combine(ys, p["oidx"][s], p["ow"][s], local_pos, eoff, E)
    g = bits(got[torch.from_numpy(s).cuda()])
    assert combine_rel_err(g, ref) <= 1e-3
    np.testing.assert_array_equal(g, ref)
    # the bench's own output (GPU weights): within one bf16 unit plus the
    # weight-difference bound
    gc = bits(p["comb"][torch.from_numpy(s).cuda()])
    gf = (gc.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    of = (ref.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    yf = np.abs((ys.astype(np.uint32) << 16).view(np.float32).astype(np.float64)).reshape(S, K, H)
    T = (np.abs(p["ow"][s].astype(np.float64))[..., None] * yf).sum(1)
    bound = bf16_ulp(of) + (weight_rtol() + 2 * K * 2.0 ** -24) * T
    assert np.all(np.abs(gf - of) <= bound * 1.0001)


def test_fullsize_host_pipeline_equals_device_path(prefill):
    """The bench's end-to-end schedule at full size: HostPipeline steps over
    page-locked huge-page host buffers (ep_host_alloc), copies overlapped
    across steps.  Its results equal the device path's (checked above against
    the oracle on sampled tokens) bit for bit, as do its dispatched FP8 rows
    and layout."""
    from combine_ep_route_topk_gb300 import pipeline as pl
    p = prefill
    w, inp = p["w"], p["inp"]
    N, E, K, H, R = inp["N"], w.E, w.K, w.H, w.R

    def host(t):
        h = pl.host_empty(tuple(t.shape), t.dtype)
        h.copy_(t)
        return h
    x_h, lg_h, ro_h, y_h = (host(inp[k]) for k in ("x", "logits", "rank_offsets", "y"))
    outs = [pl.host_empty((N, H), torch.bfloat16) for _ in range(2)]
    hp = pl.HostPipeline(N, E, K, H, R, ep.EP_DTYPE_FP8_E4M3_B128)
    for out_h in outs:
        hp.step(x_h, lg_h, ro_h, y_h, out_h)
    hp.synchronize()
    comb = p["comb"].cpu()
    for out_h in outs:
        assert torch.equal(out_h, comb)
    assert torch.equal(hp.out, p["q"])
    assert torch.equal(hp.scales, p["qs"])
    for name in ("counts", "expert_offsets", "pos", "row_src"):
        assert torch.equal(getattr(hp.layout, name), getattr(p["lay"], name)), name
