"""Schedules built from the entry points (combine_ep_route_topk_gb300.pipeline):
two-micro-batch overlap on two streams, chunked ("ant-moving") rounds with a
bounded dispatch buffer, and the native host-buffer pipeline.

Each schedule's final combined output is checked against the CPU oracle run
over the whole batch: the oracle routes, lays out and dispatches the batch,
applies the same expert stand-in on the CPU to its own dispatched rows, and
combines.  The stand-in depends only on a row's values and its expert id, so
a token's combined output does not depend on how a schedule splits the batch
into micro-batches or rounds.  Both sides use their own gate weights, which
differ by float ulps, so the bound is the whole-path one: one bf16 unit plus
(weight_rtol + 2 K 2^-24) * sum_k |w_k| |y_k| per element, with at least
99.9 % of the outputs bit-identical.  Every micro-batch / round layout must
also match the oracle bit for bit, and each schedule's output must equal the
single-batch GPU path's (per-token work is unchanged: same routing, same FMA
chain) as an extra check."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_route_topk_gb300 as ep
from combine_ep_route_topk_gb300 import pipeline as pl
from combine_ep_route_topk_gb300 import workloads as wl

from _util import bf16_ulp, bits, np_, weight_rtol

pytestmark = pytest.mark.gpu

# exact powers of two for the expert stand-in (no exp2 rounding on either side)
_POW2 = (1.0, 2.0, 4.0)


def _row_experts(lay, E):
    counts = lay.expert_offsets[1:] - lay.expert_offsets[:-1]
    return torch.repeat_interleave(torch.arange(E, device=counts.device), counts.long())


def _scaled(out, scales, lay, E, n_rows):
    """Expert stand-in: row of expert e times 2^(e % 3) (exact in bf16), after
    dequantising FP8 rows (code * block scale, one float multiply), rounded
    to bf16."""
    if scales is None:
        rows = out[:n_rows].float()
    else:
        H = out.shape[1]
        codes = out[:n_rows].view(torch.float8_e4m3fn).float().view(n_rows, H // 128, 128)
        rows = (codes * scales[:n_rows, :, None]).view(n_rows, H)
    e = _row_experts(lay, E)
    assert e.numel() == n_rows
    p2 = torch.tensor(_POW2, dtype=torch.float32, device=rows.device)[(e % 3).long()]
    return (rows * p2[:, None]).to(torch.bfloat16)


def _oracle_scaled(out, scales, eoff, E):
    """The same stand-in on the CPU, from the oracle's dispatched rows (bf16
    bit patterns, or FP8 codes and scales) in its expert-major order; the
    codes decode exactly to float, the products are single float roundings,
    and the bf16 rounding is the oracle's.  Returns bf16 bit patterns."""
    if scales is None:
        rows = oracle.bf16_to_float(out)
    else:
        n, H = out.shape
        table = oracle.fp8_e4m3_decode_table().astype(np.float32)
        rows = (table[out].reshape(n, H // 128, 128) * scales[:, :, None]).reshape(n, H)
    e = np.repeat(np.arange(E), np.diff(eoff))
    assert e.size == rows.shape[0]
    rows = rows * np.asarray(_POW2, np.float32)[e % 3][:, None]
    assert rows.dtype == np.float32
    return oracle.float_to_bf16(rows).reshape(rows.shape)


_ORACLE = {}


def _oracle_scaled_chain(name, seed, inp, K, E, dtype, emap=None):
    """Whole batch through the oracle with the CPU stand-in as the experts
    (cached per workload and seed)."""
    key = (name, seed, dtype, None if emap is None else emap.tobytes())
    if key not in _ORACLE:
        idx, wt = oracle.route_topk(inp["logits"].numpy(), K, expert_map=emap)
        lay = oracle.layout(idx, inp["rank_offsets"].numpy(), E)
        out, sc = oracle.dispatch(bits(inp["x"]), idx, lay["pos"], lay["expert_offsets"], E,
                                  dtype=dtype)
        y = _oracle_scaled(out, sc, lay["expert_offsets"], E)
        comb = oracle.combine(y, idx, wt, lay["pos"], lay["expert_offsets"], E)
        _ORACLE[key] = dict(idx=idx, w=wt, lay=lay, out=out, scales=sc, y=y, comb=comb)
    return _ORACLE[key]


def _abs_weighted_sum(y_bits, idx, wts, lay, E, layout=ep.EP_LAYOUT_CONTIG, cap=0):
    """T[t, h] = sum_k |w[t,k]| * |y[row(t,k), h]| over delivered picks."""
    N, K = idx.shape
    yf = np.abs((y_bits.reshape(-1, y_bits.shape[-1]).astype(np.uint32) << 16)
                .view(np.float32).astype(np.float64))
    T = np.zeros((N, yf.shape[1]))
    for k in range(K):
        p = lay["pos"][:, k].astype(np.int64)
        e = idx[:, k].astype(np.int64)
        ok = (p >= 0) & (e >= 0) & (e < E)
        if layout == ep.EP_LAYOUT_CONTIG:
            row = p
        else:
            slot = p - lay["expert_offsets"][np.clip(e, 0, E - 1)]
            ok &= (slot >= 0) & (slot < cap)
            row = e * cap + slot
        T[ok] += np.abs(wts[ok, k].astype(np.float64))[:, None] * yf[row[ok]]
    return T


def _assert_matches_oracle(comb, o, K, E, layout=ep.EP_LAYOUT_CONTIG, cap=0):
    """Combined output (bf16 tensor) against the oracle's, each side with its
    own gate weights: within the whole-path bound, nearly all identical."""
    gc, oc = bits(comb), o["comb"]
    assert gc.shape == oc.shape
    gf = (gc.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    of = (oc.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if "T" not in o:
        o["T"] = _abs_weighted_sum(o["y"], o["idx"], o["w"], o["lay"], E, layout, cap)
    bound = bf16_ulp(of) + (weight_rtol() + 2 * K * 2.0 ** -24) * o["T"]
    assert np.all(np.abs(gf - of) <= bound * 1.0001)
    assert np.mean(gc == oc) > 0.999


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
def test_two_batch_overlap_matches_oracle(name, dtype, groups):
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
    o = _oracle_scaled_chain(name, 5, inp, K, E, dtype)
    _assert_matches_oracle(comb, o, K, E)
    xb = bits(inp["x"])
    for mb in mbs:
        oidx = o["idx"][mb.t0:mb.t1]
        np.testing.assert_array_equal(np_(mb.idx), oidx)
        np.testing.assert_allclose(np_(mb.wt), o["w"][mb.t0:mb.t1], rtol=weight_rtol())
        olay = oracle.layout(oidx, np_(mb.ro), E)
        for nm in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
            np.testing.assert_array_equal(np_(getattr(mb.lay, nm)), olay[nm], err_msg=nm)
        oout, osc = oracle.dispatch(xb[mb.t0:mb.t1], oidx, olay["pos"], olay["expert_offsets"],
                                    E, dtype=dtype)
        got = np_(mb.out) if dtype == ep.EP_DTYPE_FP8_E4M3_B128 else bits(mb.out)
        np.testing.assert_array_equal(got, oout)
        if osc is not None:
            np.testing.assert_array_equal(np_(mb.scales), osc)
    ref = _single_batch(inp, w, dtype)
    torch.cuda.synchronize()
    assert torch.equal(comb.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("name,dtype,T", [("lumpy", ep.EP_DTYPE_BF16, 300),
                                          ("skew", ep.EP_DTYPE_BF16, 4096),
                                          ("prefill", ep.EP_DTYPE_FP8_E4M3_B128, 640)])
@pytest.mark.parametrize("sets", [1, 2, 3])
def test_chunked_rounds_match_oracle(name, dtype, T, sets):
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
    o = _oracle_scaled_chain(name, 6, inp, K, E, dtype)
    _assert_matches_oracle(comb, o, K, E)
    for t0, t1, lay in rounds:
        olay = oracle.layout(o["idx"][t0:t1], np.array(pl.round_rank_offsets(offs, t0, t1),
                                                       np.int32), E)
        for nm in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
            np.testing.assert_array_equal(np_(getattr(lay, nm)), olay[nm], err_msg=nm)
    ref = _single_batch(inp, w, dtype)
    torch.cuda.synchronize()
    assert torch.equal(comb.view(torch.int16), ref.view(torch.int16))


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


def _bf16_cpu(bits_np):
    return torch.from_numpy(np.ascontiguousarray(bits_np).view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("name,dtype", [("lumpy", ep.EP_DTYPE_BF16),
                                        ("prefill", ep.EP_DTYPE_FP8_E4M3_B128)])
def test_host_pipeline_matches_oracle(name, dtype):
    """Steps over pinned host buffers, copies overlapped across steps.  The
    expert outputs y come from the oracle (its dispatched rows through the
    CPU stand-in).  Every step's result matches the oracle's combine within
    the whole-path bound, the last step's dispatched rows (and FP8 scales)
    equal the oracle's bit for bit, and every result also equals the
    single-batch GPU path's on the same inputs (including a reused buffer
    set)."""
    w = wl.WORKLOADS[name]
    if name == "prefill":
        w = w.scaled(batch=("uniform", 200, 300))
    E, K, H = w.E, w.K, w.H
    for seed in (21, 22):  # the seeds draw different batch sizes: one pipeline each
        inp = wl.make_inputs(w, seed=seed, with_y=False)
        N = inp["N"]
        o = _oracle_scaled_chain(name, seed, inp, K, E, dtype)
        y_h = _pinned(_bf16_cpu(o["y"]))
        idx, wt = ep.ep_route_topk(inp["logits"].cuda(), K)
        lay = ep.ep_dispatch_layout(idx, inp["rank_offsets"].cuda(), E)
        single = ep.ep_combine(y_h.cuda(), idx, wt, lay.pos, lay.expert_offsets, E).cpu()
        hp = pl.HostPipeline(N, E, K, H, w.R, dtype)
        outs = [torch.empty(N, H, dtype=torch.bfloat16, pin_memory=True) for _ in range(3)]
        args = [_pinned(t) for t in (inp["x"], inp["logits"], inp["rank_offsets"])]
        for out_h in outs:
            hp.step(*args, y_h, out_h)
        hp.synchronize()
        for out_h in outs:
            _assert_matches_oracle(out_h, o, K, E)
            assert torch.equal(out_h, single)
        if dtype == ep.EP_DTYPE_BF16:
            np.testing.assert_array_equal(bits(hp.out), o["out"])
        else:
            np.testing.assert_array_equal(np_(hp.out), o["out"])
            np.testing.assert_array_equal(np_(hp.scales), o["scales"])
        for nm in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
            np.testing.assert_array_equal(np_(getattr(hp.layout, nm)), o["lay"][nm], err_msg=nm)


def test_host_pipeline_alternating_inputs():
    """Alternating two input sets of one size through a depth-2 pipeline: each
    step's result is its own inputs' (no buffer set is overwritten early),
    against the oracle and against the single-batch GPU path."""
    w = wl.WORKLOADS["lumpy"]
    E, K, H = w.E, w.K, w.H
    g = torch.Generator().manual_seed(3)
    N, R = 700, 4
    ro = torch.tensor([0, 100, 350, 351, 700], dtype=torch.int32)
    sets, refs = [], []
    for _ in range(2):
        logits = torch.randn(N, E, generator=g)
        x = torch.randn(N, H, generator=g).to(torch.bfloat16)
        y = torch.randn(N * K, H, generator=g).to(torch.bfloat16)
        oidx, ow = oracle.route_topk(logits.numpy(), K)
        olay = oracle.layout(oidx, ro.numpy(), E)
        refs.append(dict(idx=oidx, w=ow, lay=olay, y=bits(y),
                         comb=oracle.combine(bits(y), oidx, ow, olay["pos"],
                                             olay["expert_offsets"], E)))
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
        _assert_matches_oracle(o, refs[i], K, E)
        assert torch.equal(o, sets[i][4])


def test_host_pipeline_masked_with_expert_map():
    """The decode shape (masked capacity, overflow dropped) with a balanced
    renumbering map computed by the oracle from the batch's own routing:
    each step's result matches the oracle's masked combine, the delivered
    slots of the masked buffer equal the oracle's dispatch, and the result
    equals the single-batch GPU path's."""
    w = wl.WORKLOADS["decode"].scaled(batch=("uniform", 20, 60))
    E, K, H, cap = w.E, w.K, w.H, 4  # small capacity: some picks overflow
    MASKED = ep.EP_LAYOUT_MASKED
    inp = wl.make_inputs(w, seed=9, with_y=False)
    N = inp["N"]
    lg_np, ro_np = inp["logits"].numpy(), inp["rank_offsets"].numpy()
    i0, _ = oracle.route_topk(lg_np, K)
    emap_np = oracle.balance_map(oracle.layout(i0, ro_np, E)["counts"])
    oidx, ow = oracle.route_topk(lg_np, K, expert_map=emap_np)
    olay = oracle.layout(oidx, ro_np, E, cap)
    assert olay["overflow"] > 0
    g = torch.Generator().manual_seed(4)
    y = torch.randn(E, cap, H, generator=g).to(torch.bfloat16)
    oout, _ = oracle.dispatch(bits(inp["x"]), oidx, olay["pos"], olay["expert_offsets"], E,
                              layout=oracle.LAYOUT_MASKED, cap=cap)
    o = dict(idx=oidx, w=ow, lay=olay, y=bits(y),
             comb=oracle.combine(bits(y), oidx, ow, olay["pos"], olay["expert_offsets"], E,
                                 layout=oracle.LAYOUT_MASKED, cap=cap))
    emap = torch.from_numpy(emap_np).cuda()
    logits, ro = inp["logits"].cuda(), inp["rank_offsets"].cuda()
    idx, wt = ep.ep_route_topk(logits, K, expert_map=emap)
    lay = ep.ep_dispatch_layout(idx, ro, E, cap)
    single = ep.ep_combine(y.cuda(), idx, wt, lay.pos, lay.expert_offsets, E, MASKED, cap).cpu()
    hp = pl.HostPipeline(N, E, K, H, w.R, ep.EP_DTYPE_BF16, cap=cap, expert_map=emap)
    outs = [torch.empty(N, H, dtype=torch.bfloat16, pin_memory=True) for _ in range(3)]
    args = [_pinned(t) for t in (inp["x"], inp["logits"], inp["rank_offsets"], y)]
    for out_h in outs:
        hp.step(*args, out_h)
    hp.synchronize()
    for out_h in outs:
        _assert_matches_oracle(out_h, o, K, E, MASKED, cap)
        assert torch.equal(out_h, single)
    # only the delivered slots of the masked buffer are defined
    m = olay["masked_m"]
    np.testing.assert_array_equal(np_(hp.layout.masked_m), m)
    assert int(hp.layout.overflow_count.item()) == olay["overflow"]
    got = bits(hp.out).reshape(E, cap, H)
    ref = oout.reshape(E, cap, H)
    for e in range(E):
        np.testing.assert_array_equal(got[e, :m[e]], ref[e, :m[e]])


def test_host_alloc_buffers_through_the_pipeline():
    """Host buffers from ep_host_alloc (page-locked, huge-page backed) as the
    pipeline's inputs and outputs: results match the oracle, the device-timed
    copy durations of the last step are positive, and the buffers return to
    the library when dropped."""
    import gc
    w = wl.WORKLOADS["lumpy"]
    E, K, H = w.E, w.K, w.H
    inp = wl.make_inputs(w, seed=31, with_y=False)
    N = inp["N"]
    o = _oracle_scaled_chain("lumpy", 31, inp, K, E, ep.EP_DTYPE_BF16)

    def host(t):
        h = pl.host_empty(tuple(t.shape), t.dtype)
        assert h.is_pinned()
        h.copy_(t)
        return h
    args = [host(t) for t in (inp["x"], inp["logits"], inp["rank_offsets"],
                              _bf16_cpu(o["y"]))]
    outs = [pl.host_empty((N, H), torch.bfloat16) for _ in range(3)]
    hp = pl.HostPipeline(N, E, K, H, w.R, ep.EP_DTYPE_BF16)
    for out_h in outs:
        hp.step(*args, out_h)
    hp.synchronize()
    t_in, t_out = hp.copy_ms()
    assert t_in > 0 and t_out > 0
    for out_h in outs:
        _assert_matches_oracle(out_h, o, K, E)
    hp.close()
    del args, outs
    gc.collect()
