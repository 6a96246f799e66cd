"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Integer and byte work (top-K ids, counts, offsets, permutation, dispatched
bf16 rows, FP8 codes and scales) must be bit-exact.  Gate weights are float
(tolerance derived in _util.weight_rtol).  Combine must be within relative
error 1e-3 (absolute floor 1e-2 for outputs near zero) when both sides get
the same inputs; it is in fact expected bit-exact, because both run the same
fp32 FMA chain in pick order.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_route_topk_gb300 import (EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3_B128, EP_LAYOUT_CONTIG,
                                         EP_LAYOUT_MASKED, ep_combine, ep_dispatch,
                                         ep_dispatch_layout, ep_expert_balance_map, ep_route_topk)
from combine_ep_route_topk_gb300 import workloads as wl

from _util import bf16_ulp, bits, combine_rel_err, from_bits, np_, weight_rtol

pytestmark = pytest.mark.gpu

COMBINE_RTOL = 1e-3


def _small(name):
    """The workload at a size the oracle finishes in seconds."""
    w = wl.WORKLOADS[name]
    if name == "prefill":  # 8 ranks x ~256 tokens, ragged
        return w.scaled(batch=("uniform", 200, 300))
    return w


def _check_layout(gpu, ref, cap):
    np.testing.assert_array_equal(np_(gpu.counts), ref["counts"])
    np.testing.assert_array_equal(np_(gpu.expert_offsets), ref["expert_offsets"])
    np.testing.assert_array_equal(np_(gpu.rank_expert_offsets), ref["rank_expert_offsets"])
    np.testing.assert_array_equal(np_(gpu.pos), ref["pos"])
    np.testing.assert_array_equal(np_(gpu.row_src), ref["row_src"])
    if cap > 0:
        np.testing.assert_array_equal(np_(gpu.masked_m), ref["masked_m"])
        assert int(np_(gpu.overflow_count)[0]) == ref["overflow"]


# ---------------------------------------------------------------- routing ---

def test_worked_example_on_gpu():
    import test_oracle
    logits, picks = test_oracle._read_worked_example()
    idx, w = ep_route_topk(torch.from_numpy(logits).cuda(), 2)
    np.testing.assert_array_equal(np_(idx), picks)
    ref_idx, ref_w = oracle.route_topk(logits, 2)
    np.testing.assert_allclose(np_(w), ref_w, rtol=weight_rtol())


@pytest.mark.parametrize("E,K", [(16, 2), (16, 16), (100, 7), (128, 4), (128, 8), (256, 4),
                                 (256, 8), (256, 2), (384, 8), (512, 32), (1024, 8), (33, 1),
                                 (1, 1)])
def test_route_topk_random(E, K):
    g = torch.Generator().manual_seed(E * 7 + K)
    N = 777  # ragged against the 8-token blocks
    logits = torch.randn(N, E, generator=g)
    idx, w = ep_route_topk(logits.cuda(), K)
    ref_idx, ref_w = oracle.route_topk(logits.numpy(), K)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_allclose(np_(w), ref_w, rtol=weight_rtol())


@pytest.mark.parametrize("E,K", [(16, 2), (128, 4), (256, 8), (100, 5)])
def test_route_topk_ties_and_signed_zero(E, K):
    rng = np.random.default_rng(E + K)
    vals = rng.choice(np.array([-1.0, -0.0, 0.0, 0.25, 1.0], np.float32), size=(300, E))
    idx, w = ep_route_topk(torch.from_numpy(vals).cuda(), K)
    ref_idx, ref_w = oracle.route_topk(vals, K)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_allclose(np_(w), ref_w, rtol=weight_rtol())


def test_route_topk_expert_map():
    g = torch.Generator().manual_seed(12)
    logits = torch.randn(500, 128, generator=g)
    emap = torch.randperm(128, generator=g).to(torch.int32)
    idx, w = ep_route_topk(logits.cuda(), 4, expert_map=emap.cuda())
    ref_idx, ref_w = oracle.route_topk(logits.numpy(), 4, expert_map=emap.numpy())
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_allclose(np_(w), ref_w, rtol=weight_rtol())


@pytest.mark.parametrize("E,K", [(128, 4), (256, 8), (1024, 8)])
def test_route_topk_logits_not_16_byte_aligned(E, K):
    """Logits that start 4 bytes past a 16-byte boundary (legal: 4-byte
    aligned) take the scalar-load kernels; same picks and weights."""
    g = torch.Generator().manual_seed(E + K)
    N = 203
    flat = torch.randn(N * E + 1, generator=g)
    dev = flat.cuda()
    logits = dev[1:].view(N, E)
    assert logits.data_ptr() % 16 == 4
    idx, w = ep_route_topk(logits, K)
    ref_idx, ref_w = oracle.route_topk(flat[1:].view(N, E).numpy(), K)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_allclose(np_(w), ref_w, rtol=weight_rtol())


@pytest.mark.parametrize("N", [1, 2, 15, 17])
def test_route_topk_few_tokens(N):
    """Fewer tokens than one block serves (one or two tokens per warp)."""
    g = torch.Generator().manual_seed(N)
    logits = torch.randn(N, 256, generator=g)
    idx, w = ep_route_topk(logits.cuda(), 8)
    ref_idx, ref_w = oracle.route_topk(logits.numpy(), 8)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_allclose(np_(w), ref_w, rtol=weight_rtol())


def test_route_topk_empty_batch():
    idx, w = ep_route_topk(torch.empty(0, 16, device="cuda"), 2)
    torch.cuda.synchronize()
    assert idx.shape == (0, 2)


# ----------------------------------------------------------------- layout ---

@pytest.fixture(params=["small", "cluster", "kernels"])
def layout_path(request, monkeypatch):
    """The layout's three implementations: one block per expert (problems up
    to 16384 picks, the default there), one thread-block cluster (the same
    sizes with at most 64 ranks whose chunk rows fit in shared memory, when
    the first is off: EP_LAYOUT_SMALL=0) and the three kernels (every size;
    forced with EP_LAYOUT_CLUSTER=0).  Sizes a path does not serve fall to
    the next one."""
    monkeypatch.delenv("EP_LAYOUT_CLUSTER", raising=False)
    monkeypatch.delenv("EP_LAYOUT_SMALL", raising=False)
    if request.param == "kernels":
        monkeypatch.setenv("EP_LAYOUT_CLUSTER", "0")
    elif request.param == "cluster":
        monkeypatch.setenv("EP_LAYOUT_SMALL", "0")
    return request.param


@pytest.mark.parametrize("name,seed", [("toy", 0), ("lumpy", 0), ("lumpy", 1), ("lumpy", 2),
                                       ("lumpy", 3), ("lumpy", 4), ("decode", 0), ("prefill", 0),
                                       ("skew", 0)])
def test_layout_parity(name, seed, layout_path):
    w = _small(name)
    inp = wl.make_inputs(w, seed=seed, with_y=False)
    idx, _ = oracle.route_topk(inp["logits"].numpy(), w.K)
    for cap in sorted({0, w.cap, wl.masked_cap_overflow(inp["N"], w.K, w.E)}):
        ref = oracle.layout(idx, inp["rank_offsets"].numpy(), w.E, cap)
        gpu = ep_dispatch_layout(torch.from_numpy(idx).cuda(), inp["rank_offsets"].cuda(), w.E,
                                 cap)
        _check_layout(gpu, ref, cap)


@pytest.mark.parametrize("B,E,K,cap", [
    ([0, 5, 0, 0, 37, 0, 1, 0], 16, 2, 3),      # empty ranks
    ([0, 0, 0, 0], 8, 2, 1),                     # N = 0
    ([70], 8, 1, 4),                             # one rank, K = 1
    ([33] * 64, 1024, 32, 2),                    # E = 1024, K = 32, many ranks
    ([1] * 1024, 64, 4, 100),                    # R = 1024
    ([5000, 1, 3000], 256, 8, 64),               # chunks > 32 tokens, ragged
    ([125] * 8, 1024, 8, 16),                    # E = 1024: 90 KB of shared memory per CTA
    ([64] * 8, 1024, 32, 40),                    # 16384 picks: the largest one-launch case
    ([2048, 1], 16, 8, 2000),                    # just over it: the three kernels
    ([16] * 64, 64, 4, 3),                       # 64 ranks: the widest one-cluster chunk table
    ([0, 3] * 32 + [5], 32, 2, 1),               # 65 ranks, empty ones: the three kernels
    ([1] * 1024, 16, 2, 1),                      # R = 1024 with one-token ranks
])
def test_layout_edge_cases(B, E, K, cap, layout_path):
    g = torch.Generator().manual_seed(len(B) * E + K)
    N = sum(B)
    offs = np.concatenate([[0], np.cumsum(B)]).astype(np.int32)
    logits = torch.randn(N, E, generator=g).numpy()
    idx, _ = oracle.route_topk(logits, K) if N else (np.zeros((0, K), np.int32), None)
    ref = oracle.layout(idx, offs, E, cap)
    gpu = ep_dispatch_layout(torch.from_numpy(idx).cuda(), torch.from_numpy(offs).cuda(), E, cap)
    _check_layout(gpu, ref, cap)


def test_worked_example_layout_on_gpu(layout_path):
    """The CUDA layout of the worked table's routes equals the values derived
    by hand from the pages (no oracle in between)."""
    import test_oracle
    g = test_oracle.read_worked_layout()
    ro = torch.arange(5, dtype=torch.int32, device="cuda")
    lay = ep_dispatch_layout(torch.from_numpy(g["picks"]).cuda(), ro, 16)
    np.testing.assert_array_equal(np_(lay.expert_offsets), g["expert_offsets"])
    np.testing.assert_array_equal(np_(lay.pos), g["pos"])
    np.testing.assert_array_equal(np_(lay.row_src), g["row_src"])
    np.testing.assert_array_equal(np_(lay.counts), g["counts"])
    np.testing.assert_array_equal(np_(lay.rank_expert_offsets), g["rank_expert_offsets"])
    masked = ep_dispatch_layout(torch.from_numpy(g["picks"]).cuda(), ro, 16, 1)
    np.testing.assert_array_equal(np_(masked.masked_m), g["cap1_masked_m"])
    assert int(np_(masked.overflow_count)[0]) == g["cap1_overflow"][0]


def test_layout_all_tokens_one_expert_and_invalid_ids(layout_path):
    N, E, K = 300, 16, 2
    idx = np.zeros((N, K), np.int32)
    idx[:, 1] = np.arange(N) % E
    idx[idx[:, 1] == 0, 1] = -1          # "no pick"
    idx[7, 1] = 99                       # out of range: also "no pick"
    offs = np.array([0, 100, 100, 250, N], np.int32)
    cap = 40
    ref = oracle.layout(idx, offs, E, cap)
    assert ref["overflow"] > 0
    gpu = ep_dispatch_layout(torch.from_numpy(idx).cuda(), torch.from_numpy(offs).cuda(), E, cap)
    _check_layout(gpu, ref, cap)


@pytest.mark.parametrize("B,E,K,small,cluster", [
    ([128] * 8, 256, 8, 1, 1),        # the decode shape
    ([64] * 8, 1024, 32, 1, 1),       # 16384 picks
    ([2048, 1], 16, 8, 3, 3),         # 16392 picks: three kernels
    ([16] * 64, 64, 4, 1, 1),         # 64 ranks
    ([16] * 65, 65, 4, 1, 3),         # 65 ranks: too many for one cluster
    ([1] * 1024, 64, 4, 1, 3),        # 1024 ranks
    ([4096] * 8, 256, 8, 3, 3),       # the prefill shape
])
def test_layout_path_choice(B, E, K, small, cluster, monkeypatch):
    """Which implementation serves a size (launches per layout call): by
    default, with the one-block-per-expert path off, and with the three
    kernels forced."""
    from combine_ep_route_topk_gb300 import ep as epb
    monkeypatch.delenv("EP_LAYOUT_CLUSTER", raising=False)
    monkeypatch.delenv("EP_LAYOUT_SMALL", raising=False)
    N = sum(B)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(B)]), dtype=torch.int32, device="cuda")
    idx = torch.zeros(N, K, dtype=torch.int32, device="cuda")
    for env, expect in ((None, small), (("EP_LAYOUT_SMALL", "0"), cluster),
                        (("EP_LAYOUT_CLUSTER", "0"), 3)):
        if env:
            monkeypatch.setenv(*env)
        before = epb.lib().ep_kernel_launch_count()
        ep_dispatch_layout(idx, offs, E)
        assert epb.lib().ep_kernel_launch_count() - before == expect, env
    torch.cuda.synchronize()


# --------------------------------------------------------------- dispatch ---

def _dispatch_both(x_t, idx, lay, E, layout, cap, dtype):
    N, H = x_t.shape
    K = idx.shape[1]
    rows = N * K if layout == EP_LAYOUT_CONTIG else E * cap
    if dtype == EP_DTYPE_BF16:
        ref_out = np.full((rows, H), 0xFFFF, np.uint16)
        gpu_out = torch.full((rows, H), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        ref_s, gpu_s = None, None
    else:
        ref_out = np.full((rows, H), 0xFF, np.uint8)
        gpu_out = torch.full((rows, H), 0xFF, dtype=torch.uint8, device="cuda")
        ref_s = np.full((rows, H // 128), -1.0, np.float32)
        gpu_s = torch.full((rows, H // 128), -1.0, device="cuda")
    oracle.dispatch(bits(x_t), idx, lay["pos"], lay["expert_offsets"], E, layout=layout, cap=cap,
                    dtype=dtype, out=ref_out, out_scales=ref_s)
    ep_dispatch(x_t.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(lay["pos"]).cuda(),
                torch.from_numpy(lay["expert_offsets"]).cuda(), E, layout, cap, dtype,
                out=gpu_out, out_scales=gpu_s)
    if dtype == EP_DTYPE_BF16:
        np.testing.assert_array_equal(bits(gpu_out), ref_out)
    else:
        np.testing.assert_array_equal(np_(gpu_out), ref_out)
        np.testing.assert_array_equal(np_(gpu_s).view(np.uint32), ref_s.view(np.uint32))


@pytest.mark.parametrize("name", ["toy", "lumpy", "decode", "prefill", "skew"])
@pytest.mark.parametrize("layout", [EP_LAYOUT_CONTIG, EP_LAYOUT_MASKED])
@pytest.mark.parametrize("dtype", [EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3_B128])
def test_dispatch_parity(name, layout, dtype):
    w = _small(name)
    if dtype == EP_DTYPE_FP8_E4M3_B128 and w.H % 128:
        pytest.skip("FP8 needs H % 128 == 0")
    inp = wl.make_inputs(w, seed=0, with_y=False)
    idx, _ = oracle.route_topk(inp["logits"].numpy(), w.K)
    cap = 0
    if layout == EP_LAYOUT_MASKED:
        cap = w.cap if w.cap > 0 else wl.masked_cap_overflow(inp["N"], w.K, w.E)
    lay = oracle.layout(idx, inp["rank_offsets"].numpy(), w.E, cap)
    _dispatch_both(inp["x"], idx, lay, w.E, layout, cap, dtype)


def test_fp8_encoding_exhaustive_on_gpu():
    """Every finite bf16 value with |v| <= 448, in 128-column blocks whose
    first element is 448 (so amax = 448, scale = 1 and the code is E4M3(v)),
    against the oracle's encoder."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_to_float(allb)
    keep = allb[np.isfinite(v) & (np.abs(v) <= 448.0)]
    per = 127
    nrow = (len(keep) + per - 1) // per
    blocks = np.zeros((nrow, 128), np.uint16)
    blocks[:, 0] = oracle.float_to_bf16(np.array([448.0], np.float32))[0]
    flat = np.zeros(nrow * per, np.uint16)
    flat[:len(keep)] = keep
    blocks[:, 1:] = flat.reshape(nrow, per)
    H = 1024
    N = (nrow + 7) // 8
    xb = np.zeros((N * 8, 128), np.uint16)
    xb[:nrow] = blocks
    x = from_bits(xb.reshape(N, H), "cpu")
    idx = np.zeros((N, 1), np.int32)
    lay = oracle.layout(idx, np.array([0, N], np.int32), 1)
    _dispatch_both(x, idx, lay, 1, EP_LAYOUT_CONTIG, 0, EP_DTYPE_FP8_E4M3_B128)


# ---------------------------------------------------------------- combine ---

def _combine_both(y_t, idx, wts, lay, E, layout, cap):
    ref = oracle.combine(bits(y_t), idx, wts, lay["pos"], lay["expert_offsets"], E, layout=layout,
                         cap=cap)
    got = ep_combine(y_t.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(wts).cuda(),
                     torch.from_numpy(lay["pos"]).cuda(),
                     torch.from_numpy(lay["expert_offsets"]).cuda(), E, layout, cap)
    return bits(got), ref


@pytest.mark.parametrize("name", ["toy", "lumpy", "decode", "prefill", "skew"])
def test_combine_parity(name):
    w = _small(name)
    inp = wl.make_inputs(w, seed=0)
    idx, wts = oracle.route_topk(inp["logits"].numpy(), w.K)
    cap = w.cap if w.layout == EP_LAYOUT_MASKED else 0
    lay = oracle.layout(idx, inp["rank_offsets"].numpy(), w.E, cap)
    got, ref = _combine_both(inp["y"], idx, wts, lay, w.E, w.layout, cap)
    assert combine_rel_err(got, ref) <= COMBINE_RTOL
    np.testing.assert_array_equal(got, ref)  # same FMA chain: bit-exact


def test_combine_masked_with_overflow_and_runtime_k():
    w = wl.WORKLOADS["lumpy"].scaled(K=3, H=256)
    inp = wl.make_inputs(w, seed=3, with_y=False)
    idx, wts = oracle.route_topk(inp["logits"].numpy(), w.K)
    cap = wl.masked_cap_overflow(inp["N"], w.K, w.E)
    lay = oracle.layout(idx, inp["rank_offsets"].numpy(), w.E, cap)
    assert lay["overflow"] > 0
    g = torch.Generator().manual_seed(5)
    y = torch.randn(w.E * cap, w.H, generator=g).to(torch.bfloat16)
    got, ref = _combine_both(y, idx, wts, lay, w.E, EP_LAYOUT_MASKED, cap)
    assert combine_rel_err(got, ref) <= COMBINE_RTOL
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("H,dtype", [(8, EP_DTYPE_BF16), (136, EP_DTYPE_BF16),
                                     (16392, EP_DTYPE_BF16), (128, EP_DTYPE_FP8_E4M3_B128),
                                     (16512, EP_DTYPE_FP8_E4M3_B128)])
@pytest.mark.parametrize("layout", [EP_LAYOUT_CONTIG, EP_LAYOUT_MASKED])
def test_dispatch_combine_hidden_sizes(H, dtype, layout):
    """Smallest rows (one 16-byte vector, one scale block) and rows longer
    than one pass of a block (several column passes with a ragged last one,
    in dispatch and in combine)."""
    g = torch.Generator().manual_seed(H + layout)
    B, E, K = [9, 0, 28], 16, 3
    N = sum(B)
    offs = np.concatenate([[0], np.cumsum(B)]).astype(np.int32)
    idx, wts = oracle.route_topk(torch.randn(N, E, generator=g).numpy(), K)
    cap = 5 if layout == EP_LAYOUT_MASKED else 0
    lay = oracle.layout(idx, offs, E, cap)
    x = (torch.randn(N, H, generator=g) * 3).to(torch.bfloat16)
    _dispatch_both(x, idx, lay, E, layout, cap, dtype)
    rows = N * K if layout == EP_LAYOUT_CONTIG else E * cap
    y = torch.randn(rows, H, generator=g).to(torch.bfloat16)
    got, ref = _combine_both(y, idx, wts, lay, E, layout, cap)
    np.testing.assert_array_equal(got, ref)


# ----------------------------------------------------- whole path, on GPU ---

def _gpu_chain(inp, w, layout, cap, dtype, emap=None):
    d = {}
    idx, wt = ep_route_topk(inp["logits"].cuda(), w.K, expert_map=emap)
    lay = ep_dispatch_layout(idx, inp["rank_offsets"].cuda(), w.E, cap)
    out, sc = ep_dispatch(inp["x"].cuda(), idx, lay.pos, lay.expert_offsets, w.E, layout, cap,
                          dtype)
    comb = ep_combine(inp["y"].cuda(), idx, wt, lay.pos, lay.expert_offsets, w.E, layout, cap)
    torch.cuda.synchronize()
    return dict(idx=idx, w=wt, lay=lay, out=out, scales=sc, comb=comb)


def _oracle_chain(inp, w, layout, cap, dtype, emap=None):
    idx, wt = oracle.route_topk(inp["logits"].numpy(), w.K, expert_map=emap)
    lay = oracle.layout(idx, inp["rank_offsets"].numpy(), w.E, cap)
    out, sc = oracle.dispatch(bits(inp["x"]), idx, lay["pos"], lay["expert_offsets"], w.E,
                              layout=layout, cap=cap, dtype=dtype)
    yb = bits(inp["y"])
    comb = oracle.combine(yb, idx, wt, lay["pos"], lay["expert_offsets"], w.E,
                          layout=layout, cap=cap)
    return dict(idx=idx, w=wt, lay=lay, out=out, scales=sc, comb=comb, y=yb)


def _compare_chain(g, o, w, layout, cap, dtype):
    np.testing.assert_array_equal(np_(g["idx"]), o["idx"])
    np.testing.assert_allclose(np_(g["w"]), o["w"], rtol=weight_rtol())
    _check_layout(g["lay"], o["lay"], cap)
    if layout == EP_LAYOUT_MASKED:  # rows past masked_m are unspecified
        H = w.H
        gm = (bits(g["out"]) if dtype == EP_DTYPE_BF16 else np_(g["out"])).reshape(w.E, cap, H)
        om = o["out"].reshape(w.E, cap, H)
        for e in range(w.E):
            m = o["lay"]["masked_m"][e]
            np.testing.assert_array_equal(gm[e, :m], om[e, :m])
    elif dtype == EP_DTYPE_BF16:
        np.testing.assert_array_equal(bits(g["out"]), o["out"])
    else:
        np.testing.assert_array_equal(np_(g["out"]), o["out"])
        np.testing.assert_array_equal(np_(g["scales"]), o["scales"])
    # combine with each side's own weights: the weights differ by float ulps
    # (relative weight_rtol), so the two fp32 sums differ by at most
    # (weight_rtol + 2 K 2^-24) * T with T = sum_k |w_k| |y_k|, and the bf16
    # roundings by one more unit; nearly all outputs are identical
    gc, oc = bits(g["comb"]), o["comb"]
    gf = (gc.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    of = (oc.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    T = _abs_weighted_sum(o["y"], o["idx"], o["w"], o["lay"], w.E, layout, cap)
    bound = bf16_ulp(of) + (weight_rtol() + 2 * w.K * 2.0 ** -24) * T
    assert np.all(np.abs(gf - of) <= bound * 1.0001)
    assert np.mean(gc == oc) > 0.999


def _abs_weighted_sum(y_bits, idx, wts, lay, E, layout, cap):
    """T[t, h] = sum_k |w[t,k]| * |y[row(t,k), h]| over delivered picks."""
    N, K = idx.shape
    yf = np.abs((y_bits.reshape(-1, y_bits.shape[-1]).astype(np.uint32) << 16)
                .view(np.float32).astype(np.float64))
    T = np.zeros((N, yf.shape[1]))
    pos = lay["pos"]
    for k in range(K):
        p = pos[:, k].astype(np.int64)
        e = idx[:, k].astype(np.int64)
        ok = (p >= 0) & (e >= 0) & (e < E)
        if layout == EP_LAYOUT_CONTIG:
            row = p
        else:
            slot = p - lay["expert_offsets"][np.clip(e, 0, E - 1)]
            ok &= (slot >= 0) & (slot < cap)
            row = e * cap + slot
        T[ok] += np.abs(wts[ok, k].astype(np.float64))[:, None] * yf[row[ok]]
    return T


@pytest.mark.parametrize("name", ["toy", "lumpy", "decode", "prefill", "skew"])
def test_whole_path_parity(name):
    w = _small(name)
    inp = wl.make_inputs(w, seed=1)
    cap = w.cap if w.layout == EP_LAYOUT_MASKED else 0
    g = _gpu_chain(inp, w, w.layout, cap, w.dtype)
    o = _oracle_chain(inp, w, w.layout, cap, w.dtype)
    _compare_chain(g, o, w, w.layout, cap, w.dtype)


def test_skew_relabel_chain():
    """Balanced renumbering on the same batch's counts, then the renumbered
    route, layout, dispatch and combine: map and ids bit-exact."""
    w = wl.WORKLOADS["skew"]
    inp = wl.make_inputs(w, seed=0)
    idx0, _ = ep_route_topk(inp["logits"].cuda(), w.K)
    lay0 = ep_dispatch_layout(idx0, inp["rank_offsets"].cuda(), w.E)
    emap = ep_expert_balance_map(lay0.counts, )
    oidx0, _ = oracle.route_topk(inp["logits"].numpy(), w.K)
    olay0 = oracle.layout(oidx0, inp["rank_offsets"].numpy(), w.E)
    oemap = oracle.balance_map(olay0["counts"])
    np.testing.assert_array_equal(np_(emap), oemap)
    g = _gpu_chain(inp, w, EP_LAYOUT_CONTIG, 0, EP_DTYPE_BF16, emap=emap)
    o = _oracle_chain(inp, w, EP_LAYOUT_CONTIG, 0, EP_DTYPE_BF16, emap=oemap)
    _compare_chain(g, o, w, EP_LAYOUT_CONTIG, 0, EP_DTYPE_BF16)
    # the renumbering balances the per-rank expert load
    per = w.E // w.R
    naive = olay0["counts"].sum(0).reshape(w.R, per).sum(1)
    bal = o["lay"]["counts"].sum(0).reshape(w.R, per).sum(1)
    assert bal.max() <= naive.max()


@pytest.mark.parametrize("E,R", [(8, 2), (16, 8), (256, 8), (1024, 1024), (1024, 4), (12, 3)])
def test_balance_map_parity(E, R):
    rng = np.random.default_rng(E + R)
    counts = rng.integers(0, 1000, size=(R, E)).astype(np.int32)
    counts[:, rng.integers(0, E, size=E // 4)] = 0
    got = ep_expert_balance_map(torch.from_numpy(counts).cuda())
    np.testing.assert_array_equal(np_(got), oracle.balance_map(counts))


def test_identity_experts_round_trip():
    """combine(dispatch(x)) == x under identity experts (weights sum to 1)."""
    w = wl.WORKLOADS["lumpy"]
    inp = wl.make_inputs(w, seed=4, with_y=False)
    x = inp["x"].cuda()
    idx, wt = ep_route_topk(inp["logits"].cuda(), w.K)
    for layout, cap in [(EP_LAYOUT_CONTIG, 0), (EP_LAYOUT_MASKED, inp["N"] * w.K)]:
        lay = ep_dispatch_layout(idx, inp["rank_offsets"].cuda(), w.E, cap)
        y, _ = ep_dispatch(x, idx, lay.pos, lay.expert_offsets, w.E, layout, cap)
        back = ep_combine(y, idx, wt, lay.pos, lay.expert_offsets, w.E, layout, cap)
        assert torch.equal(back.view(torch.int16), x.view(torch.int16))


def test_cuda_graph_capture_masked_decode():
    """route -> layout -> masked dispatch -> combine captured once in a CUDA
    graph (static shapes, no host reads) and replayed on new logits."""
    w = wl.WORKLOADS["decode"].scaled(H=512)
    inp = wl.make_inputs(w, seed=0)
    N, E, K, cap = inp["N"], w.E, w.K, w.cap
    logits = inp["logits"].cuda()
    ro = inp["rank_offsets"].cuda()
    x = inp["x"].cuda()
    y = inp["y"].cuda()
    idx = torch.empty(N, K, dtype=torch.int32, device="cuda")
    wt = torch.empty(N, K, device="cuda")
    from combine_ep_route_topk_gb300 import alloc_layout, ep_dispatch_layout_workspace_size
    lay = alloc_layout(N, E, K, w.R, cap, "cuda")
    ws = torch.empty(ep_dispatch_layout_workspace_size(N, E, K, w.R), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(E * cap, w.H, dtype=torch.bfloat16, device="cuda")
    comb = torch.empty(N, w.H, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def step():
        ep_route_topk(logits, K, topk_idx=idx, topk_w=wt)
        ep_dispatch_layout(idx, ro, E, cap, out=lay, workspace=ws)
        ep_dispatch(x, idx, lay.pos, lay.expert_offsets, E, EP_LAYOUT_MASKED, cap, out=out)
        ep_combine(y, idx, wt, lay.pos, lay.expert_offsets, E, EP_LAYOUT_MASKED, cap, out=comb)

    with torch.cuda.stream(s):
        step()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (11, 12):
        new = wl.make_inputs(w, seed=seed, with_y=False)["logits"]
        logits.copy_(new.cuda())
        graph.replay()
        torch.cuda.synchronize()
        o = _oracle_chain(dict(inp, logits=new), w, EP_LAYOUT_MASKED, cap, EP_DTYPE_BF16)
        g = dict(idx=idx, w=wt, lay=lay, out=out, scales=None, comb=comb)
        _compare_chain(g, o, w, EP_LAYOUT_MASKED, cap, EP_DTYPE_BF16)


@pytest.mark.parametrize("per_rank", [100, 600])  # one-launch layout / three kernels
def test_cuda_graph_capture_contiguous_fp8(per_rank):
    """route -> layout -> FP8 contiguous dispatch -> combine captured once in
    a CUDA graph and replayed on new logits, tokens and expert outputs copied
    into the captured buffers; every replay matches the oracle."""
    w = wl.WORKLOADS["prefill"].scaled(batch=("fixed", per_rank), H=1024)
    inp = wl.make_inputs(w, seed=0)
    N, E, K, R = inp["N"], w.E, w.K, w.R
    logits, ro = inp["logits"].cuda(), inp["rank_offsets"].cuda()
    x, y = inp["x"].cuda(), inp["y"].cuda()
    idx = torch.empty(N, K, dtype=torch.int32, device="cuda")
    wt = torch.empty(N, K, device="cuda")
    from combine_ep_route_topk_gb300 import alloc_layout, ep_dispatch_layout_workspace_size
    lay = alloc_layout(N, E, K, R, 0, "cuda")
    ws = torch.empty(ep_dispatch_layout_workspace_size(N, E, K, R), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(N * K, w.H, dtype=torch.uint8, device="cuda")
    sc = torch.empty(N * K, w.H // 128, device="cuda")
    comb = torch.empty(N, w.H, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def step():
        ep_route_topk(logits, K, topk_idx=idx, topk_w=wt)
        ep_dispatch_layout(idx, ro, E, 0, out=lay, workspace=ws)
        ep_dispatch(x, idx, lay.pos, lay.expert_offsets, E, EP_LAYOUT_CONTIG, 0,
                    EP_DTYPE_FP8_E4M3_B128, out=out, out_scales=sc)
        ep_combine(y, idx, wt, lay.pos, lay.expert_offsets, E, EP_LAYOUT_CONTIG, 0, out=comb)

    with torch.cuda.stream(s):
        step()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (21, 22):
        new = wl.make_inputs(w, seed=seed)
        # same rank sizes: the captured rank offsets stay valid
        assert torch.equal(new["rank_offsets"], inp["rank_offsets"])
        logits.copy_(new["logits"].cuda())
        x.copy_(new["x"].cuda())
        y.copy_(new["y"].cuda())
        graph.replay()
        torch.cuda.synchronize()
        o = _oracle_chain(new, w, EP_LAYOUT_CONTIG, 0, EP_DTYPE_FP8_E4M3_B128)
        g = dict(idx=idx, w=wt, lay=lay, out=out, scales=sc, comb=comb)
        _compare_chain(g, o, w, EP_LAYOUT_CONTIG, 0, EP_DTYPE_FP8_E4M3_B128)


def test_concurrent_host_threads_on_their_own_streams():
    """Two host threads run the whole path on their own streams and inputs at
    the same time, several times over: every result equals the one the same
    inputs give alone (the library keeps no shared state on this path)."""
    import threading
    cases = []
    for name, seed in (("lumpy", 1), ("skew", 2)):
        w = wl.WORKLOADS[name]
        inp = wl.make_inputs(w, seed=seed)
        g = _gpu_chain(inp, w, EP_LAYOUT_CONTIG, 0, EP_DTYPE_BF16)
        cases.append((w, {k: v.cuda() for k, v in inp.items() if torch.is_tensor(v)},
                      {k: (v.clone() if torch.is_tensor(v) else v) for k, v in g.items()}))
    errors = []

    def worker(w, dev_inp, ref):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(5):
                    idx, wt = ep_route_topk(dev_inp["logits"], w.K)
                    lay = ep_dispatch_layout(idx, dev_inp["rank_offsets"], w.E)
                    out, _ = ep_dispatch(dev_inp["x"], idx, lay.pos, lay.expert_offsets, w.E)
                    comb = ep_combine(dev_inp["y"], idx, wt, lay.pos, lay.expert_offsets, w.E)
                    s.synchronize()
                    assert torch.equal(idx, ref["idx"]) and torch.equal(wt, ref["w"])
                    assert torch.equal(lay.pos, ref["lay"].pos)
                    assert torch.equal(out.view(torch.int16), ref["out"].view(torch.int16))
                    assert torch.equal(comb.view(torch.int16), ref["comb"].view(torch.int16))
        except Exception as exc:  # reported on the main thread
            errors.append(repr(exc))

    threads = [threading.Thread(target=worker, args=c) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
