"""Seeded random configurations of the whole path against the CPU oracle,
stage by stage, so that no stage's inputs come from the CUDA path:
  - route: random E, K (E not a multiple of 32, odd K, K = E), ties;
  - layout: random ranks (empty ones, up to 70), capacities, some picks
    invalid or duplicated within a token, on the three layout implementations
    (one block per expert, one cluster, three kernels);
  - dispatch: bf16 or FP8 rows, contiguous or masked, from the oracle's layout;
  - combine: from the oracle's weights and layout, bit-exact.
Sizes are small so that the oracle finishes in seconds, except for the
dispatch cases at 4096 to 6000 tokens (the bulk-copy kernels)."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_route_topk_gb300 import (EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3_B128, EP_LAYOUT_CONTIG,
                                         EP_LAYOUT_MASKED, ep_combine, ep_dispatch,
                                         ep_dispatch_layout, ep_route_topk)

from _util import bits, np_, weight_rtol

pytestmark = pytest.mark.gpu


def _config(rng):
    K = int(rng.integers(1, 33))
    E = int(rng.integers(K, 300)) if rng.random() < 0.8 else K
    R = int(rng.integers(1, 71))
    B = rng.integers(0, 41, size=R)
    B[rng.random(R) < 0.2] = 0  # some empty ranks
    fp8 = rng.random() < 0.4
    H = int(rng.choice([128, 256, 384])) if fp8 else 8 * int(rng.integers(1, 66))
    masked = rng.random() < 0.4
    cap = int(rng.integers(1, 12)) if masked else 0
    return E, K, R, B, H, fp8, masked, cap


@pytest.mark.parametrize("seed", range(200))
def test_random_configuration(seed, monkeypatch):
    rng = np.random.default_rng(1000 + seed)
    E, K, R, B, H, fp8, masked, cap = _config(rng)
    N = int(B.sum())
    offs = np.concatenate([[0], np.cumsum(B)]).astype(np.int32)
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(N, E, generator=g)
    if rng.random() < 0.3:  # coarse values: many exact ties
        logits = torch.round(logits * 2) / 2
    x = (torch.randn(N, H, generator=g) * 4).to(torch.bfloat16)
    layout = EP_LAYOUT_MASKED if masked else EP_LAYOUT_CONTIG
    dtype = EP_DTYPE_FP8_E4M3_B128 if fp8 else EP_DTYPE_BF16

    # route
    oidx, ow = oracle.route_topk(logits.numpy(), K)
    idx, w = ep_route_topk(logits.cuda(), K)
    np.testing.assert_array_equal(np_(idx), oidx)
    np.testing.assert_allclose(np_(w), ow, rtol=weight_rtol())

    # Downstream stages take the oracle's picks, in about a third of the cases
    # with some made invalid (-1, E or beyond: "no pick") or duplicated within
    # their token, which the layout, dispatch and combine must handle too.
    if rng.random() < 0.35 and N:
        oidx = oidx.copy()
        hit = rng.random(oidx.shape) < 0.1
        choice = rng.integers(0, 3, size=oidx.shape)
        bad = np.where(choice == 0, -1, np.where(choice == 1, E, E + 7)).astype(np.int32)
        dup = np.repeat(oidx[:, :1], K, axis=1)
        oidx = np.where(hit & (choice < 2), bad, oidx)
        oidx = np.where(hit & (choice == 2), dup, oidx).astype(np.int32)

    # layout of those picks, both implementations
    olay = oracle.layout(oidx, offs, E, cap)
    for path in ("small", "cluster", "kernels"):
        monkeypatch.delenv("EP_LAYOUT_CLUSTER", raising=False)
        monkeypatch.delenv("EP_LAYOUT_SMALL", raising=False)
        if path == "kernels":
            monkeypatch.setenv("EP_LAYOUT_CLUSTER", "0")
        elif path == "cluster":
            monkeypatch.setenv("EP_LAYOUT_SMALL", "0")
        lay = ep_dispatch_layout(torch.from_numpy(oidx).cuda(), torch.from_numpy(offs).cuda(),
                                 E, cap)
        for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
            np.testing.assert_array_equal(np_(getattr(lay, name)), olay[name],
                                          err_msg=f"{name} ({path})")
        if cap:
            np.testing.assert_array_equal(np_(lay.masked_m), olay["masked_m"])
            assert int(np_(lay.overflow_count)[0]) == olay["overflow"]
    monkeypatch.delenv("EP_LAYOUT_CLUSTER", raising=False)
    monkeypatch.delenv("EP_LAYOUT_SMALL", raising=False)

    # dispatch from the oracle's layout
    pos_d = torch.from_numpy(olay["pos"]).cuda()
    eoff_d = torch.from_numpy(olay["expert_offsets"]).cuda()
    idx_d = torch.from_numpy(oidx).cuda()
    oout, osc = oracle.dispatch(bits(x), oidx, olay["pos"], olay["expert_offsets"], E,
                                layout=layout, cap=cap, dtype=dtype)
    out, sc = ep_dispatch(x.cuda(), idx_d, pos_d, eoff_d, E, layout, cap, dtype)
    got = bits(out) if dtype == EP_DTYPE_BF16 else np_(out)
    if masked:  # rows past masked_m are unspecified
        gm, om = got.reshape(E, cap, H), oout.reshape(E, cap, H)
        for e in range(E):
            m = olay["masked_m"][e]
            np.testing.assert_array_equal(gm[e, :m], om[e, :m])
            if fp8:
                np.testing.assert_array_equal(
                    np_(sc).reshape(E, cap, -1)[e, :m].view(np.uint32),
                    osc.reshape(E, cap, -1)[e, :m].view(np.uint32))
    else:  # rows past the delivered ones (invalid picks) are never written
        n = int(olay["expert_offsets"][E])
        np.testing.assert_array_equal(got[:n], oout[:n])
        if fp8:
            np.testing.assert_array_equal(np_(sc)[:n].view(np.uint32), osc[:n].view(np.uint32))

    # combine of random expert outputs with the oracle's weights and layout
    rows = N * K if not masked else E * cap
    y = torch.randn(rows, H, generator=g).to(torch.bfloat16)
    ocomb = oracle.combine(bits(y), oidx, ow, olay["pos"], olay["expert_offsets"], E,
                           layout=layout, cap=cap)
    comb = ep_combine(y.cuda(), idx_d, torch.from_numpy(ow).cuda(), pos_d, eoff_d, E, layout,
                      cap)
    np.testing.assert_array_equal(bits(comb), ocomb)


@pytest.mark.parametrize("seed", range(80))
def test_random_fused_route_layout(seed):
    """ep_route_layout (one cooperative kernel where an instance exists, else
    route + layout) on random sizes, including E of 128 / 256 / 512 / 1024
    (16-byte loads) and the scalar instances, against the oracle's route
    then layout; the status word stays 0."""
    from combine_ep_route_topk_gb300 import ep_route_layout
    rng = np.random.default_rng(5000 + seed)
    K = int(rng.integers(1, 33))
    E = int(rng.choice([128, 256, 512, 1024])) if rng.random() < 0.5 else \
        int(rng.integers(K, 300))
    E = max(E, K)
    R = int(rng.integers(1, 71))
    B = rng.integers(0, 60, size=R)
    B[rng.random(R) < 0.2] = 0
    cap = int(rng.integers(1, 12)) if rng.random() < 0.4 else 0
    N = int(B.sum())
    offs = np.concatenate([[0], np.cumsum(B)]).astype(np.int32)
    g = torch.Generator().manual_seed(7000 + seed)
    logits = torch.randn(N, E, generator=g)
    if rng.random() < 0.3:
        logits = torch.round(logits * 2) / 2
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    idx, w, lay = ep_route_layout(logits.cuda(), torch.from_numpy(offs).cuda(), K, cap,
                                  status=status)
    torch.cuda.synchronize()
    oidx, ow = oracle.route_topk(logits.numpy(), K)
    olay = oracle.layout(oidx, offs, E, cap)
    np.testing.assert_array_equal(np_(idx), oidx)
    np.testing.assert_allclose(np_(w), ow, rtol=weight_rtol())
    for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
        np.testing.assert_array_equal(np_(getattr(lay, name)), olay[name], err_msg=name)
    if cap:
        np.testing.assert_array_equal(np_(lay.masked_m), olay["masked_m"])
        assert int(np_(lay.overflow_count)[0]) == olay["overflow"]
    assert int(status.item()) == 0  # the call completed (fused or two kernels)


@pytest.mark.parametrize("seed", range(60))
def test_random_balance_map_and_expert_map(seed):
    """Balanced renumbering on random count matrices (ties, idle experts,
    counts near the int32 limit, frequencies past 2^32) equals the oracle's
    greedy; routing through
    a random map with some out-of-range entries gives the oracle's picks."""
    from combine_ep_route_topk_gb300 import ep_expert_balance_map
    rng = np.random.default_rng(9000 + seed)
    R = int(rng.choice([1, 2, 3, 4, 8, 16, 32, 64, 1024]))
    E = R * int(rng.integers(1, max(2, 1024 // R) + 1))
    E = min(E, 1024 - (1024 % R))
    kind = seed % 4
    if kind == 0:
        counts = rng.integers(0, 1000, size=(R, E))
    elif kind == 1:  # few distinct values: many frequency ties
        counts = rng.integers(0, 3, size=(R, E)) * 5
    elif kind == 2:  # large counts: totals near the int32 limit
        counts = rng.integers(0, (2 ** 31 - 1) // max(1, R), size=(R, E))
    else:  # every count near the int32 limit: frequencies up to R * 2^31
        counts = rng.integers(2 ** 31 - 64, 2 ** 31, size=(R, E))
    counts = counts.astype(np.int32)
    counts[:, rng.random(E) < 0.2] = 0
    got = ep_expert_balance_map(torch.from_numpy(counts).cuda())
    np.testing.assert_array_equal(np_(got), oracle.balance_map(counts))

    K = int(rng.integers(1, min(E, 32) + 1))
    emap = rng.permutation(E).astype(np.int32)
    emap[rng.random(E) < 0.05] = E + 3  # out of range: those picks become "no pick"
    g = torch.Generator().manual_seed(9000 + seed)
    logits = torch.randn(97, E, generator=g)
    idx, w = ep_route_topk(logits.cuda(), K, expert_map=torch.from_numpy(emap).cuda())
    oidx, ow = oracle.route_topk(logits.numpy(), K, expert_map=emap)
    np.testing.assert_array_equal(np_(idx), oidx)
    np.testing.assert_allclose(np_(w), ow, rtol=weight_rtol())


@pytest.mark.parametrize("seed", range(60))
def test_random_route_dispatch(seed):
    """ep_route_dispatch (two launches up to 2048 tokens and 16384 picks,
    else route + layout + dispatch) on random sizes, layouts, dtypes and
    expert maps (some entries out of range), against the oracle's route,
    layout and dispatch: every output bit-exact, weights within tolerance."""
    from combine_ep_route_topk_gb300 import ep_route_dispatch
    rng = np.random.default_rng(11000 + seed)
    K = int(rng.integers(1, 17))
    E = int(rng.choice([128, 256, 512])) if rng.random() < 0.5 else int(rng.integers(K, 300))
    E = max(E, K)
    R = int(rng.integers(1, 40))
    B = rng.integers(0, 3000 // R + 1, size=R)  # up to about 3000 tokens: both sides of 2048
    B[rng.random(R) < 0.2] = 0
    N = int(B.sum())
    offs = np.concatenate([[0], np.cumsum(B)]).astype(np.int32)
    fp8 = rng.random() < 0.4
    H = int(rng.choice([128, 256])) if fp8 else 8 * int(rng.integers(1, 40))
    masked = rng.random() < 0.5
    cap = int(rng.integers(1, 3 * max(1, N * K // E) + 2)) if masked else \
        (int(rng.integers(1, 8)) if rng.random() < 0.3 else 0)
    layout = EP_LAYOUT_MASKED if masked else EP_LAYOUT_CONTIG
    dtype = EP_DTYPE_FP8_E4M3_B128 if fp8 else EP_DTYPE_BF16
    emap = None
    if rng.random() < 0.3:
        emap = rng.permutation(E).astype(np.int32)
        emap[rng.random(E) < 0.05] = -1
    g = torch.Generator().manual_seed(11000 + seed)
    logits = torch.randn(N, E, generator=g)
    if rng.random() < 0.3:
        logits = torch.round(logits * 2) / 2
    x = (torch.randn(N, H, generator=g) * 4).to(torch.bfloat16)

    idx, w, lay, out, sc = ep_route_dispatch(
        logits.cuda(), torch.from_numpy(offs).cuda(), x.cuda(), K, layout, cap, dtype,
        expert_map=None if emap is None else torch.from_numpy(emap).cuda())
    torch.cuda.synchronize()
    oidx, ow = oracle.route_topk(logits.numpy(), K, expert_map=emap) if N else \
        (np.zeros((0, K), np.int32), np.zeros((0, K), np.float32))
    np.testing.assert_array_equal(np_(idx), oidx)
    np.testing.assert_allclose(np_(w), ow, rtol=weight_rtol())
    olay = oracle.layout(oidx, offs, E, cap)
    for name in ("counts", "expert_offsets", "rank_expert_offsets", "pos", "row_src"):
        np.testing.assert_array_equal(np_(getattr(lay, name)), olay[name], err_msg=name)
    if cap:
        np.testing.assert_array_equal(np_(lay.masked_m), olay["masked_m"])
        assert int(np_(lay.overflow_count)[0]) == olay["overflow"]
    oout, osc = oracle.dispatch(bits(x), oidx, olay["pos"], olay["expert_offsets"], E,
                                layout=layout, cap=cap, dtype=dtype)
    got = bits(out) if dtype == EP_DTYPE_BF16 else np_(out)
    if masked:  # rows past masked_m are unspecified
        gm, om = got.reshape(E, cap, H), oout.reshape(E, cap, H)
        for e in range(E):
            m = olay["masked_m"][e]
            np.testing.assert_array_equal(gm[e, :m], om[e, :m])
            if fp8:
                np.testing.assert_array_equal(np_(sc).reshape(E, cap, -1)[e, :m],
                                              osc.reshape(E, cap, -1)[e, :m])
    else:  # rows past the valid picks are not written
        nv = olay["expert_offsets"][E]
        np.testing.assert_array_equal(got[:nv], oout[:nv])
        if fp8:
            np.testing.assert_array_equal(np_(sc)[:nv], osc[:nv])


@pytest.mark.parametrize("seed", range(100))
def test_random_bulk_dispatch(seed):
    """Dispatch at 4096 to 6000 tokens, where each destination row leaves
    shared memory in one bulk copy: random E, K, H, ranks, capacity, bf16 or
    FP8, some picks invalid or duplicated, from the oracle's layout, against
    the oracle's rows (and scales)."""
    rng = np.random.default_rng(9000 + seed)
    K = int(rng.integers(1, 17))
    E = int(rng.integers(K, 300))
    R = int(rng.integers(1, 17))
    N = int(rng.integers(4096, 6001))
    cuts = np.sort(rng.integers(0, N + 1, size=R - 1))
    offs = np.concatenate([[0], cuts, [N]]).astype(np.int32)
    fp8 = rng.random() < 0.5
    H = 128 * int(rng.integers(1, 9)) if fp8 else 8 * int(rng.integers(1, 257))
    masked = rng.random() < 0.4
    cap = int(rng.integers(1, 2 * N * K // E + 2)) if masked else 0
    layout = EP_LAYOUT_MASKED if masked else EP_LAYOUT_CONTIG
    dtype = EP_DTYPE_FP8_E4M3_B128 if fp8 else EP_DTYPE_BF16
    g = torch.Generator().manual_seed(9500 + seed)
    oidx, _ = oracle.route_topk(torch.randn(N, E, generator=g).numpy(), K)
    if rng.random() < 0.35:
        oidx = oidx.copy()
        hit = rng.random(oidx.shape) < 0.05
        oidx[hit] = rng.choice(np.array([-1, E], np.int32), size=int(hit.sum()))
    x = (torch.randn(N, H, generator=g) * 4).to(torch.bfloat16)
    olay = oracle.layout(oidx, offs, E, cap)
    oout, osc = oracle.dispatch(bits(x), oidx, olay["pos"], olay["expert_offsets"], E,
                                layout=layout, cap=cap, dtype=dtype)
    out, sc = ep_dispatch(x.cuda(), torch.from_numpy(oidx).cuda(),
                          torch.from_numpy(olay["pos"]).cuda(),
                          torch.from_numpy(olay["expert_offsets"]).cuda(), E, layout, cap, dtype)
    got = bits(out) if dtype == EP_DTYPE_BF16 else np_(out)
    if masked:  # rows past masked_m are unspecified
        gm, om = got.reshape(E, cap, H), oout.reshape(E, cap, H)
        for e in range(E):
            m = olay["masked_m"][e]
            np.testing.assert_array_equal(gm[e, :m], om[e, :m])
            if fp8:
                np.testing.assert_array_equal(
                    np_(sc).reshape(E, cap, -1)[e, :m].view(np.uint32),
                    osc.reshape(E, cap, -1)[e, :m].view(np.uint32))
    else:
        n = int(olay["expert_offsets"][E])
        np.testing.assert_array_equal(got[:n], oout[:n])
        if fp8:
            np.testing.assert_array_equal(np_(sc)[:n].view(np.uint32), osc[:n].view(np.uint32))
