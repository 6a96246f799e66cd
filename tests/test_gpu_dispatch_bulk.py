"""Dispatch from 4096 tokens on, where each destination row is written by a
bulk shared-to-global copy, against the oracle (rows, FP8 codes and scales
bit-exact), and against the thread-store kernels (EP_DISPATCH_BULK=0).

Cases: ragged ranks, both layouts with capacity drops, bf16 and FP8, rows
from 16 bytes up to the 32 KB staging limit, and rows above it (thread
stores at every size)."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_route_topk_gb300 import (EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3_B128, EP_LAYOUT_CONTIG,
                                         EP_LAYOUT_MASKED, ep_dispatch)

from _util import bits, np_

pytestmark = pytest.mark.gpu

BF16, FP8 = EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3_B128
CONTIG, MASKED = EP_LAYOUT_CONTIG, EP_LAYOUT_MASKED


def _problem(seed, B, E, K, H, cap):
    g = np.random.default_rng(seed)
    N = int(sum(B))
    offs = np.concatenate([[0], np.cumsum(B)]).astype(np.int32)
    logits = g.standard_normal((N, E)).astype(np.float32)
    x = torch.from_numpy(g.standard_normal((N, H)).astype(np.float32)).to(torch.bfloat16)
    idx, _ = oracle.route_topk(logits, K)
    lay = oracle.layout(idx, offs, E, cap)
    return x, idx, lay


def _gpu(x, idx, lay, E, layout, cap, dtype, rows):
    """Dispatch into a buffer pre-filled with 0xFF bytes; returns (its bytes,
    the scales)."""
    N, H = x.shape
    row_bytes = H * (2 if dtype == BF16 else 1)
    buf = torch.full((rows * row_bytes,), 0xFF, dtype=torch.uint8, device="cuda")
    out = buf.view(torch.bfloat16).view(rows, H) if dtype == BF16 else buf.view(rows, H)
    sc = torch.full((rows, H // 128), -1.0, device="cuda") if dtype == FP8 else None
    ep_dispatch(x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(lay["pos"]).cuda(),
                torch.from_numpy(lay["expert_offsets"]).cuda(), E, layout, cap, dtype,
                out=out, out_scales=sc)
    torch.cuda.synchronize()
    return np_(buf).copy(), (None if sc is None else np_(sc).copy())


def _check(x, idx, lay, E, layout, cap, dtype, monkeypatch):
    N, H = x.shape
    K = idx.shape[1]
    rows = N * K if layout == CONTIG else E * cap
    if dtype == BF16:
        ref = np.full((rows, H), 0xFFFF, np.uint16)
        ref_s = None
    else:
        ref = np.full((rows, H), 0xFF, np.uint8)
        ref_s = np.full((rows, H // 128), -1.0, np.float32)
    oracle.dispatch(bits(x), idx, lay["pos"], lay["expert_offsets"], E, layout=layout, cap=cap,
                    dtype=dtype, out=ref, out_scales=ref_s)
    monkeypatch.delenv("EP_DISPATCH_BULK", raising=False)
    got, got_s = _gpu(x, idx, lay, E, layout, cap, dtype, rows)
    monkeypatch.setenv("EP_DISPATCH_BULK", "0")
    thr, thr_s = _gpu(x, idx, lay, E, layout, cap, dtype, rows)
    monkeypatch.delenv("EP_DISPATCH_BULK")
    np.testing.assert_array_equal(got, ref.reshape(-1).view(np.uint8))
    np.testing.assert_array_equal(thr, got)
    if dtype == FP8:
        np.testing.assert_array_equal(got_s.view(np.uint32), ref_s.view(np.uint32))
        np.testing.assert_array_equal(thr_s.view(np.uint32), got_s.view(np.uint32))


@pytest.mark.parametrize("B,E,K,H,layout,cap,dtype", [
    ([600, 0, 1000, 1, 999, 1496], 256, 8, 7168, CONTIG, 0, FP8),   # 4096 tokens, the prefill shape
    ([600, 0, 1000, 1, 999, 1496], 256, 8, 7168, CONTIG, 0, BF16),
    ([2050, 2051], 128, 4, 2880, CONTIG, 0, BF16),                  # the skew shape, H % 128 != 0
    ([4100], 64, 2, 128, MASKED, 100, FP8),                          # one scale per row, drops
    ([1024] * 4 + [7], 256, 8, 1024, MASKED, 130, BF16),            # drops
    ([3000, 1097], 16, 2, 8, CONTIG, 0, BF16),                       # 16-byte rows
    ([2048, 2048], 32, 2, 16384, CONTIG, 0, BF16),                  # 32 KB rows: the staging limit
    ([4096], 8, 2, 16384, MASKED, 900, FP8),                         # 16 KB codes, drops
    ([4096], 1024, 32, 256, CONTIG, 0, BF16),                       # K = 32 copies per token, E = 1024
    ([4096], 64, 4, 512, MASKED, 1, FP8),                           # capacity 1: almost all dropped
    ([2000, 2096], 4, 4, 32896, CONTIG, 0, FP8),                    # 32,896-byte codes: thread stores
])
def test_bulk_dispatch_matches_oracle_and_thread_stores(B, E, K, H, layout, cap, dtype,
                                                        monkeypatch):
    x, idx, lay = _problem(sum(B) + E + K + H, B, E, K, H, cap)
    _check(x, idx, lay, E, layout, cap, dtype, monkeypatch)


def test_rows_above_the_staging_limit_take_thread_stores(monkeypatch):
    x, idx, lay = _problem(6, [4096], 16, 2, 16392, 0)  # 32784-byte bf16 rows
    _check(x, idx, lay, 16, CONTIG, 0, BF16, monkeypatch)


def _kernel_names(fn):
    """Names of the dispatch kernels fn launches.  The first profiler session
    of a process can come back empty while the profiler starts up, so an
    empty capture is taken once more."""
    from torch.profiler import ProfilerActivity, profile
    for _ in range(2):
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if "dispatch" in e.name]
        if names:
            return names
    return []


@pytest.mark.parametrize("N,env,expect", [(4096, None, "bulk"), (4095, None, "thread"),
                                          (4096, "0", "thread")])
def test_which_dispatch_kernel_runs(N, env, expect, monkeypatch):
    """The bulk-copy kernels run from 4096 tokens on unless EP_DISPATCH_BULK=0
    (kernel names from the CUDA profiler)."""
    x, idx, lay = _problem(9, [N], 16, 2, 256, 0)
    if env is None:
        monkeypatch.delenv("EP_DISPATCH_BULK", raising=False)
    else:
        monkeypatch.setenv("EP_DISPATCH_BULK", env)
    xd, idd = x.cuda(), torch.from_numpy(idx).cuda()
    pos, eo = torch.from_numpy(lay["pos"]).cuda(), torch.from_numpy(lay["expert_offsets"]).cuda()
    names = _kernel_names(lambda: ep_dispatch(xd, idd, pos, eo, 16, CONTIG, 0, FP8))
    if not names:
        pytest.skip("the CUDA profiler recorded no kernels here")
    assert len(names) == 1, names
    assert ("bulk" in names[0]) == (expect == "bulk"), names
