"""Repeatability: the whole path run 100 times on the same inputs gives the
same bits every time.  No position depends on the order of atomics, and the
fused kernel's and the cluster layout's barriers order every phase; a race
would show as a difference between repetitions."""
import pytest
import torch

from combine_ep_route_topk_gb300 import (EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3_B128, EP_LAYOUT_CONTIG,
                                         EP_LAYOUT_MASKED, ep_combine, ep_dispatch,
                                         ep_dispatch_layout, ep_route_layout, ep_route_topk)
from combine_ep_route_topk_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _run(inp, w, layout, cap, dtype, fused):
    logits, ro = inp["logits"], inp["rank_offsets"]
    if fused:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        idx, wt, lay = ep_route_layout(logits, ro, w.K, cap, status=status)
    else:
        status = None
        idx, wt = ep_route_topk(logits, w.K)
        lay = ep_dispatch_layout(idx, ro, w.E, cap)
    out, sc = ep_dispatch(inp["x"], idx, lay.pos, lay.expert_offsets, w.E, layout, cap, dtype)
    comb = ep_combine(inp["y"], idx, wt, lay.pos, lay.expert_offsets, w.E, layout, cap)
    res = [idx, wt, lay.counts, lay.expert_offsets, lay.rank_expert_offsets, lay.pos,
           lay.row_src, comb]
    if layout == EP_LAYOUT_CONTIG:  # every masked row past masked_m is unspecified
        res += [out] + ([sc] if sc is not None else [])
    else:
        res += [lay.masked_m, lay.overflow_count]
    if status is not None:
        res.append(status)
    return res


@pytest.mark.parametrize("name,layout,dtype,fused,small", [
    ("prefill", EP_LAYOUT_CONTIG, EP_DTYPE_FP8_E4M3_B128, False, True),  # three layout kernels
    ("decode", EP_LAYOUT_MASKED, EP_DTYPE_BF16, False, True),    # one block per expert
    ("decode", EP_LAYOUT_MASKED, EP_DTYPE_BF16, False, False),   # one-cluster layout
    ("decode", EP_LAYOUT_MASKED, EP_DTYPE_BF16, True, True),     # cooperative kernel
])
def test_hundred_repetitions_are_bit_identical(name, layout, dtype, fused, small, monkeypatch):
    monkeypatch.delenv("EP_LAYOUT_CLUSTER", raising=False)
    if small:
        monkeypatch.delenv("EP_LAYOUT_SMALL", raising=False)
    else:
        monkeypatch.setenv("EP_LAYOUT_SMALL", "0")
    w = wl.WORKLOADS[name]
    if name == "prefill":
        w = w.scaled(batch=("fixed", 600), H=1024)
    cap = w.cap if layout == EP_LAYOUT_MASKED else 0
    inp = {k: (v.cuda() if torch.is_tensor(v) else v)
           for k, v in wl.make_inputs(w, seed=3).items()}
    first = [t.clone() for t in _run(inp, w, layout, cap, dtype, fused)]
    for _ in range(100):
        again = _run(inp, w, layout, cap, dtype, fused)
        for a, b in zip(first, again):
            assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)
    if fused:
        assert int(first[-1].item()) == 0
