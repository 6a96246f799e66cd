"""Seeded synthetic workloads for the EP route / layout / dispatch / combine path.

This module only draws random inputs; it holds none of the method's
arithmetic (no routing, counting, quantisation or reduction), so the CUDA
library and the CPU oracle can both consume exactly the same tensors.

Shapes follow the source pages' workloads:
  toy      "Anatomy of a High-Performance EP Kernel", "What we have to do":
           8 ranks, one token each, E = 16 experts (2 per rank), K = 2
  lumpy    the same 16-expert setup with per-rank batches B_i and a
           per-expert logit bias, so that some experts draw no tokens (the
           page's figure notes four of sixteen experts idle in one step)
  decode   DeepSeek-R1 shape from "21K output tokens/s DeepSeek inference on
           MI300X", "Parallelization method": 256 experts, 8 active, DP8/EP8
           (32 experts per rank); H = 7168; masked layout, capacity 128
  prefill  same model shape, 8 x 4096 tokens, FP8 E4M3 1x128 contiguous
  skew     128 experts, K = 4, H = 2880, Zipf(1.2) expert popularity,
           experts renumbered by the balanced partition of the same report's
           "Load balancing across GPUs" section
The serving benchmark the pages measure on (ShareGPT prompts through a full
server) is not used: these synthetic tensors stand in for it.

Draw order from one torch.Generator seeded with ``seed``:
B_i, per-expert bias, logits, x, y.  On ``device='cuda'`` the same recipe
runs on the CUDA generator (different numbers, same distributions): both
implementations always consume the very same tensors, wherever drawn.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

LAYOUT_CONTIG = 0
LAYOUT_MASKED = 1
DTYPE_BF16 = 0
DTYPE_FP8 = 1


@dataclass(frozen=True)
class Workload:
    name: str
    R: int                  # logical data-parallel ranks
    E: int                  # experts (E / R per rank)
    K: int                  # experts per token
    H: int                  # hidden size
    batch: tuple            # ("fixed", B) | ("uniform", lo, hi) | ("uniform_to_total", lo, hi, total)
    bias: str = "none"      # "none" | "normal1.5" | "zipf1.2"
    layout: int = LAYOUT_CONTIG
    dtype: int = DTYPE_BF16
    cap: int = 0            # masked capacity per expert (0: contiguous only)
    relabel: bool = False   # renumber experts by the balanced partition

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "toy": Workload("toy", R=8, E=16, K=2, H=128, batch=("fixed", 1), cap=8),
    "lumpy": Workload("lumpy", R=8, E=16, K=2, H=1024, batch=("uniform", 64, 256),
                      bias="normal1.5"),
    "decode": Workload("decode", R=8, E=256, K=8, H=7168, batch=("fixed", 128),
                       layout=LAYOUT_MASKED, cap=128),
    "prefill": Workload("prefill", R=8, E=256, K=8, H=7168, batch=("fixed", 4096),
                        dtype=DTYPE_FP8),
    "skew": Workload("skew", R=8, E=128, K=4, H=2880,
                     batch=("uniform_to_total", 1024, 3072, 16384), bias="zipf1.2",
                     relabel=True),
}


def _batch_sizes(w: Workload, g: torch.Generator) -> list:
    kind = w.batch[0]
    if kind == "fixed":
        return [w.batch[1]] * w.R
    lo, hi = w.batch[1], w.batch[2]
    b = torch.randint(lo, hi + 1, (w.R,), generator=g, device=g.device).cpu().tolist()
    if kind == "uniform":
        return b
    # rescale to an exact total: floor shares, remainder to the largest
    # fractional parts (ties: lower rank)
    total = w.batch[3]
    s = sum(b)
    q = [bi * total // s for bi in b]
    rem = [bi * total % s for bi in b]
    left = total - sum(q)
    order = sorted(range(w.R), key=lambda r: (-rem[r], r))
    for r in order[:left]:
        q[r] += 1
    return q


def _bias(w: Workload, g: torch.Generator) -> torch.Tensor | None:
    if w.bias == "none":
        return None
    if w.bias == "normal1.5":
        return torch.randn(w.E, generator=g, device=g.device, dtype=torch.float32) * 1.5
    if w.bias == "zipf1.2":
        # popularity rank j_e in 1..E; log-probability bias -1.2 ln j_e
        j = torch.randperm(w.E, generator=g, device=g.device).to(torch.float32) + 1.0
        return -1.2 * torch.log(j)
    raise ValueError(w.bias)


def _randn_bf16(shape, g: torch.Generator, chunk_rows: int = 4096) -> torch.Tensor:
    """N(0,1) drawn in float32 row chunks, rounded to bf16."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=g.device)
    flat = out.view(-1, shape[-1]) if len(shape) > 1 else out.view(1, -1)
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=g.device,
                                  dtype=torch.float32).to(torch.bfloat16)
    return out


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu", with_y: bool = True) -> dict:
    """Returns rank_offsets int32 [R+1], logits float32 [N,E], x bf16 [N,H]
    and (with_y) y bf16 expert outputs: [N*K, H] for the contiguous layout,
    [E, cap, H] for the masked one."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B = _batch_sizes(w, g)
    offs = [0]
    for b in B:
        offs.append(offs[-1] + b)
    N = offs[-1]
    bias = _bias(w, g)
    logits = torch.randn((N, w.E), generator=g, device=device, dtype=torch.float32)
    if bias is not None:
        logits += bias
    x = _randn_bf16((N, w.H), g)
    out = dict(workload=w, seed=seed, B=B, N=N,
               rank_offsets=torch.tensor(offs, dtype=torch.int32, device=device),
               logits=logits, x=x)
    if with_y:
        if w.layout == LAYOUT_CONTIG:
            out["y"] = _randn_bf16((N * w.K, w.H), g)
        else:
            out["y"] = _randn_bf16((w.E, w.cap, w.H), g)
    return out


def masked_cap_overflow(N: int, K: int, E: int) -> int:
    """A capacity 25% above the mean per-expert load: exercises overflow on
    lumpy routing."""
    return int(math.ceil(1.25 * N * K / E))
