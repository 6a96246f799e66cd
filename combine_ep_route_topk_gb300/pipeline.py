"""Schedules of the EP path built from the library's entry points.

two_batch_overlap
    "21K output tokens/s DeepSeek inference on MI300X", "Computation-
    communication overlapping", and "Expert Parallelism" (SGLang docs),
    "Two-Batch Overlap": the batch is split into two micro-batches whose
    stages run on two streams, so one micro-batch's latency-bound routing and
    layout overlap the other's HBM-bound dispatch and combine.  On one GPU the
    micro-batches are the first and second half of the logical ranks; each
    has its own expert-major layout.

chunked
    "Expert Parallelism" (SGLang docs), "Ascend NPU guidance", the ant-moving
    function: a long sequence is sent in rounds of a fixed number of tokens,
    so the dispatch buffer is bounded by round_tokens * K rows instead of
    N * K.  Each round routes, lays out and dispatches its tokens, hands the
    dispatched rows to the caller's expert function, and combines the
    result into the round's slice of the output.  Given two (or more) round
    buffer sets, rounds alternate over the sets' streams, so one round's
    latency-bound routing and layout run under the previous round's
    HBM-bound dispatch and combine.

HostPipeline
    Steps whose inputs and result live in pinned host memory: the binding of
    the library's native pipeline (ep_host_pipeline_*).  Copies in, kernels
    and copies out run on three streams, and the device side of the inputs
    and the result is double-buffered, so one step's copies in overlap the
    previous step's kernels and copy out.  The host link, not HBM, bounds
    such a step.

host_empty
    A CPU tensor in the library's page-locked host memory (ep_host_alloc):
    huge-page backed, so that the host pipeline's multi-gigabyte copies do
    not slow down whenever the kernel reactivates the pages of an ordinary
    pinned buffer.

All only call the C ABI through the binding (every step runs in the
library's kernels); the host work is slicing and stream ordering.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import ep as _ep


@dataclass
class MicroBatch:
    """Views and buffers of one micro-batch (tokens [t0, t1) of the batch)."""
    t0: int
    t1: int
    logits: torch.Tensor
    x: torch.Tensor
    ro: torch.Tensor            # rank offsets relative to t0, on the device
    idx: torch.Tensor
    wt: torch.Tensor
    lay: _ep.Layout
    ws: torch.Tensor
    out: torch.Tensor           # dispatched rows (bf16 or FP8 codes)
    scales: torch.Tensor | None
    comb: torch.Tensor          # view into the combined output
    stream: torch.cuda.Stream


def split_by_ranks(rank_offsets_host, parts=2):
    """Contiguous rank groups: [(rank_lo, rank_hi)], ranks split evenly."""
    R = len(rank_offsets_host) - 1
    bounds = [round(i * R / parts) for i in range(parts + 1)]
    return [(bounds[i], bounds[i + 1]) for i in range(parts) if bounds[i] < bounds[i + 1]]


def make_micro_batches(logits, x, rank_offsets, K, dtype, comb, parts=2, rank_groups=None):
    """Buffers for `parts` micro-batches of contiguous rank groups (ranks split
    evenly), or for the groups [(rank_lo, rank_hi)] given in `rank_groups`,
    which must tile 0..R in order (an uneven split, e.g. a small first group
    whose routing and layout are the only ones not hidden under another
    micro-batch's dispatch and combine)."""
    dev = logits.device
    E = logits.shape[1]
    H = x.shape[1]
    offs = rank_offsets.cpu().tolist()
    R = len(offs) - 1
    groups = split_by_ranks(offs, parts) if rank_groups is None else list(rank_groups)
    if (not groups or groups[0][0] != 0 or groups[-1][1] != R or
            any(a[1] != b[0] for a, b in zip(groups, groups[1:])) or
            any(lo >= hi for lo, hi in groups)):
        raise ValueError(f"rank groups {groups} do not tile ranks 0..{R} in order")
    mbs = []
    for lo, hi in groups:
        t0, t1 = offs[lo], offs[hi]
        n = t1 - t0
        ro = torch.tensor([o - t0 for o in offs[lo:hi + 1]], dtype=torch.int32, device=dev)
        fp8 = dtype == _ep.EP_DTYPE_FP8_E4M3_B128
        mbs.append(MicroBatch(
            t0=t0, t1=t1, logits=logits[t0:t1], x=x[t0:t1], ro=ro,
            idx=torch.empty(n, K, dtype=torch.int32, device=dev),
            wt=torch.empty(n, K, dtype=torch.float32, device=dev),
            lay=_ep.alloc_layout(n, E, K, hi - lo, 0, dev),
            ws=torch.empty(_ep.ep_dispatch_layout_workspace_size(n, E, K, hi - lo),
                           dtype=torch.uint8, device=dev),
            out=torch.empty(n * K, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev),
            scales=torch.empty(n * K, H // 128, dtype=torch.float32, device=dev) if fp8 else None,
            comb=comb[t0:t1], stream=torch.cuda.Stream(device=dev)))
    return mbs


def two_batch_overlap(mbs, K, dtype, expert_out, main_stream=None):
    """Run route -> layout -> dispatch -> combine for every micro-batch on its
    own stream; `expert_out(mb)` returns the bf16 expert outputs [rows, H] for
    the micro-batch (called on its stream after its dispatch).  The calling
    stream waits for all micro-batches at the end."""
    main = torch.cuda.current_stream() if main_stream is None else main_stream
    for mb in mbs:
        mb.stream.wait_stream(main)
    for mb in mbs:
        with torch.cuda.stream(mb.stream):
            E = mb.logits.shape[1]
            _ep.ep_route_topk(mb.logits, K, topk_idx=mb.idx, topk_w=mb.wt)
            _ep.ep_dispatch_layout(mb.idx, mb.ro, E, 0, out=mb.lay, workspace=mb.ws)
            _ep.ep_dispatch(mb.x, mb.idx, mb.lay.pos, mb.lay.expert_offsets, E,
                            _ep.EP_LAYOUT_CONTIG, 0, dtype, out=mb.out, out_scales=mb.scales)
            y = expert_out(mb)
            _ep.ep_combine(y, mb.idx, mb.wt, mb.lay.pos, mb.lay.expert_offsets, E,
                           _ep.EP_LAYOUT_CONTIG, 0, out=mb.comb)
    for mb in mbs:
        main.wait_stream(mb.stream)


@dataclass
class ChunkBuffers:
    """Round-sized buffers: the dispatch buffer holds round_tokens * K rows.
    `stream` is the stream of the rounds that use this set when rounds
    alternate over several sets."""
    round_tokens: int
    idx: torch.Tensor
    wt: torch.Tensor
    ws: torch.Tensor
    out: torch.Tensor
    scales: torch.Tensor | None
    stream: torch.cuda.Stream | None = None

    @property
    def dispatch_bytes(self) -> int:
        b = self.out.numel() * self.out.element_size()
        if self.scales is not None:
            b += self.scales.numel() * 4
        return b


def make_chunk_buffers(round_tokens, E, K, H, R, dtype, device, sets=1):
    """One round buffer set (sets == 1), or a list of `sets` sets, each with
    its own stream, for rounds that alternate over them."""
    fp8 = dtype == _ep.EP_DTYPE_FP8_E4M3_B128
    T = round_tokens

    def one(stream):
        return ChunkBuffers(
            round_tokens=T,
            idx=torch.empty(T, K, dtype=torch.int32, device=device),
            wt=torch.empty(T, K, dtype=torch.float32, device=device),
            ws=torch.empty(_ep.ep_dispatch_layout_workspace_size(T, E, K, R), dtype=torch.uint8,
                           device=device),
            out=torch.empty(T * K, H, dtype=torch.uint8 if fp8 else torch.bfloat16,
                            device=device),
            scales=(torch.empty(T * K, H // 128, dtype=torch.float32, device=device)
                    if fp8 else None),
            stream=stream)

    if sets == 1:
        return one(None)
    return [one(torch.cuda.Stream(device=device)) for _ in range(sets)]


def round_rank_offsets(rank_offsets_host, t0, t1):
    """Rank offsets of the round [t0, t1): each rank's tokens clipped to the
    round, relative to t0 (ranks with no token in the round are empty)."""
    return [min(max(o, t0), t1) - t0 for o in rank_offsets_host]


def chunk_rank_offsets(rank_offsets_host, N, T, device):
    """Device tensor [rounds, R+1] of every round's rank offsets."""
    R = len(rank_offsets_host) - 1
    starts = list(range(0, N, T))
    return torch.tensor([round_rank_offsets(rank_offsets_host, t0, min(N, t0 + T))
                         for t0 in starts], dtype=torch.int32).reshape(len(starts),
                                                                      R + 1).to(device)


def chunked(logits, x, rank_offsets_host, K, dtype, bufs, expert_out, comb, ro_rounds=None):
    """Ant-moving rounds over the packed token sequence.  `bufs` is one
    ChunkBuffers (rounds in order on the current stream) or a list of them
    (make_chunk_buffers(..., sets=n)): round j then uses set j mod n on that
    set's stream, and the current stream waits for every round at the end.
    `expert_out(t0, n, out_rows, scales, layout)` returns the bf16 expert
    outputs [n*K, H] of the round's dispatched rows (called on the round's
    stream).  Results land in comb[t0:t1] for each round.  `ro_rounds`
    (chunk_rank_offsets) may be passed to skip the upload.  Returns
    [(t0, t1, layout)] per round (the layouts for inspection)."""
    sets = list(bufs) if isinstance(bufs, (list, tuple)) else [bufs]
    N, E = logits.shape
    T = sets[0].round_tokens
    starts = list(range(0, N, T))
    # every round's rank offsets in one upload, before the first launch
    ro_all = ro_rounds if ro_rounds is not None else \
        chunk_rank_offsets(rank_offsets_host, N, T, logits.device)
    main = torch.cuda.current_stream(logits.device)
    multi = len(sets) > 1
    if multi:
        for b in sets:
            if b.stream is None:
                raise ValueError("alternating rounds need buffer sets with streams "
                                 "(make_chunk_buffers(..., sets=n))")
            b.stream.wait_stream(main)
    rounds = []
    for j, t0 in enumerate(starts):
        b = sets[j % len(sets)]
        t1 = min(N, t0 + T)
        n = t1 - t0
        with torch.cuda.stream(b.stream if multi else main):
            ro = ro_all[j]
            idx, wt = b.idx[:n], b.wt[:n]
            _ep.ep_route_topk(logits[t0:t1], K, topk_idx=idx, topk_w=wt)
            lay = _ep.ep_dispatch_layout(idx, ro, E, 0, workspace=b.ws)
            out = b.out[:n * K]
            scales = None if b.scales is None else b.scales[:n * K]
            _ep.ep_dispatch(x[t0:t1], idx, lay.pos, lay.expert_offsets, E, _ep.EP_LAYOUT_CONTIG,
                            0, dtype, out=out, out_scales=scales)
            y = expert_out(t0, n, out, scales, lay)
            _ep.ep_combine(y, idx, wt, lay.pos, lay.expert_offsets, E, _ep.EP_LAYOUT_CONTIG, 0,
                           out=comb[t0:t1])
        rounds.append((t0, t1, lay))
    if multi:
        for b in sets:
            main.wait_stream(b.stream)
    return rounds


def host_empty(shape, dtype):
    """Uninitialised CPU tensor of `shape` and `dtype` in page-locked,
    huge-page-backed host memory from ep_host_alloc (include/ep.h).  Copies
    to and from it run asynchronously, like those of torch's pinned memory.
    The memory returns to the library (ep_host_free) when the last tensor
    that views it is gone."""
    import ctypes
    import math
    L = _ep.lib()
    nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
    ptr = ctypes.c_void_p()
    _ep._check("ep_host_alloc", L.ep_host_alloc(max(1, nbytes), ctypes.byref(ptr)))
    addr = ptr.value

    def _free(_self, addr=addr, L=L):
        L.ep_host_free(ctypes.c_void_p(addr))

    # a ctypes array over the mapping that frees it when collected; the
    # tensor keeps it alive
    owner_t = type("HostBytes", (ctypes.c_uint8 * max(1, nbytes),), {"__del__": _free})
    owner = owner_t.from_address(addr)
    t = torch.frombuffer(owner, dtype=torch.uint8)[:nbytes]
    return t.view(dtype).view(shape)


class HostPipeline:
    """route -> layout -> dispatch -> combine over host buffers, pipelined:
    the binding of the library's native pipeline (ep_host_pipeline_* in
    include/ep.h), which owns three streams and the events that order them.

    Each `step(x_h, logits_h, rank_offsets_h, y_h, out_h)` enqueues: the
    copies in of the step's logits, rank offsets, tokens x and expert outputs
    y (CPU tensors, pinned for the copies to overlap; the shapes of the
    single-batch path); route and layout once the logits are in, dispatch once
    x is in, combine once y is in; the copy of the combined [N, H] bf16 result
    to out_h.  `depth` device buffer sets rotate, so step i + 1's copies in run
    under step i's kernels and copy out; a set is reused only after the
    kernels and the copy out of the step that last used it are done.

    y holds the expert outputs of the dispatched rows in the step's own
    expert-major order ([N*K, H] contiguous; [E, cap, H] when cap > 0, the
    masked layout), as the caller's expert stage would produce them.
    `expert_map` (device int32 [E], optional) renumbers experts in routing,
    the same map every step.  The host tensors must stay untouched until the
    step's copies are done: `synchronize()` (or `join()` and a sync of the
    calling stream) waits for every step enqueued so far.  After it, `out`
    (and `scales` for FP8) hold the last step's dispatched rows and `layout`
    its layout (views into the pipeline's workspace).
    """

    def __init__(self, N, E, K, H, R, dtype=_ep.EP_DTYPE_BF16, device="cuda", cap=0,
                 expert_map=None, depth=2):
        import ctypes
        L = _ep.lib()
        dev = torch.device(device)
        if dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.N, self.E, self.K, self.H, self.R = N, E, K, H, R
        self.dtype, self.cap, self.depth = dtype, cap, depth
        self.layout_kind = _ep.EP_LAYOUT_MASKED if cap > 0 else _ep.EP_LAYOUT_CONTIG
        self.rows = _ep.dispatch_rows(N, K, E, self.layout_kind, cap)
        size = L.ep_host_pipeline_workspace_size(N, E, K, H, R, cap, dtype, depth)
        if size == 0:
            raise _ep.EPError(f"host pipeline: unsupported sizes N={N} E={E} K={K} H={H} "
                              f"R={R} cap={cap} depth={depth}")
        self.device = dev
        self.expert_map = expert_map  # the pipeline reads it on every step
        emap = None if expert_map is None else _ep._dev(expert_map, torch.int32, "expert_map",
                                                        (E,))
        with torch.cuda.device(dev):
            self.workspace = torch.empty(size, dtype=torch.uint8, device=dev)
            self._h = ctypes.c_void_p()
            _ep._check("ep_host_pipeline_create", L.ep_host_pipeline_create(
                N, E, K, H, R, cap, dtype, depth, emap,
                ctypes.c_void_p(self.workspace.data_ptr()), size, ctypes.byref(self._h)))
        fp8 = dtype == _ep.EP_DTYPE_FP8_E4M3_B128
        self.out = self._view(9, (self.rows, H), torch.uint8 if fp8 else torch.bfloat16)
        self.scales = self._view(10, (self.rows, H // 128), torch.float32) if fp8 else None
        self.topk_idx = self._view(0, (N, K), torch.int32)
        self.topk_w = self._view(1, (N, K), torch.float32)
        self.layout = _ep.Layout(
            self._view(2, (R, E), torch.int32), self._view(3, (E + 1,), torch.int32),
            self._view(4, (R, E), torch.int32), self._view(5, (N, K), torch.int32),
            self._view(6, (N * K,), torch.int32),
            self._view(7, (E,), torch.int32) if cap > 0 else None,
            self._view(8, (1,), torch.int32) if cap > 0 else None)

    def _view(self, which, shape, dtype):
        """Tensor view of one of the pipeline's device buffers (its workspace)."""
        import ctypes
        ptr, nbytes = ctypes.c_void_p(), ctypes.c_size_t()
        _ep._check("ep_host_pipeline_buffer", _ep.lib().ep_host_pipeline_buffer(
            self._h, which, ctypes.byref(ptr), ctypes.byref(nbytes)))
        off = ptr.value - self.workspace.data_ptr()
        return self.workspace[off:off + nbytes.value].view(dtype).view(shape)

    def _host(self, t, dtype, numel, name):
        import ctypes
        if not isinstance(t, torch.Tensor) or t.is_cuda:
            raise _ep.EPError(f"{name} must be a CPU tensor")
        if t.dtype != dtype or not t.is_contiguous() or t.numel() != numel:
            raise _ep.EPError(f"{name} must be a contiguous {dtype} tensor of {numel} elements")
        return ctypes.c_void_p(t.data_ptr())

    def step(self, x_h, logits_h, rank_offsets_h, y_h, out_h):
        N, E, K, H, R = self.N, self.E, self.K, self.H, self.R
        args = (self._host(logits_h, torch.float32, N * E, "logits_h"),
                self._host(rank_offsets_h, torch.int32, R + 1, "rank_offsets_h"),
                self._host(x_h, torch.bfloat16, N * H, "x_h"),
                self._host(y_h, torch.bfloat16, self.rows * H, "y_h"),
                self._host(out_h, torch.bfloat16, N * H, "out_h"))
        with torch.cuda.device(self.device):
            _ep._check("ep_host_pipeline_step", _ep.lib().ep_host_pipeline_step(
                self._h, *args, _ep._stream(None)))

    def join(self, stream=None):
        """Make `stream` (default: the current one) wait for every step."""
        with torch.cuda.device(self.device):
            _ep._check("ep_host_pipeline_join",
                       _ep.lib().ep_host_pipeline_join(self._h, _ep._stream(stream)))

    def copy_ms(self):
        """(h2d_ms, d2h_ms): device-timed copies in and copy out of the last
        step, once it is done (after synchronize())."""
        import ctypes
        a, b = ctypes.c_float(), ctypes.c_float()
        with torch.cuda.device(self.device):
            _ep._check("ep_host_pipeline_copy_ms", _ep.lib().ep_host_pipeline_copy_ms(
                self._h, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def synchronize(self):
        with torch.cuda.device(self.device):
            s = torch.cuda.current_stream()
            self.join(s)
            s.synchronize()

    def close(self):
        """Wait for the pipeline and release its streams and events."""
        h, self._h = getattr(self, "_h", None), None
        if h is not None and h.value:
            with torch.cuda.device(self.device):
                _ep._check("ep_host_pipeline_destroy", _ep.lib().ep_host_pipeline_destroy(h))

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: the library may be gone
            pass
