"""Thin Python binding of libep_gb300 (the C ABI declared in include/ep.h).

Argument marshalling only: every function checks that its tensors are CUDA
tensors of the expected dtype and shape, passes their device pointers and the
current CUDA stream to the C function of the same name, and raises EPError
on a non-zero status.  Output tensors may be passed in (for reuse or CUDA
graph capture) or are allocated with torch.empty.  There is no CPU path: if
the shared library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from collections import namedtuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libep_gb300.so")

EP_LAYOUT_CONTIG = 0
EP_LAYOUT_MASKED = 1
EP_DTYPE_BF16 = 0
EP_DTYPE_FP8_E4M3_B128 = 1

_lib = None


class EPError(RuntimeError):
    pass


def lib():
    """The loaded libep_gb300 (loads it on first use; raises if it is absent)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise EPError(f"{LIB_PATH} is not built; run combine_ep_route_topk_gb300.build.build() "
                          "(nvcc, sm_103a). There is no fallback implementation.")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.ep_route_topk.argtypes = [P, i32, i32, i32, P, P, P, P]
        L.ep_expert_balance_map.argtypes = [P, i32, i32, P, P]
        L.ep_dispatch_layout_workspace_size.argtypes = [i32, i32, i32, i32]
        L.ep_dispatch_layout_workspace_size.restype = sz
        L.ep_dispatch_layout.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P,
                                         sz, P]
        L.ep_route_layout_workspace_size.argtypes = [i32, i32, i32, i32]
        L.ep_route_layout_workspace_size.restype = sz
        L.ep_route_layout.argtypes = [P, P, i32, i32, i32, i32, P, i32, P, P, P, P, P, P, P, P, P,
                                      P, P, sz, P]
        L.ep_route_layout.restype = ctypes.c_int
        L.ep_dispatch.argtypes = [P, i32, i32, i32, i32, P, P, P, ctypes.c_int, i32, ctypes.c_int,
                                  P, P, P]
        L.ep_combine.argtypes = [P, i32, i32, i32, i32, P, P, P, P, ctypes.c_int, i32, P, P]
        L.ep_selftest_wait_timeout.argtypes = [P, P, sz, P]
        L.ep_route_dispatch_workspace_size.argtypes = [i32, i32, i32, i32]
        L.ep_route_dispatch_workspace_size.restype = sz
        L.ep_route_dispatch.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, ctypes.c_int, i32,
                                        ctypes.c_int, P, P, P, P, P, P, P, P, P, P, P, P, sz, P]
        L.ep_route_dispatch.restype = ctypes.c_int
        L.ep_host_pipeline_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32,
                                                      ctypes.c_int, i32]
        L.ep_host_pipeline_workspace_size.restype = sz
        L.ep_host_pipeline_create.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.c_int, i32, P,
                                              P, sz, ctypes.POINTER(P)]
        L.ep_host_pipeline_step.argtypes = [P, P, P, P, P, P, P]
        L.ep_host_pipeline_join.argtypes = [P, P]
        L.ep_host_pipeline_copy_ms.argtypes = [P, ctypes.POINTER(ctypes.c_float),
                                               ctypes.POINTER(ctypes.c_float)]
        L.ep_host_pipeline_copy_ms.restype = ctypes.c_int
        L.ep_host_pipeline_buffer.argtypes = [P, ctypes.c_int, ctypes.POINTER(P),
                                              ctypes.POINTER(sz)]
        L.ep_host_pipeline_destroy.argtypes = [P]
        L.ep_host_alloc.argtypes = [sz, ctypes.POINTER(P)]
        L.ep_host_alloc.restype = ctypes.c_int
        L.ep_host_free.argtypes = [P]
        L.ep_host_free.restype = ctypes.c_int
        for f in ("ep_route_topk", "ep_expert_balance_map", "ep_dispatch_layout", "ep_dispatch",
                  "ep_combine"):
            getattr(L, f).restype = ctypes.c_int
        L.ep_status_string.argtypes = [ctypes.c_int]
        L.ep_status_string.restype = ctypes.c_char_p
        L.ep_last_cuda_error.argtypes = []
        L.ep_last_cuda_error.restype = ctypes.c_char_p
        L.ep_kernel_launch_count.argtypes = []
        L.ep_kernel_launch_count.restype = ctypes.c_uint64
        L.ep_abi_version.argtypes = []
        L.ep_abi_version.restype = ctypes.c_int32
        _lib = L
    return _lib


def _check(name, status):
    if status != 0:
        L = lib()
        raise EPError(f"{name}: {L.ep_status_string(status).decode()}"
                      f" {L.ep_last_cuda_error().decode()}".rstrip())


def _dev(t, dtype, name, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise EPError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise EPError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise EPError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise EPError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _opt(t, dtype, name, shape=None):
    return None if t is None else _dev(t, dtype, name, shape)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


def ep_kernel_launch_count() -> int:
    return int(lib().ep_kernel_launch_count())


def ep_route_topk(logits, K, expert_map=None, topk_idx=None, topk_w=None, stream=None):
    """logits float32 [N, E] -> (topk_idx int32 [N, K], topk_w float32 [N, K])."""
    N, E = logits.shape
    if topk_idx is None:
        topk_idx = _empty((N, K), torch.int32, logits)
    if topk_w is None:
        topk_w = _empty((N, K), torch.float32, logits)
    _check("ep_route_topk", lib().ep_route_topk(
        _dev(logits, torch.float32, "logits"), N, E, K,
        _opt(expert_map, torch.int32, "expert_map", (E,)),
        _dev(topk_idx, torch.int32, "topk_idx", (N, K)),
        _dev(topk_w, torch.float32, "topk_w", (N, K)), _stream(stream)))
    return topk_idx, topk_w


def ep_expert_balance_map(counts, expert_map=None, stream=None):
    """counts int32 [R, E] -> expert_map int32 [E] (old id -> new id)."""
    R, E = counts.shape
    if expert_map is None:
        expert_map = _empty((E,), torch.int32, counts)
    _check("ep_expert_balance_map", lib().ep_expert_balance_map(
        _dev(counts, torch.int32, "counts"), R, E,
        _dev(expert_map, torch.int32, "expert_map", (E,)), _stream(stream)))
    return expert_map


def ep_dispatch_layout_workspace_size(N, E, K, R) -> int:
    return int(lib().ep_dispatch_layout_workspace_size(N, E, K, R))


Layout = namedtuple("Layout", "counts expert_offsets rank_expert_offsets pos row_src masked_m "
                              "overflow_count")


def alloc_layout(N, E, K, R, cap, device):
    def z(*s):
        return torch.empty(s, dtype=torch.int32, device=device)
    return Layout(z(R, E), z(E + 1), z(R, E), z(N, K), z(N * K),
                  z(E) if cap > 0 else None, z(1) if cap > 0 else None)


def ep_dispatch_layout(topk_idx, rank_offsets, E, cap=0, out: Layout | None = None,
                       workspace=None, stream=None) -> Layout:
    """Counts, offsets and the stable expert-major permutation of the picks."""
    N, K = topk_idx.shape
    R = rank_offsets.shape[0] - 1
    if out is None:
        out = alloc_layout(N, E, K, R, cap, topk_idx.device)
    need = ep_dispatch_layout_workspace_size(N, E, K, R)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=topk_idx.device)
    _check("ep_dispatch_layout", lib().ep_dispatch_layout(
        _dev(topk_idx, torch.int32, "topk_idx"), _dev(rank_offsets, torch.int32, "rank_offsets"),
        R, N, E, K, cap,
        _dev(out.counts, torch.int32, "counts", (R, E)),
        _dev(out.expert_offsets, torch.int32, "expert_offsets", (E + 1,)),
        _dev(out.rank_expert_offsets, torch.int32, "rank_expert_offsets", (R, E)),
        _dev(out.pos, torch.int32, "pos", (N, K)),
        _dev(out.row_src, torch.int32, "row_src", (N * K,)),
        _opt(out.masked_m, torch.int32, "masked_m", (E,)),
        _opt(out.overflow_count, torch.int32, "overflow_count", (1,)),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))
    return out


def ep_route_layout_workspace_size(N, E, K, R) -> int:
    return int(lib().ep_route_layout_workspace_size(N, E, K, R))


def ep_route_layout(logits, rank_offsets, K, cap=0, expert_map=None, topk_idx=None,
                    topk_w=None, out: Layout | None = None, status=None, workspace=None,
                    stream=None):
    """ep_route_topk + ep_dispatch_layout in one cooperative kernel.
    Returns (topk_idx, topk_w, Layout)."""
    N, E = logits.shape
    R = rank_offsets.shape[0] - 1
    if topk_idx is None:
        topk_idx = _empty((N, K), torch.int32, logits)
    if topk_w is None:
        topk_w = _empty((N, K), torch.float32, logits)
    if out is None:
        out = alloc_layout(N, E, K, R, cap, logits.device)
    need = ep_route_layout_workspace_size(N, E, K, R)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=logits.device)
    _check("ep_route_layout", lib().ep_route_layout(
        _dev(logits, torch.float32, "logits"), _dev(rank_offsets, torch.int32, "rank_offsets"),
        R, N, E, K, _opt(expert_map, torch.int32, "expert_map", (E,)), cap,
        _dev(topk_idx, torch.int32, "topk_idx", (N, K)),
        _dev(topk_w, torch.float32, "topk_w", (N, K)),
        _dev(out.counts, torch.int32, "counts", (R, E)),
        _dev(out.expert_offsets, torch.int32, "expert_offsets", (E + 1,)),
        _dev(out.rank_expert_offsets, torch.int32, "rank_expert_offsets", (R, E)),
        _dev(out.pos, torch.int32, "pos", (N, K)),
        _dev(out.row_src, torch.int32, "row_src", (N * K,)),
        _opt(out.masked_m, torch.int32, "masked_m", (E,)),
        _opt(out.overflow_count, torch.int32, "overflow_count", (1,)),
        _opt(status, torch.int32, "status", (1,)),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))
    return topk_idx, topk_w, out


def ep_route_dispatch_workspace_size(N, E, K, R) -> int:
    return int(lib().ep_route_dispatch_workspace_size(N, E, K, R))


def ep_route_dispatch(logits, rank_offsets, x, K, layout=EP_LAYOUT_CONTIG, cap=0,
                      dtype=EP_DTYPE_BF16, expert_map=None, topk_idx=None, topk_w=None,
                      lay: Layout | None = None, out=None, out_scales=None, workspace=None,
                      stream=None):
    """ep_route_topk + ep_dispatch_layout + ep_dispatch in one call (two
    launches up to 2048 tokens and 16384 picks).  Returns (topk_idx, topk_w,
    Layout, out, out_scales) as the three calls would."""
    N, E = logits.shape
    H = x.shape[1]
    R = rank_offsets.shape[0] - 1
    if topk_idx is None:
        topk_idx = _empty((N, K), torch.int32, logits)
    if topk_w is None:
        topk_w = _empty((N, K), torch.float32, logits)
    if lay is None:
        lay = alloc_layout(N, E, K, R, cap, logits.device)
    rows = dispatch_rows(N, K, E, layout, cap)
    if dtype == EP_DTYPE_BF16:
        if out is None:
            out = _empty((rows, H), torch.bfloat16, x)
        po = _dev(out, torch.bfloat16, "out")
    else:
        if out is None:
            out = _empty((rows, H), torch.uint8, x)
        if out_scales is None:
            out_scales = _empty((rows, H // 128), torch.float32, x)
        po = _dev(out, torch.uint8, "out")
    if out.numel() != rows * H:
        raise EPError(f"out must hold {rows} x {H} elements")
    if out_scales is not None and out_scales.numel() != rows * (H // 128):
        raise EPError(f"out_scales must hold {rows} x {H // 128} elements")
    if workspace is None:
        workspace = torch.empty(ep_route_dispatch_workspace_size(N, E, K, R), dtype=torch.uint8,
                                device=logits.device)
    _check("ep_route_dispatch", lib().ep_route_dispatch(
        _dev(logits, torch.float32, "logits"), _dev(rank_offsets, torch.int32, "rank_offsets"),
        _dev(x, torch.bfloat16, "x"), R, N, H, E, K,
        _opt(expert_map, torch.int32, "expert_map", (E,)), layout, cap, dtype,
        _dev(topk_idx, torch.int32, "topk_idx", (N, K)),
        _dev(topk_w, torch.float32, "topk_w", (N, K)),
        _dev(lay.counts, torch.int32, "counts", (R, E)),
        _dev(lay.expert_offsets, torch.int32, "expert_offsets", (E + 1,)),
        _dev(lay.rank_expert_offsets, torch.int32, "rank_expert_offsets", (R, E)),
        _dev(lay.pos, torch.int32, "pos", (N, K)),
        _dev(lay.row_src, torch.int32, "row_src", (N * K,)),
        _opt(lay.masked_m, torch.int32, "masked_m", (E,)),
        _opt(lay.overflow_count, torch.int32, "overflow_count", (1,)), po,
        _opt(out_scales, torch.float32, "out_scales"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))
    return topk_idx, topk_w, lay, out, out_scales


def dispatch_rows(N, K, E, layout, cap):
    return N * K if layout == EP_LAYOUT_CONTIG else E * cap


def ep_dispatch(x, topk_idx, pos, expert_offsets, E, layout=EP_LAYOUT_CONTIG, cap=0,
                dtype=EP_DTYPE_BF16, out=None, out_scales=None, stream=None):
    """Scatter x [N, H] bf16 into the expert-major buffer.  Returns
    (out, out_scales): out bf16 [rows, H] or uint8 FP8 codes [rows, H];
    out_scales float32 [rows, H/128] for FP8, else None."""
    N, H = x.shape
    K = topk_idx.shape[1]
    rows = dispatch_rows(N, K, E, layout, cap)
    if dtype == EP_DTYPE_BF16:
        if out is None:
            out = _empty((rows, H), torch.bfloat16, x)
        po = _dev(out, torch.bfloat16, "out")
    else:
        if out is None:
            out = _empty((rows, H), torch.uint8, x)
        if out_scales is None:
            out_scales = _empty((rows, H // 128), torch.float32, x)
        po = _dev(out, torch.uint8, "out")
    if out.numel() != rows * H:
        raise EPError(f"out must hold {rows} x {H} elements")
    if out_scales is not None and out_scales.numel() != rows * (H // 128):
        raise EPError(f"out_scales must hold {rows} x {H // 128} elements")
    _check("ep_dispatch", lib().ep_dispatch(
        _dev(x, torch.bfloat16, "x"), N, H, E, K, _dev(topk_idx, torch.int32, "topk_idx", (N, K)),
        _dev(pos, torch.int32, "pos", (N, K)),
        _opt(expert_offsets, torch.int32, "expert_offsets", (E + 1,)), layout, cap, dtype, po,
        _opt(out_scales, torch.float32, "out_scales"), _stream(stream)))
    return out, out_scales


def ep_combine(y, topk_idx, topk_w, pos, expert_offsets, E, layout=EP_LAYOUT_CONTIG, cap=0,
               out=None, stream=None):
    """K-way weighted sum of expert outputs y back to token order: [N, H] bf16."""
    N, K = topk_idx.shape
    H = y.shape[-1]
    rows = dispatch_rows(N, K, E, layout, cap)
    if y.numel() != rows * H:
        raise EPError(f"y must hold {rows} x {H} elements")
    if out is None:
        out = _empty((N, H), torch.bfloat16, y)
    _check("ep_combine", lib().ep_combine(
        _dev(y, torch.bfloat16, "y"), N, H, E, K, _dev(topk_idx, torch.int32, "topk_idx", (N, K)),
        _dev(topk_w, torch.float32, "topk_w", (N, K)), _dev(pos, torch.int32, "pos", (N, K)),
        _opt(expert_offsets, torch.int32, "expert_offsets", (E + 1,)), layout, cap,
        _dev(out, torch.bfloat16, "out", (N, H)), _stream(stream)))
    return out


def ep_selftest_wait_timeout(stream=None):
    """Runs the bounded-wait self-test (a grid barrier that can never complete
    gives up, sets the status word to 1 and returns).  Returns the device
    status tensor (int32 [1]); read it after synchronising."""
    dev = torch.device("cuda", torch.cuda.current_device())
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    _check("ep_selftest_wait_timeout", lib().ep_selftest_wait_timeout(
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        _stream(stream)))
    # keep the workspace alive until the kernel has run
    ws.record_stream(torch.cuda.current_stream(dev) if stream is None else stream)
    return status
