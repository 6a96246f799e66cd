"""CPU oracle for the MoE expert-parallel route / layout / dispatch / combine path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product library never calls it and shares no code with it.

The arithmetic lives in ``ep_oracle.c`` (plain C, one thread); this module
only marshals numpy arrays into it.  bf16 tensors travel as their uint16 bit
patterns; FP8 codes as uint8.

Parity status per function (what pins it is in ``tests/test_oracle.py``):
  route_topk      pinned: worked example t0..t3, torch.topk on distinct rows,
                  brute-force repeated arg-max with ties, closed-form weights,
                  scipy softmax renormalisation
  balance_map     pinned: hand-worked example, zero-frequency identity,
                  permutation/contiguity invariants, exhaustive optimum bound
  layout          pinned: numpy stable argsort, bincount, invariants
  dispatch        pinned: fancy-indexing copy; FP8 codes via torch's
                  float8_e4m3fn cast and an exhaustive nearest-code search
  combine         pinned: identity round trip (exact), K=1 copy, float64
                  exact sum within the fp32-chain + bf16 rounding bound
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

LAYOUT_CONTIG = 0
LAYOUT_MASKED = 1
DTYPE_BF16 = 0
DTYPE_FP8 = 1


def _lib():
    global _LIB
    if _LIB is None:
        # EP_ORACLE_LIB lets the mutation tests load a deliberately broken copy
        path = os.environ.get("EP_ORACLE_LIB") or _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_route_topk.argtypes = [P, i64, i32, i32, P, P, P]
        lib.oracle_balance_map.argtypes = [P, i32, i32, P]
        lib.oracle_layout.argtypes = [P, P, i32, i64, i32, i32, i32, P, P, P, P, P, P, P]
        lib.oracle_dispatch.argtypes = [P, i64, i32, i32, i32, P, P, P, ctypes.c_int, i32,
                                        ctypes.c_int, P, P]
        lib.oracle_combine.argtypes = [P, i64, i32, i32, i32, P, P, P, P, ctypes.c_int, i32, P]
        lib.oracle_fp8_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_fp8_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_fp8_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_fp8_e4m3_decode.restype = ctypes.c_double
        lib.oracle_float_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_float_to_bf16.restype = ctypes.c_uint16
        lib.oracle_fp8_e4m3_encode_n.argtypes = [P, i64, P]
        lib.oracle_float_to_bf16_n.argtypes = [P, i64, P]
        _LIB = lib
    return _LIB


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def route_topk(logits, K, expert_map=None):
    """logits float32 [N, E] -> (topk_idx int32 [N, K], topk_w float32 [N, K])."""
    logits = _c(logits, np.float32)
    N, E = logits.shape
    emap = None if expert_map is None else _c(expert_map, np.int32)
    idx = np.empty((N, K), np.int32)
    w = np.empty((N, K), np.float32)
    _lib().oracle_route_topk(_p(logits), N, E, K, _p(emap), _p(idx), _p(w))
    return idx, w


def balance_map(counts):
    """counts int32 [R, E] -> expert_map int32 [E] (old id -> new id)."""
    counts = _c(counts, np.int32)
    R, E = counts.shape
    emap = np.empty(E, np.int32)
    _lib().oracle_balance_map(_p(counts), R, E, _p(emap))
    return emap


def layout(topk_idx, rank_offsets, E, cap=0):
    """Returns a dict with counts [R,E], expert_offsets [E+1],
    rank_expert_offsets [R,E], pos [N,K], row_src [N*K] and, when cap > 0,
    masked_m [E] and overflow (int)."""
    topk_idx = _c(topk_idx, np.int32)
    rank_offsets = _c(rank_offsets, np.int32)
    N, K = topk_idx.shape
    R = rank_offsets.shape[0] - 1
    counts = np.empty((R, E), np.int32)
    eoff = np.empty(E + 1, np.int32)
    reoff = np.empty((R, E), np.int32)
    pos = np.empty((N, K), np.int32)
    row_src = np.empty(N * K, np.int32)
    masked_m = np.zeros(E, np.int32)
    overflow = np.zeros(1, np.int32)
    _lib().oracle_layout(_p(topk_idx), _p(rank_offsets), R, N, E, K, cap, _p(counts), _p(eoff),
                         _p(reoff), _p(pos), _p(row_src), _p(masked_m), _p(overflow))
    out = dict(counts=counts, expert_offsets=eoff, rank_expert_offsets=reoff, pos=pos,
               row_src=row_src)
    if cap > 0:
        out["masked_m"] = masked_m
        out["overflow"] = int(overflow[0])
    return out


def dispatch(x_bits, topk_idx, pos, expert_offsets, E, layout=LAYOUT_CONTIG, cap=0,
             dtype=DTYPE_BF16, out=None, out_scales=None):
    """x_bits uint16 [N, H] (bf16 patterns).  Returns (out, out_scales):
    contiguous rows = N*K, masked rows = E*cap; out is uint16 (bf16) or uint8
    (FP8 codes); out_scales float32 [rows, H/128] for FP8, else None.
    Rows that receive no pick keep whatever ``out`` held (zeros if new)."""
    x_bits = _c(x_bits, np.uint16)
    topk_idx = _c(topk_idx, np.int32)
    pos = _c(pos, np.int32)
    expert_offsets = _c(expert_offsets, np.int32)
    N, H = x_bits.shape
    K = topk_idx.shape[1]
    rows = N * K if layout == LAYOUT_CONTIG else E * cap
    if out is None:
        out = np.zeros((rows, H), np.uint16 if dtype == DTYPE_BF16 else np.uint8)
    if dtype == DTYPE_FP8 and out_scales is None:
        out_scales = np.zeros((rows, H // 128), np.float32)
    _lib().oracle_dispatch(_p(x_bits), N, H, E, K, _p(topk_idx), _p(pos), _p(expert_offsets),
                           layout, cap, dtype, _p(out), _p(out_scales))
    return out, (out_scales if dtype == DTYPE_FP8 else None)


def combine(y_bits, topk_idx, topk_w, pos, expert_offsets, E, layout=LAYOUT_CONTIG, cap=0):
    """y_bits uint16 [rows, H] bf16 expert outputs -> out uint16 [N, H] (bf16)."""
    y_bits = _c(y_bits, np.uint16)
    topk_idx = _c(topk_idx, np.int32)
    topk_w = _c(topk_w, np.float32)
    pos = _c(pos, np.int32)
    expert_offsets = _c(expert_offsets, np.int32)
    N, K = topk_idx.shape
    H = y_bits.shape[-1]
    out = np.empty((N, H), np.uint16)
    _lib().oracle_combine(_p(y_bits), N, H, E, K, _p(topk_idx), _p(topk_w), _p(pos),
                          _p(expert_offsets), layout, cap, _p(out))
    return out


def fp8_e4m3_encode(v):
    """float32 values -> OCP E4M3FN codes (round to nearest even, satfinite)."""
    v = _c(np.asarray(v, np.float32).ravel(), np.float32)
    codes = np.empty(v.size, np.uint8)
    _lib().oracle_fp8_e4m3_encode_n(_p(v), v.size, _p(codes))
    return codes


def fp8_e4m3_decode_table():
    lib = _lib()
    return np.array([lib.oracle_fp8_e4m3_decode(c) for c in range(256)], np.float64)


def float_to_bf16(v):
    """float32 values -> bf16 bit patterns (round to nearest even)."""
    v = _c(np.asarray(v, np.float32).ravel(), np.float32)
    bits = np.empty(v.size, np.uint16)
    _lib().oracle_float_to_bf16_n(_p(v), v.size, _p(bits))
    return bits


def bf16_to_float(bits):
    """Exact widening of bf16 patterns to float32 (a bit shift)."""
    bits = np.asarray(bits, np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)
