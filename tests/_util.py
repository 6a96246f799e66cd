"""Helpers shared by the tests: conversions between torch tensors and the
oracle's numpy arrays (bf16 as uint16 bit patterns).  No method arithmetic."""
import numpy as np
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy uint16 bf16 bit patterns -> bf16 tensor."""
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)


def np_(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def bf16_ulp(mag: np.ndarray) -> np.ndarray:
    """One bf16 unit in the last place at magnitude |mag| (normal range)."""
    mag = np.maximum(np.abs(mag.astype(np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(mag)) - 7)


def weight_rtol():
    """Relative tolerance of the float32 gate weights against the oracle's
    double-precision softmax rounded once to float.  Per pick: the logit
    difference l_k - l_0 carries one float rounding (relative 2^-24, i.e. an
    absolute error |d| 2^-24 in the exponent), expf is within 2 ulp, the sum
    of K terms adds up to K/2 ulp, the division half an ulp: for |d| <= 40
    and K <= 32 the total stays below (40 + 2 + 16 + 1) * 2^-23 < 1e-5."""
    return 1e-5


def combine_rel_err(got_bits: np.ndarray, ref_bits: np.ndarray, floor: float = 1e-2) -> float:
    """max |got - ref| / max(|ref|, floor) over all elements (bf16 inputs)."""
    g = (got_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = (ref_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if g.size == 0:
        return 0.0
    return float(np.max(np.abs(g - r) / np.maximum(np.abs(r), floor)))
