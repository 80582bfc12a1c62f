"""Comparison helpers for the GPU parity tests."""

from __future__ import annotations

import numpy as np
import torch

from int8_quantized_linear_gb300 import synthetic


def bits(t: torch.Tensor) -> np.ndarray:
    return synthetic.bf16_bits(t)


def from_bits(b: np.ndarray, device="cpu") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b, np.uint16).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_ordered(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers whose differences count ulps (+0 == -0)."""
    b = b.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def max_ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> int:
    return int(np.abs(bf16_ordered(a_bits) - bf16_ordered(b_bits)).max(initial=0))


def rel_frobenius(y: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(y - ref) / den) if den > 0 else float(np.linalg.norm(y))


def frob_bar(ref: np.ndarray, bar: float) -> float:
    """The relative-Frobenius bar a bf16 output of `ref` can be held to: `bar`,
    or, where even the correctly rounded result misses it, that rounding
    floor with 5 % room (outputs whose energy sits in a few elements driven
    by outlier channels, each rounded with up to 2^-8 relative error).  The
    floor comes from the oracle's result alone."""
    rounded = torch.from_numpy(np.ascontiguousarray(ref, dtype=np.float64)).to(torch.bfloat16).double().numpy()
    return max(bar, 1.05 * rel_frobenius(rounded, ref))


def guarded(shape, dtype, device, fill, guard=256):
    """A tensor view followed by a guard band of sentinel values."""
    n = int(np.prod(shape)) if len(shape) else 1
    buf = torch.full((n + guard,), fill, dtype=dtype, device=device)
    return buf, buf[:n].view(*shape)


def guard_intact(buf: torch.Tensor, n: int, fill) -> bool:
    tail = buf[n:]
    return bool((tail == fill).all().item())
