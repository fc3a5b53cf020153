"""bf16 <-> fp32 conversions, written from their definitions (oracle; test infrastructure).

bf16 keeps the sign, the 8 exponent bits and the top 7 mantissa bits of an
IEEE fp32 number. Widening is exact: the 16 bits go to the top of an fp32 word.
Narrowing rounds to nearest, ties to even, on the discarded low 16 bits; a NaN
stays a quiet NaN. The all-reduce widens bf16 gradients to fp32 to accumulate
and rounds the averaged result back once (the fused kernel's statement: bf16 in,
fp32 accumulate, result cast back).
"""
from __future__ import annotations

import numpy as np


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 patterns -> fp32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 values -> uint16 bf16 patterns, round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    hi = u >> np.uint32(16)               # truncated pattern
    rem = u & np.uint32(0xFFFF)           # discarded bits
    half = np.uint32(0x8000)
    odd = (hi & np.uint32(1)) == 1
    up = (rem > half) | ((rem == half) & odd)
    out = hi + up.astype(np.uint32)       # a carry runs into the exponent, as it should
    is_nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    out = np.where(is_nan, hi | np.uint32(0x0040), out)
    return out.astype(np.uint16)
