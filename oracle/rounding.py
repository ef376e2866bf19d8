"""Round-to-nearest-even to fp32 and bf16 (test infrastructure only).

fp32: numpy's float64 -> float32 conversion (IEEE 754 round to nearest even).
bf16: fp32 bit pattern, round to nearest even at bit 16, NaN kept quiet.
"""
from __future__ import annotations

import numpy as np


def to_f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def f32_to_bf16_bits(x) -> np.ndarray:
    f = np.ascontiguousarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    nan = (b & 0x7F800000) == 0x7F800000
    nan &= (b & 0x007FFFFF) != 0
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    r = np.where(nan, (b >> 16) | 0x40, r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_bf16(x) -> np.ndarray:
    """Value of x (double) after rounding to fp32 and then to bf16, returned as float32."""
    return bf16_bits_to_f32(f32_to_bf16_bits(to_f32(x)))
