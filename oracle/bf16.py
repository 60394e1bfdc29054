"""bf16 conversions for the oracle (test infrastructure only).

bf16 is the storage type of every activation and of the KV cache in the engines
the path comes from ("2. Weight Loading and GPU Buffer Design", opening
section: 1 sign, 8 exponent, 7 mantissa bits; "one element = 2 bytes").

Values travel as uint16 bit patterns so that comparisons are bit-exact.
"""
from __future__ import annotations

import numpy as np


def to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns to float64.  Exact: bf16 is the top half of fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def from_f32_rne(x) -> np.ndarray:
    """Round fp32 values to bf16, nearest-even, returning uint16 bit patterns.

    The 16 low bits are dropped after adding 0x7FFF plus the lowest kept bit,
    which rounds ties to the even neighbour.  Overflow carries into the
    exponent and yields +-Inf, as IEEE rounding requires.  NaN stays NaN.
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = ((u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    quiet_nan = ((u >> np.uint64(16)) | np.uint64(0x0040)) & np.uint64(0xFFFF)
    out = np.where(np.isnan(f), quiet_nan, rounded)
    return out.astype(np.uint16)


def from_f64_via_f32(x) -> np.ndarray:
    """fp64 -> fp32 (nearest) -> bf16 (nearest); used only for display of results."""
    return from_f32_rne(np.asarray(x, dtype=np.float64).astype(np.float32))
