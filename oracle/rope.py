"""Rotary position embedding for the oracle (test infrastructure only).

The samir-vllm article ("Gestion de la KV cache et strategies de batching")
states that each new token's K is written at its absolute RoPE position; the
tiny-vllm chapter ("What else is set up in the initialization block") builds a
RoPE frequency table once at start-up but does not print it.  Where the pages
are silent this module takes these readings:

* frequencies are an input: 32 FP64 values ``inv_freq[i]``; the default is
  Llama-3.2's published setting (theta = 500000 with "llama3" scaling:
  factor 32, low 1, high 4, original context 8192);
* pairs are half-split: dimension i rotates with dimension i + 32;
* the table holds fp32 values: ``cos[p][i] = fp32(cos(p * inv_freq[i]))``
  with the product and the cosine taken in FP64;
* the rotation of a bf16 pair (x0, x1) by (c, s) is done in fp32 with every
  operation rounded to nearest and no fused multiply-add:
      r0 = fp32(fp32(x0*c) - fp32(x1*s)),  r1 = fp32(fp32(x0*s) + fp32(x1*c)),
  and each result is rounded to bf16 (nearest-even).  This fixed order makes
  the appended bytes unique.

fp32 arithmetic is emulated by computing each operation in FP64 and rounding
to fp32: for +, -, * of fp32 operands this double rounding equals a single
fp32 rounding because 53 >= 2*24 + 2 (S. A. Figueroa, "When is double rounding
innocuous?", 1995); the product of a bf16 and an fp32 is even exact in FP64.
"""
from __future__ import annotations

import math

import numpy as np

from . import bf16

HEAD_DIM = 64
PAIRS = HEAD_DIM // 2


def inv_freq_plain(theta: float = 500000.0, head_dim: int = HEAD_DIM) -> np.ndarray:
    """inv_freq[i] = theta ** (-(2 i) / head_dim) for i in [0, head_dim / 2)."""
    return np.array([math.pow(theta, -(2.0 * i) / head_dim) for i in range(head_dim // 2)],
                    dtype=np.float64)


def inv_freq_llama3(theta: float = 500000.0, factor: float = 32.0, low_freq_factor: float = 1.0,
                    high_freq_factor: float = 4.0, original_max_pos: int = 8192,
                    head_dim: int = HEAD_DIM) -> np.ndarray:
    """Llama 3 frequency scaling of the plain table.

    Components whose wavelength 2*pi/f is shorter than original/high are kept;
    longer than original/low are divided by `factor`; in between they are
    blended linearly in original/wavelength.
    """
    low_wavelen = original_max_pos / low_freq_factor
    high_wavelen = original_max_pos / high_freq_factor
    out = []
    for f in inv_freq_plain(theta, head_dim):
        f = float(f)
        wavelen = 2.0 * math.pi / f
        if wavelen < high_wavelen:
            out.append(f)
        elif wavelen > low_wavelen:
            out.append(f / factor)
        else:
            smooth = (original_max_pos / wavelen - low_freq_factor) / (high_freq_factor - low_freq_factor)
            out.append((1.0 - smooth) * f / factor + smooth * f)
    return np.array(out, dtype=np.float64)


def table(inv_freq, max_pos: int):
    """fp32 cos/sin tables [max_pos][32]: fp32(cos(p * inv_freq[i])), FP64 inside."""
    inv_freq = np.asarray(inv_freq, dtype=np.float64)
    cos = np.empty((max_pos, inv_freq.shape[0]), dtype=np.float32)
    sin = np.empty_like(cos)
    for p in range(max_pos):
        for i, f in enumerate(inv_freq):
            ang = float(p) * float(f)
            cos[p, i] = np.float32(math.cos(ang))
            sin[p, i] = np.float32(math.sin(ang))
    return cos, sin


def _f32(x):
    """Round FP64 values to the nearest fp32, returned as FP64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def rotate_bf16(x_bits, cos_row, sin_row) -> np.ndarray:
    """Rotate bf16 vectors [..., 64] by one position's table row; returns bf16 bits.

    Pairs (i, i + 32) for i < 32, fp32 operation order as in the module notes.
    """
    x = bf16.to_f64(x_bits)
    x0, x1 = x[..., :PAIRS], x[..., PAIRS:]
    c = np.asarray(cos_row, dtype=np.float32).astype(np.float64)
    s = np.asarray(sin_row, dtype=np.float32).astype(np.float64)
    r0 = _f32(_f32(x0 * c) - _f32(x1 * s))
    r1 = _f32(_f32(x0 * s) + _f32(x1 * c))
    return np.concatenate([bf16.from_f32_rne(r0.astype(np.float32)),
                           bf16.from_f32_rne(r1.astype(np.float32))], axis=-1)


def rotate_exact(x, pos: float, inv_freq) -> np.ndarray:
    """The same rotation in plain FP64 with no rounding (for invariant checks)."""
    x = np.asarray(x, dtype=np.float64)
    ang = float(pos) * np.asarray(inv_freq, dtype=np.float64)
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., :PAIRS], x[..., PAIRS:]
    return np.concatenate([x0 * c - x1 * s, x0 * s + x1 * c], axis=-1)
