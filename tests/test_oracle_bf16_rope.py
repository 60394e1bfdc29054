"""Pins for the oracle's bf16 conversions and RoPE (CPU only).

Each check reaches the oracle from outside it: hand-written bit patterns,
torch's own bf16 cast, numpy float32 arithmetic, the complex-multiplication
form of a rotation, and the relative-position property of RoPE.
"""
import math

import numpy as np
import pytest
import torch

from oracle import bf16, rope


# ---------------------------------------------------------------- bf16 ------

def test_widen_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x7F80, 0xFF80, 0x0001, 0x7F7F, 0x0000, 0x8000], np.uint16)
    want = [1.0, -2.0, math.inf, -math.inf, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, 0.0, -0.0]
    got = bf16.to_f64(bits)
    for g, w in zip(got, want):
        assert g == w and math.copysign(1, g) == math.copysign(1, w)


def test_round_hand_ties():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0 (0x3F80)
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even) -> 0x3F82
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, 3.4e38, -3.4e38],
                 dtype=np.float32)
    assert list(bf16.from_f32_rne(x)) == [0x3F80, 0x3F82, 0x3F81, 0x7F80, 0xFF80]


def test_round_matches_torch_cast():
    rng = np.random.default_rng(7)
    with np.errstate(over="ignore"):
        x = _round_inputs(rng)
    x = x[~np.isnan(x)]
    ours = bf16.from_f32_rne(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def _round_inputs(rng):
    return np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-39).astype(np.float32),   # subnormals
        (rng.standard_normal(20000) * 1e38).astype(np.float32),    # near overflow
        rng.integers(0, 2 ** 32, 50000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])


# ---------------------------------------------------------------- RoPE ------

def test_inv_freq_plain_closed_form():
    f = rope.inv_freq_plain(500000.0)
    assert f.shape == (32,)
    assert f[0] == 1.0
    assert f[16] == pytest.approx(500000.0 ** -0.5, rel=1e-15)
    assert np.allclose(f[1:] / f[:-1], 500000.0 ** (-1 / 32), rtol=1e-13)


def test_inv_freq_llama3_bands():
    base = rope.inv_freq_plain(500000.0)
    f = rope.inv_freq_llama3(500000.0, 32.0, 1.0, 4.0, 8192)
    wavelen = 2 * math.pi / base
    short = wavelen < 8192 / 4          # kept as is
    long_ = wavelen > 8192 / 1          # divided by the factor
    mid = ~short & ~long_
    assert short.sum() == 15 and long_.sum() == 14 and mid.sum() == 3
    assert np.array_equal(f[short], base[short])
    assert np.allclose(f[long_], base[long_] / 32.0, rtol=1e-15)
    # the blend stays strictly between the two limits and is monotone in i
    assert np.all(f[mid] < base[mid]) and np.all(f[mid] > base[mid] / 32)
    assert np.all(np.diff(f) < 0)


def test_table_position_zero_and_unit_circle():
    f = rope.inv_freq_llama3()
    cos, sin = rope.table(f, 64)
    assert cos.dtype == np.float32 and cos.shape == (64, 32)
    assert np.all(cos[0] == 1.0) and np.all(sin[0] == 0.0)
    r = cos.astype(np.float64) ** 2 + sin.astype(np.float64) ** 2
    assert np.max(np.abs(r - 1)) < 4 * 2.0 ** -24


def test_table_matches_vectorised_fp64():
    f = rope.inv_freq_llama3()
    cos, sin = rope.table(f, 2048)
    ang = np.arange(2048, dtype=np.float64)[:, None] * f[None, :]
    # numpy's own cos/sin, rounded to fp32: at most one fp32 ulp away
    for ours, ref in ((cos, np.cos(ang)), (sin, np.sin(ang))):
        d = np.abs(ours.astype(np.float64) - ref)
        ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
        assert np.all(d <= ulp)


def _rand_bits(rng, shape):
    x = rng.standard_normal(shape).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_rotate_position_zero_is_identity():
    rng = np.random.default_rng(1)
    x = _rand_bits(rng, (100, 64))
    cos, sin = rope.table(rope.inv_freq_llama3(), 1)
    y = rope.rotate_bf16(x, cos[0], sin[0])
    # equal as values (a -0.0 input could come back as +0.0; randn never gives one)
    assert np.array_equal(bf16.to_f64(y), bf16.to_f64(x))
    assert np.array_equal(y, x)


def test_rotate_fp32_order_matches_numpy_float32():
    rng = np.random.default_rng(2)
    x = _rand_bits(rng, (500, 64))
    cos, sin = rope.table(rope.inv_freq_llama3(), 2048)
    pos = rng.integers(0, 2048, 500)
    xf = bf16.to_f64(x).astype(np.float32)
    c, s = cos[pos], sin[pos]
    r0 = xf[:, :32] * c - xf[:, 32:] * s      # numpy float32: each op rounded, no FMA
    r1 = xf[:, :32] * s + xf[:, 32:] * c
    want = np.concatenate([bf16.from_f32_rne(r0), bf16.from_f32_rne(r1)], axis=-1)
    got = np.stack([rope.rotate_bf16(x[i], cos[pos[i]], sin[pos[i]]) for i in range(500)])
    assert np.array_equal(got, want)


def test_rotation_is_complex_multiplication():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 64))
    f = rope.inv_freq_llama3()
    for p in (0, 1, 17, 2047):
        z = (x[:, :32] + 1j * x[:, 32:]) * np.exp(1j * p * f)
        want = np.concatenate([z.real, z.imag], axis=-1)
        assert np.allclose(rope.rotate_exact(x, p, f), want, rtol=0, atol=1e-12)


def test_rotation_relative_position_and_norm():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    f = rope.inv_freq_plain()
    d0 = rope.rotate_exact(q, 100, f) @ rope.rotate_exact(k, 37, f)
    for shift in (1, 50, 900):
        d = rope.rotate_exact(q, 100 + shift, f) @ rope.rotate_exact(k, 37 + shift, f)
        assert d == pytest.approx(d0, abs=1e-9)
    assert np.linalg.norm(rope.rotate_exact(k, 1234, f)) == pytest.approx(np.linalg.norm(k), rel=1e-14)


def test_rotate_bf16_close_to_exact():
    rng = np.random.default_rng(5)
    x = _rand_bits(rng, (300, 64))
    f = rope.inv_freq_llama3()
    cos, sin = rope.table(f, 2048)
    for i, p in enumerate(rng.integers(0, 2048, 300)):
        exact = rope.rotate_exact(bf16.to_f64(x[i]), p, f)
        got = bf16.to_f64(rope.rotate_bf16(x[i], cos[p], sin[p]))
        # bf16 half-ulp of the result plus the fp32 table/op error
        assert np.all(np.abs(got - exact) <= 2.0 ** -8 * np.abs(exact) + 1e-6 * (1 + np.abs(x[i]).max()))


def test_cancelling_rows_expose_a_fused_multiply_add():
    """The GPU tests' near-cancelling inputs tell the prescribed rounding (two
    rounded products, a rounded sum) from a fused multiply-add: a copy of the
    rotation with either product fused into the sum, a planted mistake, gives
    other bf16 bits in hundreds of the 73,728 values."""
    from tests._util import cancelling_rows
    cos, sin = rope.table(rope.inv_freq_llama3(), 2048)
    pos = np.array([1, 16, 47, 100, 333, 700, 1023, 1500, 2047] * 4)
    x = cancelling_rows(7, pos, 32, cos, sin)
    want = np.stack([rope.rotate_bf16(x[i], cos[p], sin[p]) for i, p in enumerate(pos)])
    f = bf16.to_f64(x)
    x0, x1 = f[..., :32], f[..., 32:]
    c = cos[pos][:, None, :].astype(np.float64)
    s = sin[pos][:, None, :].astype(np.float64)
    r32 = rope._f32
    # near cancellation both operands of the sum have nearly one exponent, so
    # the FP64 sum of an exact product (bf16 x fp32: 32 bits) and a rounded
    # one is exact and one rounding to fp32 is the fused result
    for r0, r1 in [(r32(x0 * c - r32(x1 * s)), r32(x0 * s + r32(x1 * c))),
                   (r32(r32(x0 * c) - x1 * s), r32(r32(x0 * s) + x1 * c))]:
        fused = np.concatenate([bf16.from_f32_rne(r0.astype(np.float32)),
                                bf16.from_f32_rne(r1.astype(np.float32))], axis=-1)
        differ = int(np.count_nonzero(fused != want))
        assert differ > 200, differ
