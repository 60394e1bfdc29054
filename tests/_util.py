"""Shared helpers for the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

import workloads as W
from oracle import bf16 as OB

MAX_ABS_TOL = 1.5e-2   # max |gpu - oracle| on bf16 outputs, q/k/v ~ N(0,1)
MEAN_ABS_TOL = 1e-3    # mean |gpu - oracle|


def to_dev_bf16(bits: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def to_dev_i32(a, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bits(t: torch.Tensor) -> np.ndarray:
    return W.bf16_bits(t)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(gpu.astype(np.float64) - ref)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    assert err.max() <= MAX_ABS_TOL, f"{what}: max |err| {err.max():.3e}"
    assert err.mean() <= MEAN_ABS_TOL, f"{what}: mean |err| {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def check_close_int8(gpu, ref, what=""):
    """The bf16 bar applied to the error beyond the output format's own
    rounding: max |err| <= 1.5e-2 + 2^-8 |ref| where |ref| >= 4 (a bf16 half
    step there exceeds 1.5e-2), and mean |err| <= 1e-3 + the mean distance of
    the FP64 values to their nearest bf16 (the dequantised values, unlike bf16
    pages, are not bf16 numbers, so an output dominated by one token carries
    the full rounding of the bf16 result)."""
    gpu = gpu.astype(np.float64)
    err = np.abs(gpu - ref)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    allowed = MAX_ABS_TOL + np.where(np.abs(ref) >= 4.0, 2.0 ** -8 * np.abs(ref), 0.0)
    worst = int(np.argmax(err - allowed))
    assert np.all(err <= allowed), f"{what}: |err| {err.flat[worst]:.3e} at |ref| {abs(ref.flat[worst]):.3f}"
    rounding = np.abs(ref - OB.to_f64(OB.from_f64_via_f32(ref))).mean()
    assert err.mean() <= MEAN_ABS_TOL + rounding, \
        f"{what}: mean |err| {err.mean():.3e} (output rounding alone {rounding:.3e})"
    return float(err.max()), float(err.mean())


def cancelling_rows(seed, positions, heads, cos_o, sin_o):
    """bf16 bits [len(positions), heads, 64] whose rotation at the row's
    position nearly cancels: for even pairs i, x_(i+32) ~ x_i cos / sin, so
    x_i cos - x_(i+32) sin ~ 0; for odd pairs x_(i+32) ~ -x_i sin / cos, so
    x_i sin + x_(i+32) cos ~ 0 (random where the ratio is out of range).
    Near cancellation a fused multiply-add rounds differently from the two
    rounded products and the rounded sum that the rotation prescribes, often
    enough to show in the bf16 results."""
    g = np.random.default_rng(seed)
    n = len(positions)
    pos = np.asarray(positions, np.int64)
    x0 = OB.from_f32_rne(g.standard_normal((n, heads, 32)).astype(np.float32))
    c = cos_o[pos][:, None, :].astype(np.float64)
    s = sin_o[pos][:, None, :].astype(np.float64)
    even = np.arange(32) % 2 == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(even, c / s, -s / c)
    ok = np.isfinite(ratio) & (np.abs(ratio) < 64.0)
    x1 = np.where(ok, OB.to_f64(x0) * np.where(ok, ratio, 0.0), g.standard_normal((n, heads, 32)))
    return np.concatenate([x0, OB.from_f32_rne(x1.astype(np.float32))], axis=-1)
