"""Shared helpers for the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

import workloads as W

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
