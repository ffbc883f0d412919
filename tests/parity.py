"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances (max |err| / rms(oracle)) follow the scan's stated bounds: 1e-5 for
fp32 inputs and 2e-3 for bf16 inputs, fp32 state. A y stored in bf16 carries its
own rounding (half a bf16 ulp, up to 2^-9 |y|), which no computation can beat,
so a bf16 y is checked elementwise against 2e-3 * rms(y_oracle) plus half a bf16
ulp of the oracle value; the 2e-3 bound itself is checked on fp32-y runs of the
same bf16 inputs.
"""
from __future__ import annotations

import numpy as np
import torch

TOL_F32 = 1e-5
TOL_BF16 = 2e-3


def tol_for(in_dtype) -> float:
    return TOL_BF16 if in_dtype in (torch.bfloat16, "bf16") else TOL_F32


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(got - ref))) / max(rms, 1e-30)


def assert_y_close(got: np.ndarray, ref: np.ndarray, tol: float, out_is_bf16: bool, what: str = "y"):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(got - ref)
    if out_is_bf16:
        bound = tol * rms + bf16_half_ulp(ref) * 1.0001
        bad = err > bound
        assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of bound; worst "
                               f"excess {float(np.max(err - bound)):.3e}, rms {rms:.3e}")
    else:
        r = float(np.max(err)) / max(rms, 1e-30)
        assert r <= tol, f"{what}: max|err|/rms = {r:.3e} > {tol:.1e}"


def assert_state_close(got: np.ndarray, ref: np.ndarray, tol: float, what: str = "h_last"):
    r = rel_err(got, ref)
    assert r <= tol, f"{what}: max|err|/rms = {r:.3e} > {tol:.1e}"


def sample_channels(batch: int, dim: int, count: int, seed: int = 0):
    """Deterministic channel sample: the four corners plus random (b, d) pairs."""
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (0, dim - 1), (batch - 1, 0), (batch - 1, dim - 1)}
    while len(picks) < min(count, batch * dim):
        picks.add((int(rng.integers(batch)), int(rng.integers(dim))))
    return sorted(picks)
