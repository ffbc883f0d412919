"""Seeded synthetic inputs for the selective scan, shared by the tests, the bench
and the smoke check.

This module only draws random numbers and rounds them to the storage dtype. It
holds none of the scan's arithmetic (no discretisation, no recurrence, no
gating), so both the fp64 oracle and the CUDA path can take their inputs from it
without sharing any of the method.

Value recipe (shapes follow the Mamba layer sizes on the pages):
  * u, B, C, z ~ N(0, 1); delta ~ N(0, 0.5) for the prefill scans, N(0, 1) for
    decode; D ~ N(0, 1).
  * A_dn = -(n + 1) ("S4D-real" init: A_log = log(1..N), A = -exp(A_log); Mamba SSM
    complete guide (youngju.dev), section 5 "complete Mamba implementation",
    MambaBlock.__init__). For the d_state=1 scalar scan A_d = -exp(U(log 0.5, log 4)).
  * delta_bias_d = softplus^-1(dt0_d) with dt0_d = exp(U(log 1e-3, log 1e-1)), the
    dt_min/dt_max range of the same MambaBlock.__init__, so that
    softplus(delta + bias) scatters around a per-channel dt0 in [1e-3, 1e-1].
  * h0 = 0, except the scalar scan where h0 ~ N(0, 1) per (b, d).
Random draws use numpy PCG64 with seed = base + k, k: u=1, delta=2, z=3, B=4,
C=5, A=6, D=7, bias=8, h0=9; values are drawn in fp32 and rounded once
(round-to-nearest-even) to bf16 where the config stores bf16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"

K_U, K_DELTA, K_Z, K_B, K_C, K_A, K_D, K_BIAS, K_H0 = range(1, 10)


@dataclasses.dataclass(frozen=True)
class ScanConfig:
    """One prefill-scan workload: (batch, dim, seqlen, dstate) and dtypes."""
    name: str
    batch: int
    dim: int
    seqlen: int
    dstate: int
    in_dtype: str          # u, delta, z, B, C storage dtype
    out_dtype: str         # y storage dtype
    has_D: bool
    has_z: bool
    softplus: bool
    h0: str                # "zero" | "normal"
    A_kind: str            # "s4d_real" | "scalar_loguniform"
    seed_base: int

    @property
    def channels(self) -> int:
        return self.batch * self.dim

    @property
    def tokens_channels(self) -> int:
        return self.batch * self.dim * self.seqlen


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    """Single-token decode update workload on a resident (batch, dim, dstate) state."""
    name: str
    batch: int
    dim: int
    dstate: int
    in_dtype: str
    out_dtype: str
    steps: int
    token_sets: int        # per-step inputs cycle through this many seeded sets
    seed_base: int


CONFIGS = {
    # parity-size case the oracle finishes instantly
    "tiny": ScanConfig("tiny", 1, 16, 256, 16, F32, F32, True, False, True, "zero",
                       "s4d_real", 1000),
    # d_state = 1 scalar scan (SM1)
    "sm1": ScanConfig("sm1", 8, 1536, 2048, 1, F32, F32, False, False, True, "normal",
                      "scalar_loguniform", 2000),
    # Mamba-130M-shaped layer: d_model 768, expand 2
    "mamba130m": ScanConfig("mamba130m", 8, 1536, 2048, 16, BF16, BF16, True, True, True,
                            "zero", "s4d_real", 3000),
    # Mamba-2.8B-shaped layer: d_model 2560, expand 2
    "mamba2p8b": ScanConfig("mamba2p8b", 4, 5120, 4096, 16, BF16, BF16, True, True, True,
                            "zero", "s4d_real", 4000),
    # long context, small batch x channels
    "long": ScanConfig("long", 1, 1536, 131072, 16, BF16, BF16, True, True, True, "zero",
                       "s4d_real", 4500),
    # the four-direction image scan: a 56 x 56 patch grid (3136 tokens in raster
    # order), 192 scan channels (a 96-wide embedding, expand 2), batch 8
    "vmamba56": ScanConfig("vmamba56", 8, 192, 56 * 56, 16, BF16, BF16, True, True, True, "zero",
                           "s4d_real", 9000),
}

# image grid (rows, cols) of the directional-scan workloads (seqlen = rows * cols)
IMAGE_GRIDS = {"vmamba56": (56, 56)}

DECODE_CONFIGS = {
    "decode": DecodeConfig("decode", 256, 5120, 16, BF16, BF16, 1000, 16, 5000),
}


@dataclasses.dataclass(frozen=True)
class ConvConfig:
    """Causal depthwise conv1d (+ silu) workload: the block's input x before the scan
    (batch, dim, seqlen), kernel width, and the decode batch for the update."""
    name: str
    batch: int
    dim: int
    seqlen: int
    width: int
    in_dtype: str
    out_dtype: str
    seed_base: int


CONV_CONFIGS = {
    # the conv feeding the Mamba-130M-shaped scan (d_conv = 4, the page's default)
    "conv_mamba130m": ConvConfig("conv_mamba130m", 8, 1536, 2048, 4, BF16, BF16, 6000),
    # one decode token on the decode workload's (256, 5120) channels
    "conv_decode": ConvConfig("conv_decode", 256, 5120, 1, 4, BF16, BF16, 7000),
}



@dataclasses.dataclass(frozen=True)
class SsdConfig:
    """Mamba-2 SSD workload: x (batch, seqlen, nheads, headdim), B/C (batch, seqlen,
    ngroups, dstate), all bf16 but A, D, dt_bias and the state (fp32)."""
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    ngroups: int
    dstate: int
    has_D: bool
    has_z: bool
    h0: str                # "zero" | "normal"
    out_dtype: str
    seed_base: int

    @property
    def tokens_channels(self) -> int:
        return self.batch * self.seqlen * self.nheads * self.headdim


SSD_CONFIGS = {
    # a few ragged chunks, both state widths covered by overriding dstate
    "ssd_tiny": SsdConfig("ssd_tiny", 2, 300, 4, 64, 2, 64, True, True, "normal", BF16, 8000),
    # 5120 scan channels as 80 heads of 64 (the 2.8B-shaped layer's width), d_state 64
    "ssd_5120": SsdConfig("ssd_5120", 4, 4096, 80, 64, 1, 64, True, True, "zero", BF16, 8100),
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bits (uint16) to the exact fp32 value."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal(seed: int, shape, std: float = 1.0, chunk: int = 1 << 24) -> np.ndarray:
    g = _rng(seed)
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = g.standard_normal(e - s, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out.reshape(shape)


class Tensor:
    """A generated input: storage bits/values plus the exact fp32 value view."""

    def __init__(self, values_f32: np.ndarray, dtype: str):
        self.dtype = dtype
        if dtype == BF16:
            self.storage = bf16_bits(values_f32)
        else:
            self.storage = np.ascontiguousarray(values_f32, dtype=np.float32)

    @property
    def shape(self):
        return self.storage.shape

    def f32(self) -> np.ndarray:
        """Exact stored values as fp32 (bf16 values widen exactly)."""
        if self.dtype == BF16:
            return bf16_to_f32(self.storage)
        return self.storage

    def rows_f32(self, idx) -> np.ndarray:
        s = self.storage[idx]
        return bf16_to_f32(s) if self.dtype == BF16 else np.asarray(s, dtype=np.float32)


def _inv_softplus(y: np.ndarray) -> np.ndarray:
    # softplus^-1(y) = log(exp(y) - 1), written stably for small y
    y = y.astype(np.float64)
    return (y + np.log(-np.expm1(-y))).astype(np.float32)


def delta_bias(seed: int, dim: int) -> np.ndarray:
    g = _rng(seed)
    dt0 = np.exp(g.uniform(math.log(1e-3), math.log(1e-1), size=dim))
    return _inv_softplus(dt0)


def s4d_real_A(dim: int, dstate: int) -> np.ndarray:
    return -np.tile(np.arange(1, dstate + 1, dtype=np.float32), (dim, 1))


def make_scan_inputs(cfg: ScanConfig, batch: Optional[int] = None, dim: Optional[int] = None,
                     seqlen: Optional[int] = None, dstate: Optional[int] = None) -> dict:
    """Generate the seeded inputs of a prefill-scan workload.

    Sizes can be overridden (same recipe, different shape) for parity cases.
    Returns a dict of Tensor (u, delta, z, B, C) and fp32 arrays (A, D, delta_bias, h0).
    """
    Bt = batch or cfg.batch
    Dm = dim or cfg.dim
    L = seqlen or cfg.seqlen
    N = dstate or cfg.dstate
    sb = cfg.seed_base
    out = {"batch": Bt, "dim": Dm, "seqlen": L, "dstate": N, "cfg": cfg}
    out["u"] = Tensor(_normal(sb + K_U, (Bt, Dm, L)), cfg.in_dtype)
    out["delta"] = Tensor(_normal(sb + K_DELTA, (Bt, Dm, L), std=0.5), cfg.in_dtype)
    out["z"] = Tensor(_normal(sb + K_Z, (Bt, Dm, L)), cfg.in_dtype) if cfg.has_z else None
    out["B"] = Tensor(_normal(sb + K_B, (Bt, N, L)), cfg.in_dtype)
    out["C"] = Tensor(_normal(sb + K_C, (Bt, N, L)), cfg.in_dtype)
    if cfg.A_kind == "s4d_real":
        out["A"] = s4d_real_A(Dm, N)
    else:
        g = _rng(sb + K_A)
        out["A"] = (-np.exp(g.uniform(math.log(0.5), math.log(4.0), size=(Dm, N)))).astype(np.float32)
    out["D"] = _normal(sb + K_D, (Dm,)) if cfg.has_D else None
    out["delta_bias"] = delta_bias(sb + K_BIAS, Dm)
    out["h0"] = _normal(sb + K_H0, (Bt, Dm, N)) if cfg.h0 == "normal" else None
    out["softplus"] = cfg.softplus
    return out


def make_decode_inputs(cfg: DecodeConfig, batch: Optional[int] = None,
                       dim: Optional[int] = None, token_sets: Optional[int] = None) -> dict:
    """Generate the seeded decode workload: initial state and per-step token sets.

    state ~ N(0,1) fp32 (batch, dim, dstate); per token set k: x, delta, z
    (batch, dim) and B, C (batch, dstate) ~ N(0,1) in cfg.in_dtype, seeds
    base + 100*k + {u,delta,z,B,C}. A = S4D-real, D ~ N(0,1), delta_bias as the
    prefill recipe; softplus on.
    """
    Bt = batch or cfg.batch
    Dm = dim or cfg.dim
    N = cfg.dstate
    S = token_sets or cfg.token_sets
    sb = cfg.seed_base
    sets = []
    for k in range(S):
        o = sb + 100 * (k + 1)
        sets.append({
            "x": Tensor(_normal(o + K_U, (Bt, Dm)), cfg.in_dtype),
            "delta": Tensor(_normal(o + K_DELTA, (Bt, Dm)), cfg.in_dtype),
            "z": Tensor(_normal(o + K_Z, (Bt, Dm)), cfg.in_dtype),
            "B": Tensor(_normal(o + K_B, (Bt, N)), cfg.in_dtype),
            "C": Tensor(_normal(o + K_C, (Bt, N)), cfg.in_dtype),
        })
    return {
        "batch": Bt, "dim": Dm, "dstate": N, "cfg": cfg,
        "state": _normal(sb + K_H0, (Bt, Dm, N)),
        "A": s4d_real_A(Dm, N),
        "D": _normal(sb + K_D, (Dm,)),
        "delta_bias": delta_bias(sb + K_BIAS, Dm),
        "softplus": True,
        "sets": sets,
    }


def make_conv_inputs(cfg: ConvConfig, batch: Optional[int] = None, dim: Optional[int] = None,
                     seqlen: Optional[int] = None, width: Optional[int] = None,
                     with_state: bool = True) -> dict:
    """Seeded inputs of the causal conv1d: x ~ N(0, 1) in cfg.in_dtype (batch, dim, L);
    weight (dim, width) and bias (dim) ~ U(-1/sqrt(width), 1/sqrt(width)) fp32 (the
    bound of PyTorch's default Conv1d init for a depthwise kernel, fan-in = width);
    conv_state (batch, dim, width-1) = earlier inputs, N(0, 1) rounded like x, held
    in fp32. Seeds base + {x: 1, weight: 2, bias: 3, state: 4}."""
    Bt = batch or cfg.batch
    Dm = dim or cfg.dim
    L = cfg.seqlen if seqlen is None else seqlen
    W_ = width or cfg.width
    sb = cfg.seed_base
    bound = 1.0 / math.sqrt(W_)
    out = {"batch": Bt, "dim": Dm, "seqlen": L, "width": W_, "cfg": cfg}
    out["x"] = Tensor(_normal(sb + 1, (Bt, Dm, L)), cfg.in_dtype)
    out["weight"] = _rng(sb + 2).uniform(-bound, bound, size=(Dm, W_)).astype(np.float32)
    out["bias"] = _rng(sb + 3).uniform(-bound, bound, size=(Dm,)).astype(np.float32)
    st = Tensor(_normal(sb + 4, (Bt, Dm, W_ - 1)), cfg.in_dtype).f32() if with_state else None
    out["conv_state"] = None if st is None else np.ascontiguousarray(st, dtype=np.float32)
    return out


def make_ssd_inputs(cfg: SsdConfig, batch: Optional[int] = None, seqlen: Optional[int] = None,
                    nheads: Optional[int] = None, ngroups: Optional[int] = None,
                    dstate: Optional[int] = None) -> dict:
    """Seeded inputs of an SSD workload (sizes overridable).

    x, z, B, C ~ N(0, 1) and dt ~ N(0, 0.5), stored bf16; A_h = -exp(A_log_h) with
    A_log ~ N(0, 1) (the page's Mamba2Block.__init__ draws A_log = randn(n_heads));
    dt_bias_h = softplus^-1(dt0_h), dt0_h = exp(U(log 1e-3, log 1e-1)); D ~ N(0, 1);
    h0 ~ N(0, 1) (batch, nheads, headdim, dstate) fp32 or None. Seeds base + k as
    the prefill recipe (x=1, dt=2, z=3, B=4, C=5, A=6, D=7, bias=8, h0=9).
    """
    Bt = batch or cfg.batch
    L = cfg.seqlen if seqlen is None else seqlen
    H = nheads or cfg.nheads
    G = ngroups or cfg.ngroups
    N = dstate or cfg.dstate
    P = cfg.headdim
    sb = cfg.seed_base
    out = {"batch": Bt, "seqlen": L, "nheads": H, "headdim": P, "ngroups": G, "dstate": N, "cfg": cfg}
    out["x"] = Tensor(_normal(sb + K_U, (Bt, L, H, P)), BF16)
    out["dt"] = Tensor(_normal(sb + K_DELTA, (Bt, L, H), std=0.5), BF16)
    out["z"] = Tensor(_normal(sb + K_Z, (Bt, L, H, P)), BF16) if cfg.has_z else None
    out["B"] = Tensor(_normal(sb + K_B, (Bt, L, G, N)), BF16)
    out["C"] = Tensor(_normal(sb + K_C, (Bt, L, G, N)), BF16)
    out["A"] = (-np.exp(_normal(sb + K_A, (H,)).astype(np.float64))).astype(np.float32)
    out["D"] = _normal(sb + K_D, (H,)) if cfg.has_D else None
    out["dt_bias"] = delta_bias(sb + K_BIAS, H)
    out["h0"] = _normal(sb + K_H0, (Bt, H, P, N)) if cfg.h0 == "normal" else None
    return out
