"""Move generated workloads (workloads.make_*_inputs) into torch tensors.

Storage is copied bit-for-bit: bf16 inputs keep the exact generated bits, so the
device sees the same values the fp64 oracle reads.
"""
from __future__ import annotations

import numpy as np
import torch

from . import BF16, Tensor


def to_torch(t, device="cuda", pin: bool = False):
    """Tensor or fp32 ndarray -> torch tensor (bf16 bits preserved); None stays None."""
    if t is None:
        return None
    if isinstance(t, Tensor):
        if t.dtype == BF16:
            x = torch.from_numpy(np.ascontiguousarray(t.storage).view(np.int16)).view(torch.bfloat16)
        else:
            x = torch.from_numpy(np.ascontiguousarray(t.storage))
    else:
        x = torch.from_numpy(np.ascontiguousarray(t, dtype=np.float32))
    if device == "cpu":
        return x.pin_memory() if pin else x
    return x.to(device)


def scan_to_torch(inp: dict, device="cuda", pin: bool = False) -> dict:
    keys = ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")
    return {k: to_torch(inp[k], device, pin) for k in keys}


def decode_set_to_torch(s: dict, device="cuda", pin: bool = False) -> dict:
    return {k: to_torch(v, device, pin) for k, v in s.items()}


def ssd_to_torch(inp: dict, device="cuda", pin: bool = False) -> dict:
    keys = ("x", "dt", "z", "B", "C", "A", "D", "dt_bias", "h0")
    return {k: to_torch(inp[k], device, pin) for k in keys}
