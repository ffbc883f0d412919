"""Writes the small worked cases under tests/golden/ from the fp64 oracle only.

    python tests/golden/make_golden.py

Each fixture holds its inputs (small dyadic values, exact in fp32 and bf16) and
the oracle's y and h_last, with the passage it follows:
  * exact_integer.json -- softplus off, delta = 1, A = 0, so every decay factor
    is exactly 1 and h_t = h0 + cumsum(B * u) (the recurrence of the selective
    scan loop in "Mamba SSM complete guide", section 5, with a = 1); every value
    is a small integer, so any correct implementation reproduces it bit for bit.
  * gated_small.json -- the full operation of the same section (softplus(delta +
    bias), exp(dt A), dt B u, C contraction, D skip) with the block's silu(z)
    gate and a nonzero initial state, at a ragged length (L = 37, N = 4).
  * scalar_small.json -- the d_state = 1 case of the "SM1 (Scalar Mamba1)"
    page, section details, with h0 carried in.
Nothing here comes from the CUDA path.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def _dy(rng, shape, den=8, lo=-16, hi=16):
    return (rng.integers(lo, hi + 1, size=shape) / den).astype(np.float32)


def _case(name, cite, u, delta, A, B, C, D, z, bias, softplus, h0):
    y, hl = oracle.scan(u, delta, A, B, C, D, z, bias, softplus, None if h0 is None else h0.astype(np.float64))
    lst = lambda a: None if a is None else np.asarray(a, np.float64).tolist()  # noqa: E731
    return {"name": name, "cite": cite, "softplus": bool(softplus),
            "inputs": {"u": lst(u), "delta": lst(delta), "A": lst(A), "B": lst(B), "C": lst(C), "D": lst(D),
                       "z": lst(z), "delta_bias": lst(bias), "h0": lst(h0)},
            "expected": {"y": [[[float(v).hex() for v in row] for row in m] for m in y],
                         "h_last": [[[float(v).hex() for v in row] for row in m] for m in hl]}}


def main():
    rng = np.random.default_rng(20261202)
    bt, dim, L, N = 2, 3, 21, 4
    u = rng.integers(-3, 4, size=(bt, dim, L)).astype(np.float32)
    B = rng.integers(-3, 4, size=(bt, N, L)).astype(np.float32)
    C = rng.integers(-3, 4, size=(bt, N, L)).astype(np.float32)
    D = rng.integers(-3, 4, size=(dim,)).astype(np.float32)
    h0 = rng.integers(-5, 6, size=(bt, dim, N)).astype(np.float32)
    fx = _case("exact_integer",
               "Mamba SSM complete guide, section 5, selective_scan loop with a = exp(1 * 0) = 1",
               u, np.ones_like(u), np.zeros((dim, N), np.float32), B, C, D, None, None, False, h0)
    json.dump(fx, open(os.path.join(HERE, "exact_integer.json"), "w"))

    bt, dim, L, N = 2, 3, 37, 4
    u = _dy(rng, (bt, dim, L))
    delta = _dy(rng, (bt, dim, L), den=4, lo=-4, hi=4)
    A = -np.tile(np.arange(1, N + 1, dtype=np.float32), (dim, 1))
    B = _dy(rng, (bt, N, L))
    C = _dy(rng, (bt, N, L))
    D = _dy(rng, (dim,))
    z = _dy(rng, (bt, dim, L))
    bias = np.array([-2.25, -4.5, -6.75], np.float32)
    h0 = _dy(rng, (bt, dim, N))
    fx = _case("gated_small",
               "Mamba SSM complete guide, section 5: MambaBlock.ssm (softplus of delta plus the dt_proj bias), "
               "selective_scan (exp(delta A), delta B u, C contraction, D skip) and forward (silu(z) gate)",
               u, delta, A, B, C, D, z, bias, True, h0)
    json.dump(fx, open(os.path.join(HERE, "gated_small.json"), "w"))

    bt, dim, L = 2, 5, 29
    u = _dy(rng, (bt, dim, L))
    delta = _dy(rng, (bt, dim, L), den=4, lo=-4, hi=4)
    A = -np.array([[0.5], [1.0], [2.0], [3.0], [4.0]], np.float32)
    B = _dy(rng, (bt, 1, L))
    C = _dy(rng, (bt, 1, L))
    bias = np.array([-2.25, -3.0, -4.5, -5.25, -6.75], np.float32)
    h0 = _dy(rng, (bt, dim, 1))
    fx = _case("scalar_small", "SM1 (Scalar Mamba1) page, section details: d_state = 1 with h0 carried in",
               u, delta, A, B, C, None, None, bias, True, h0)
    json.dump(fx, open(os.path.join(HERE, "scalar_small.json"), "w"))


if __name__ == "__main__":
    main()
