"""Closed forms from the pages, in numpy fp64 -- TEST INFRASTRUCTURE ONLY.

These are second, independent statements of what the selective scan computes in
special cases. The pin tests compare the sequential oracle (ssm_oracle.c)
against them; they are not used by the CUDA path.
"""
from __future__ import annotations

import numpy as np


def sm1_closed_form(dA, dBx, h0, C, segment: int = 32):
    """d_state = 1 closed form of the Scalar Mamba1 (SM1) page (aitrends.kr),
    section details: with Lc = cumprod(dA) along time,
        h = Lc * (h0 + cumsum(dBx / Lc)),  y = h * C.

    dA, dBx, C: (..., T) along the last axis; h0: (...,).
    The page divides by Lc after clamping it at 1e-6; that clamp makes the
    identity inexact once the cumulative product underflows the clamp. The
    identity itself is exact, so this evaluates it unclamped and restarts
    (rebases) the products every `segment` steps, carrying h across segment
    boundaries, which keeps Lc far from underflow. Within a segment it is the
    page's cumprod/cumsum form verbatim.
    Returns (h (..., T), y (..., T)).
    """
    dA = np.asarray(dA, np.float64)
    dBx = np.asarray(dBx, np.float64)
    C = np.asarray(C, np.float64)
    carry = np.asarray(h0, np.float64).copy()
    T = dA.shape[-1]
    h = np.empty_like(dA)
    for s in range(0, T, segment):
        e = min(T, s + segment)
        Lc = np.cumprod(dA[..., s:e], axis=-1)
        h[..., s:e] = Lc * (carry[..., None] + np.cumsum(dBx[..., s:e] / Lc, axis=-1))
        carry = h[..., e - 1]
    return h, h * C


def sm1_literal_clamped(dA, dBx, h0, C):
    """The SM1 page's three lines taken literally, clamp included:
    L = cumprod(dA); h = L * (h0 + cumsum(dBx / clamp(L, min=1e-6))); y = h * C."""
    dA = np.asarray(dA, np.float64)
    Lc = np.cumprod(dA, axis=-1)
    h = Lc * (np.asarray(h0, np.float64)[..., None] + np.cumsum(dBx / np.maximum(Lc, 1e-6), axis=-1))
    return h, h * C


def lti_kernel(A, B, C, dt, L):
    """Convolution kernel of a time-invariant discretised SSM (Mamba SSM complete
    guide (youngju.dev), section 2, "SSM as a convolution kernel"):
        K = (C.Bbar, C.Abar.Bbar, C.Abar^2.Bbar, ...), y = K * u
    for diagonal A (one channel), Abar = exp(dt*A), Bbar = dt*B (the simplified
    input matrix the page's selective_scan uses). A, B, C: (N,). Returns K (L,).
    """
    A = np.asarray(A, np.float64)
    k = np.arange(L, dtype=np.float64)[:, None]
    Abar_pow = np.exp(k * dt * A[None, :])
    return (Abar_pow * (dt * np.asarray(B, np.float64))[None, :] * np.asarray(C, np.float64)[None, :]).sum(axis=1)


def causal_conv(K, u):
    """y_t = sum_{k=0..t} K_k u_{t-k} (direct O(L^2) causal convolution)."""
    L = len(u)
    y = np.zeros(L, dtype=np.float64)
    for t in range(L):
        y[t] = np.dot(K[: t + 1][::-1], u[: t + 1])
    return y


def affine_combine(p, q):
    """Compose two steps of x <- g*x + tok: applying p = (g1, t1) then q = (g2, t2)
    gives (g2*g1, g2*t1 + t2). This is the associative element of the parallel
    scan sketched in the guide's "Hardware-Aware Algorithm" section (the printed
    up-sweep reads an already-updated gate and the wrong multiplier; this is the
    standard composition it intends)."""
    g1, t1 = p
    g2, t2 = q
    return (g2 * g1, g2 * t1 + t2)


def tree_scan(gates, tokens, order_rng=None):
    """Inclusive scan of x_t = gates_t * x_{t-1} + tokens_t from x_{-1} = 0, by
    recursive halving with a random split point (any bracketing of an associative
    operator gives the same result). Returns x (T,)."""
    T = len(gates)
    elems = [(np.float64(gates[i]), np.float64(tokens[i])) for i in range(T)]

    def reduce(lo, hi):
        if hi - lo == 1:
            return elems[lo]
        mid = lo + 1 + (order_rng.integers(0, hi - lo - 1) if order_rng is not None else (hi - lo - 1) // 2)
        return affine_combine(reduce(lo, mid), reduce(mid, hi))

    out = np.empty(T)
    for t in range(T):
        out[t] = reduce(0, t + 1)[1]
    return out
