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


def ssd_quadratic(x, dt, A, B, C, D=None, h0=None):
    """The state space duality form of the Mamba-2 SSM (Mamba SSM complete guide,
    section 6, "State Space Duality": an SSM with a scalar decay per head is a
    semi-separable matrix applied to the input). Per (batch, head), with
    cum_t = A sum_{r<=t} dt_r and the causal mask s <= t:
        M[t, s] = exp(cum_t - cum_s) (C_t . B_s) dt_s
        y_t = sum_s M[t, s] x_s + exp(cum_t) H0 C_t + D x_t
    (dt already discretised: softplus applied by the caller; no gate).
    x: (batch, L, H, P); dt: (batch, L, H); B, C: (batch, L, G, N); A, D: (H,);
    h0: (batch, H, P, N). fp64 matrix products."""
    x = np.asarray(x, np.float64); dt = np.asarray(dt, np.float64)
    B = np.asarray(B, np.float64); C = np.asarray(C, np.float64)
    bt, L, H, P = x.shape
    G = B.shape[2]
    y = np.zeros_like(x)
    for b in range(bt):
        for h in range(H):
            g = h // (H // G)
            cum = np.cumsum(dt[b, :, h]) * float(A[h])
            decay = np.exp(cum[:, None] - cum[None, :])
            mask = np.tril(np.ones((L, L), dtype=bool))
            M = np.where(mask, decay, 0.0) * (C[b, :, g, :] @ B[b, :, g, :].T) * dt[b, None, :, h]
            yh = M @ x[b, :, h, :]
            if h0 is not None:
                yh += np.exp(cum)[:, None] * (C[b, :, g, :] @ np.asarray(h0, np.float64)[b, h].T)
            if D is not None:
                yh += float(D[h]) * x[b, :, h, :]
            y[b, :, h, :] = yh
    return y


def ssd_chunked(x, dt, A, B, C, D=None, h0=None, chunk: int = 16):
    """The chunked SSD algorithm (same section: "inside a chunk, matrix products;
    across chunks, the recurrence carries the state"): per chunk of `chunk` steps,
    the intra-chunk part is the quadratic form above restricted to the chunk, the
    carried state H enters through exp(cum_t) H C_t, and the state leaves the chunk
    as H <- exp(cum_end) H + sum_s exp(cum_end - cum_s) dt_s x_s B_s^T.
    Same arguments as ssd_quadratic; returns (y, h_last)."""
    x = np.asarray(x, np.float64); dt = np.asarray(dt, np.float64)
    B = np.asarray(B, np.float64); C = np.asarray(C, np.float64)
    bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros_like(x)
    hl = np.zeros((bt, H, P, N))
    for b in range(bt):
        for h in range(H):
            g = h // (H // G)
            S = np.zeros((P, N)) if h0 is None else np.asarray(h0, np.float64)[b, h].copy()
            for c0 in range(0, L, chunk):
                c1 = min(L, c0 + chunk)
                d = dt[b, c0:c1, h]
                cum = np.cumsum(d) * float(A[h])
                Bc, Cc, xc = B[b, c0:c1, g, :], C[b, c0:c1, g, :], x[b, c0:c1, h, :]
                q = c1 - c0
                decay = np.where(np.tril(np.ones((q, q), dtype=bool)), np.exp(cum[:, None] - cum[None, :]), 0.0)
                yc = (decay * (Cc @ Bc.T) * d[None, :]) @ xc + np.exp(cum)[:, None] * (Cc @ S.T)
                if D is not None:
                    yc += float(D[h]) * xc
                y[b, c0:c1, h, :] = yc
                w = np.exp(cum[-1] - cum) * d
                S = np.exp(cum[-1]) * S + (xc * w[:, None]).T @ Bc
            hl[b, h] = S
    return y, hl
