"""Pins of the fp64 oracle: checks against what the pages and the mathematics fix,
never against the oracle itself. Each check takes an oracle.OracleLib and raises
AssertionError on a mismatch, so the same checks run on the real oracle and on
deliberately broken copies of its source (tests/test_oracle_pins.py).

Pages cited:
  [guide]  Mamba SSM complete guide (youngju.dev): section 2 "Discretization" and
           "SSM as a convolution kernel"; section 5 "Hardware-Aware Algorithm"
           (parallel scan) and "complete Mamba implementation" (selective_scan).
  [SM1]    Scalar Mamba1 (SM1) page (aitrends.kr), section details: the
           cumprod/cumsum closed form at d_state = 1.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

from oracle import forms


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = max(float(np.sqrt(np.mean(b * b))), 1e-300)
    return float(np.max(np.abs(a - b))) / scale


# ---------------------------------------------------------------------------
# 1. Brute force: the unrolled sum in exact rational arithmetic, tiny sizes.
#    h_t = (prod_{s<=t} a_s) h0 + sum_{s<=t} (prod_{s<r<=t} a_r) dt_s B_s u_s,
#    y_t = sum_n C_tn h_tn + D u_t, times silu(z_t)  ([guide] section 2, the
#    recurrence unrolled as the page does for the convolution view; section 5
#    selective_scan for dt*B and the D skip; MambaBlock.forward for the gate).
# ---------------------------------------------------------------------------
def _dyadic(rng, shape, den=8, lo=-16, hi=16):
    return (rng.integers(lo, hi + 1, size=shape) / den).astype(np.float32)


def check_bruteforce_rational(orc):
    rng = np.random.default_rng(7)
    for case in range(6):
        bt, dim, L, N = 2, 2, 1 + case % 4, 1 + case % 2
        u = _dyadic(rng, (bt, dim, L))
        delta = (rng.integers(1, 9, size=(bt, dim, L)) / 8).astype(np.float32)   # dt in (0, 1]
        bias = (rng.integers(0, 3, size=(dim,)) / 4).astype(np.float32)
        A = -(rng.integers(1, 9, size=(dim, N)) / 4).astype(np.float32)
        B = _dyadic(rng, (bt, N, L))
        C = _dyadic(rng, (bt, N, L))
        D = _dyadic(rng, (dim,)) if case % 3 else None
        z = _dyadic(rng, (bt, dim, L)) if case % 2 else None
        h0 = _dyadic(rng, (bt, dim, N)).astype(np.float64) if case >= 2 else None
        y, hl = orc.scan(u, delta, A, B, C, D, z, bias, False, h0)
        for b in range(bt):
            for d in range(dim):
                dt = [Fraction(float(delta[b, d, t])) + Fraction(float(bias[d])) for t in range(L)]
                a = [[Fraction(math.exp(float(dt[t]) * float(A[d, n]))) for n in range(N)] for t in range(L)]
                h_end = []
                for t in range(L):
                    acc = Fraction(0)
                    for n in range(N):
                        h = Fraction(float(h0[b, d, n])) if h0 is not None else Fraction(0)
                        for s in range(t + 1):
                            h *= a[s][n]
                        for s in range(t + 1):
                            w = Fraction(1)
                            for r in range(s + 1, t + 1):
                                w *= a[r][n]
                            h += w * dt[s] * Fraction(float(B[b, n, s])) * Fraction(float(u[b, d, s]))
                        acc += Fraction(float(C[b, n, t])) * h
                        if t == L - 1:
                            h_end.append(h)
                    if D is not None:
                        acc += Fraction(float(D[d])) * Fraction(float(u[b, d, t]))
                    if z is not None:
                        zz = float(z[b, d, t])
                        acc *= Fraction(zz) / (1 + Fraction(math.exp(-zz)))
                    assert abs(float(acc) - y[b, d, t]) <= 1e-14 * max(1.0, abs(float(acc))), (case, b, d, t)
                for n in range(N):
                    assert abs(float(h_end[n]) - hl[b, d, n]) <= 1e-14 * max(1.0, abs(float(h_end[n])))


def check_symbolic_two_steps(orc):
    """L = 2, N = 1 written out: y_2 = C_2 (a_2 (a_1 h0 + dt_1 B_1 u_1) + dt_2 B_2 u_2) + D u_2."""
    u = np.array([[[3.0, -2.0]]], np.float32)
    delta = np.array([[[0.5, 0.25]]], np.float32)
    A = np.array([[-2.0]], np.float32)
    B = np.array([[[1.5, -4.0]]], np.float32)
    C = np.array([[[2.0, 0.5]]], np.float32)
    D = np.array([0.75], np.float32)
    h0 = np.array([[[1.25]]])
    y, hl = orc.scan(u, delta, A, B, C, D, None, None, False, h0)
    a1, a2 = math.exp(-1.0), math.exp(-0.5)
    h1 = a1 * 1.25 + 0.5 * 1.5 * 3.0
    h2 = a2 * h1 + 0.25 * -4.0 * -2.0
    assert abs(y[0, 0, 0] - (2.0 * h1 + 0.75 * 3.0)) < 1e-14
    assert abs(y[0, 0, 1] - (0.5 * h2 + 0.75 * -2.0)) < 1e-14
    assert abs(hl[0, 0, 0] - h2) < 1e-14


# ---------------------------------------------------------------------------
# 2. Exact integer case: softplus off, delta = 1, A = 0 => Abar = exp(0) = 1,
#    so h_t = h0 + cumsum(B u) and y = C.h + D u are exact in floating point.
# ---------------------------------------------------------------------------
def check_exact_integer(orc):
    rng = np.random.default_rng(11)
    bt, dim, L, N = 3, 5, 37, 4
    u = rng.integers(-3, 4, size=(bt, dim, L)).astype(np.float32)
    delta = np.ones((bt, dim, L), np.float32)
    A = np.zeros((dim, N), np.float32)
    B = rng.integers(-3, 4, size=(bt, N, L)).astype(np.float32)
    C = rng.integers(-3, 4, size=(bt, N, L)).astype(np.float32)
    D = rng.integers(-3, 4, size=(dim,)).astype(np.float32)
    h0 = rng.integers(-5, 6, size=(bt, dim, N)).astype(np.float64)
    y, hl = orc.scan(u, delta, A, B, C, D, None, None, False, h0)
    ui = u.astype(np.int64)
    Bi = B.astype(np.int64)
    Ci = C.astype(np.int64)
    h = h0.astype(np.int64)[:, :, :, None] + np.cumsum(Bi[:, None, :, :] * ui[:, :, None, :], axis=3)
    yi = (Ci[:, None, :, :] * h).sum(axis=2) + D.astype(np.int64)[None, :, None] * ui
    assert np.array_equal(y, yi.astype(np.float64))
    assert np.array_equal(hl, h[:, :, :, -1].astype(np.float64))


# ---------------------------------------------------------------------------
# 3. Scalar functions: identities fixed by the mathematics.
#    softplus(x) - softplus(-x) = x; softplus(0) = ln 2; identity above 20
#    (PyTorch's default threshold, the reading taken for F.softplus).
#    silu(x) - silu(-x) = x; silu(0) = 0.
# ---------------------------------------------------------------------------
def check_softplus_silu(orc):
    for x in [0.1, 0.5, 1.0, 3.0, 7.5, 15.0]:
        assert abs((orc.softplus(x) - orc.softplus(-x)) - x) <= 4e-16 * max(1.0, x)
        assert abs((orc.silu(x) - orc.silu(-x)) - x) <= 4e-16 * max(1.0, x)
    assert abs(orc.softplus(0.0) - math.log(2.0)) <= 2e-16
    assert orc.softplus(25.0) == 25.0 and orc.softplus(20.5) == 20.5
    assert abs(orc.softplus(-30.0) / math.exp(-30.0) - 1.0) < 1e-12
    assert orc.silu(0.0) == 0.0
    assert abs(orc.silu(40.0) - 40.0) < 1e-12
    # inside the scan: A = 0, B = u = C = 1 => y_t = sum_{s<=t} softplus(delta_s + bias)
    rng = np.random.default_rng(3)
    L = 50
    delta = rng.standard_normal((1, 1, L)).astype(np.float32) * 3
    bias = np.array([0.625], np.float32)
    y, _ = orc.scan(np.ones((1, 1, L), np.float32), delta, np.zeros((1, 1), np.float32),
                    np.ones((1, 1, L), np.float32), np.ones((1, 1, L), np.float32), None, None,
                    bias, True, None)
    sp = np.logaddexp(0.0, delta[0, 0].astype(np.float64) + 0.625)
    assert _rel(y[0, 0], np.cumsum(sp)) < 1e-14


# ---------------------------------------------------------------------------
# 4. d_state = 1: the SM1 closed form h = Lc (h0 + cumsum(dBx / Lc)), y = h C,
#    Lc = cumprod(dA) ([SM1]; exact, per the page, at d_state = 1).
# ---------------------------------------------------------------------------
def _sm1_case(rng, bt=2, dim=4, L=600):
    u = rng.standard_normal((bt, dim, L)).astype(np.float32)
    delta = (rng.standard_normal((bt, dim, L)) * 0.5).astype(np.float32)
    dt0 = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=dim))
    bias = (dt0 + np.log(-np.expm1(-dt0))).astype(np.float32)
    A = (-np.exp(rng.uniform(math.log(0.5), math.log(4.0), size=(dim, 1)))).astype(np.float32)
    B = rng.standard_normal((bt, 1, L)).astype(np.float32)
    C = rng.standard_normal((bt, 1, L)).astype(np.float32)
    h0 = rng.standard_normal((bt, dim, 1))
    return u, delta, bias, A, B, C, h0


def check_sm1_closed_form(orc):
    rng = np.random.default_rng(21)
    u, delta, bias, A, B, C, h0 = _sm1_case(rng)
    y, hl = orc.scan(u, delta, A, B, C, None, None, bias, True, h0)
    dt = np.logaddexp(0.0, delta.astype(np.float64) + bias[None, :, None])
    dA = np.exp(dt * A[None, :, :1].astype(np.float64))
    dBx = dt * B.astype(np.float64) * u
    h, yc = forms.sm1_closed_form(dA, dBx, h0[..., 0], np.broadcast_to(C.astype(np.float64), u.shape))
    assert _rel(y, yc) < 1e-12
    assert _rel(hl[..., 0], h[..., -1]) < 1e-12


def check_sm1_literal_clamp_reading(orc):
    """The page's line with L.clamp(min=1e-6) agrees with the recurrence while the
    cumulative product stays above 1e-6, and departs from it after."""
    rng = np.random.default_rng(22)
    u, delta, bias, A, B, C, h0 = _sm1_case(rng, bt=1, dim=2, L=4000)
    A = np.full_like(A, -4.0)
    bias = np.full_like(bias, 0.5)           # dt ~ 1: cumprod falls below 1e-6 quickly
    y, _ = orc.scan(u, delta, A, B, C, None, None, bias, True, h0)
    dt = np.logaddexp(0.0, delta.astype(np.float64) + bias[None, :, None])
    dA = np.exp(dt * -4.0)
    dBx = dt * B.astype(np.float64) * u
    Lc = np.cumprod(dA, axis=-1)
    _, ylit = forms.sm1_literal_clamped(dA, dBx, h0[..., 0], C.astype(np.float64))
    ok = Lc >= 1e-6
    assert ok.any() and (~ok).any()
    scale = np.sqrt(np.mean(y * y))
    assert np.max(np.abs(ylit[ok] - y[ok])) < 1e-9 * scale
    assert np.max(np.abs(ylit[~ok] - y[~ok])) > 1e-3 * scale


# ---------------------------------------------------------------------------
# 5. Time-invariant case: dt, B, C constant over t => y = K * u + D u with
#    K_k = sum_n C_n exp(k dt A_n) dt B_n ([guide] section 2, "SSM as a
#    convolution kernel").
# ---------------------------------------------------------------------------
def check_lti_convolution(orc):
    rng = np.random.default_rng(5)
    L, N = 64, 4
    A = -np.array([[0.5, 1.0, 2.0, 4.0]], np.float32)
    dt = 0.15625
    Bn = rng.standard_normal(N).astype(np.float32)
    Cn = rng.standard_normal(N).astype(np.float32)
    u = rng.standard_normal((1, 1, L)).astype(np.float32)
    D = np.array([0.5], np.float32)
    y, _ = orc.scan(u, np.full((1, 1, L), dt, np.float32), A,
                    np.repeat(Bn[None, :, None], L, axis=2), np.repeat(Cn[None, :, None], L, axis=2),
                    D, None, None, False, None)
    K = forms.lti_kernel(A[0], Bn, Cn, dt, L)
    ref = forms.causal_conv(K, u[0, 0].astype(np.float64)) + 0.5 * u[0, 0]
    assert _rel(y[0, 0], ref) < 1e-12


# ---------------------------------------------------------------------------
# 6. Associativity: any bracketing of the affine pairs (g, tok) gives the
#    sequential result ([guide] section 5, Hardware-Aware Algorithm).
# ---------------------------------------------------------------------------
def check_tree_scan(orc):
    rng = np.random.default_rng(9)
    T = 48
    logg = np.log(rng.uniform(0.3, 0.99, size=(T,)))
    tokens = rng.standard_normal(T).astype(np.float32)
    # one channel, gate g_t = exp(-dt_t) through a time-varying dt_t = -log g_t and A = -1
    delta = (-logg).astype(np.float32)
    gates = np.exp(-delta.astype(np.float64))
    y, _ = orc.scan(np.ones((1, 1, T), np.float32), delta[None, None], np.array([[-1.0]], np.float32),
                    (tokens / delta)[None, None].astype(np.float32), np.ones((1, 1, T), np.float32),
                    None, None, None, False, None)
    tok = delta.astype(np.float64) * (tokens / delta).astype(np.float32).astype(np.float64)
    for seed in range(3):
        xs = forms.tree_scan(gates, tok, np.random.default_rng(seed))
        assert _rel(y[0, 0], xs) < 1e-13


# ---------------------------------------------------------------------------
# 7. Resume: a run over L1 then a run over L2 started from h_last equals one
#    run over L1 + L2 (state-based resume; the recurrence only carries h).
# ---------------------------------------------------------------------------
def _random_case(rng, bt, dim, L, N, z=True):
    u = rng.standard_normal((bt, dim, L)).astype(np.float32)
    delta = (rng.standard_normal((bt, dim, L)) * 0.5).astype(np.float32)
    dt0 = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=dim))
    bias = (dt0 + np.log(-np.expm1(-dt0))).astype(np.float32)
    A = -np.tile(np.arange(1, N + 1, dtype=np.float32), (dim, 1))
    B = rng.standard_normal((bt, N, L)).astype(np.float32)
    C = rng.standard_normal((bt, N, L)).astype(np.float32)
    D = rng.standard_normal(dim).astype(np.float32)
    zz = rng.standard_normal((bt, dim, L)).astype(np.float32) if z else None
    return u, delta, A, B, C, D, zz, bias


def check_resume(orc):
    rng = np.random.default_rng(13)
    u, delta, A, B, C, D, z, bias = _random_case(rng, 2, 3, 256, 16)
    h0 = rng.standard_normal((2, 3, 16))
    y, hl = orc.scan(u, delta, A, B, C, D, z, bias, True, h0)
    L1 = 100
    y1, h1 = orc.scan(u[..., :L1], delta[..., :L1], A, B[..., :L1], C[..., :L1], D, z[..., :L1], bias, True, h0)
    y2, h2 = orc.scan(u[..., L1:], delta[..., L1:], A, B[..., L1:], C[..., L1:], D, z[..., L1:], bias, True, h1)
    assert np.array_equal(np.concatenate([y1, y2], axis=-1), y)
    assert np.array_equal(h2, hl)


# ---------------------------------------------------------------------------
# 8. Recurrent / parallel duality: L single-token decode updates from h0 equal
#    the prefill scan over L ([guide] section 1/2: recurrence at inference).
# ---------------------------------------------------------------------------
def check_decode_equals_prefill(orc):
    rng = np.random.default_rng(17)
    u, delta, A, B, C, D, z, bias = _random_case(rng, 2, 3, 32, 8)
    h0 = rng.standard_normal((2, 3, 8))
    y, hl = orc.scan(u, delta, A, B, C, D, z, bias, True, h0)
    state = h0.copy()
    for t in range(32):
        yt = orc.state_update(state, u[..., t], delta[..., t], A, B[..., t], C[..., t], D, z[..., t], bias, True)
        assert np.array_equal(yt, y[..., t])
    assert np.array_equal(state, hl)


# ---------------------------------------------------------------------------
# 9. Linearity in (u, h0) for fixed dt, B, C (no gate): the map is linear.
# ---------------------------------------------------------------------------
def check_linearity(orc):
    rng = np.random.default_rng(19)
    bt, dim, L, N = 2, 3, 40, 4
    _, delta, A, B, C, D, _, bias = _random_case(rng, bt, dim, L, N, z=False)
    u1 = rng.integers(-8, 9, size=(bt, dim, L)).astype(np.float32)
    u2 = rng.integers(-8, 9, size=(bt, dim, L)).astype(np.float32)
    g1 = rng.integers(-8, 9, size=(bt, dim, N)).astype(np.float64)
    g2 = rng.integers(-8, 9, size=(bt, dim, N)).astype(np.float64)
    ya, ha = orc.scan(u1, delta, A, B, C, D, None, bias, True, g1)
    yb, hb = orc.scan(u2, delta, A, B, C, D, None, bias, True, g2)
    yc, hc = orc.scan(2 * u1 - 3 * u2, delta, A, B, C, D, None, bias, True, 2 * g1 - 3 * g2)
    assert _rel(yc, 2 * ya - 3 * yb) < 1e-13
    assert _rel(hc, 2 * ha - 3 * hb) < 1e-13


# ---------------------------------------------------------------------------
# 10. Limits: C = 0 => y = D u silu(z); dt -> 0 => the state stays at h0.
# ---------------------------------------------------------------------------
def check_limits(orc):
    rng = np.random.default_rng(23)
    u, delta, A, B, C, D, z, bias = _random_case(rng, 1, 4, 30, 4)
    y, _ = orc.scan(u, delta, A, B, np.zeros_like(C), D, z, bias, True, None)
    zz = z.astype(np.float64)
    ref = D[None, :, None].astype(np.float64) * u * (zz * 0.5 * (1.0 + np.tanh(zz / 2)))
    assert _rel(y, ref) < 1e-14
    h0 = rng.standard_normal((1, 4, 4))
    _, hl = orc.scan(u, np.full_like(delta, -60.0), A, B, C, D, z, None, True, h0)
    assert np.max(np.abs(hl - h0)) < 1e-20


# ---------------------------------------------------------------------------
# 11-13. The causal depthwise conv1d + silu before the scan ([guide] section 5,
#        "complete Mamba implementation": MambaBlock.__init__'s nn.Conv1d with
#        groups = d_inner, kernel d_conv, padding d_conv - 1, and forward's
#        trim to the first seqlen outputs and silu).
# ---------------------------------------------------------------------------
def check_conv_impulse(orc):
    """A unit impulse at t0 returns the kernel reversed (the current input meets the
    last weight: PyTorch's Conv1d is a cross-correlation), plus the bias everywhere;
    exact in fp64 for small integers."""
    dim, L, t0 = 3, 12, 4
    for width in (1, 2, 3, 4):
        w = (np.arange(dim * width, dtype=np.float32).reshape(dim, width) + 1)
        bias = np.array([0.5, -1.0, 2.0], np.float32)
        x = np.zeros((1, dim, L), np.float32)
        x[0, :, t0] = 1.0
        out, st = orc.causal_conv1d(x, w, bias, None, silu=False)
        ref = np.broadcast_to(bias[None, :, None].astype(np.float64), (1, dim, L)).copy()
        for j in range(width):
            ref[0, :, t0 + j] += w[:, width - 1 - j]
        assert np.array_equal(out, ref), (width, out, ref)
        assert np.array_equal(st, x[..., L - (width - 1):].astype(np.float64)) or width == 1


def check_conv_library(orc):
    """Equal to the library routine the page calls (torch.nn.functional.conv1d, fp64,
    padding width-1, groups = channels, first L outputs) followed by silu; with a
    state, equal to the same routine over [state | x] without padding."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(29)
    for width in (2, 3, 4):
        bt, dim, L = 2, 5, 37
        x = rng.standard_normal((bt, dim, L)).astype(np.float32)
        w = rng.standard_normal((dim, width)).astype(np.float32)
        bias = rng.standard_normal((dim,)).astype(np.float32)
        xt = torch.from_numpy(x.astype(np.float64))
        wt = torch.from_numpy(w.astype(np.float64))[:, None, :]
        bt_ = torch.from_numpy(bias.astype(np.float64))
        ref = F.silu(F.conv1d(xt, wt, bt_, padding=width - 1, groups=dim)[..., :L]).numpy()
        out, _ = orc.causal_conv1d(x, w, bias, None, silu=True)
        assert _rel(out, ref) < 1e-14
        st = rng.standard_normal((bt, dim, width - 1))
        full = torch.cat([torch.from_numpy(st), xt], dim=-1)
        ref2 = F.conv1d(full, wt, bt_, padding=0, groups=dim).numpy()
        out2, so = orc.causal_conv1d(x, w, bias, st, silu=False)
        assert _rel(out2, ref2) < 1e-14
        assert np.array_equal(so, x[..., L - (width - 1):].astype(np.float64))


def check_conv_resume_and_decode(orc):
    """conv(x1 ++ x2) = conv(x1) ++ conv(x2 from x1's final state); and L decode
    updates from a state equal one prefill call from it (same values, same state)."""
    rng = np.random.default_rng(31)
    bt, dim, L1, L2, width = 2, 3, 9, 14, 4
    x = rng.standard_normal((bt, dim, L1 + L2)).astype(np.float32)
    w = rng.standard_normal((dim, width)).astype(np.float32)
    bias = rng.standard_normal((dim,)).astype(np.float32)
    st0 = rng.standard_normal((bt, dim, width - 1))
    full, sf = orc.causal_conv1d(x, w, bias, st0, silu=True)
    a, sa = orc.causal_conv1d(x[..., :L1], w, bias, st0, silu=True)
    b, sb = orc.causal_conv1d(x[..., L1:], w, bias, sa, silu=True)
    assert np.array_equal(np.concatenate([a, b], -1), full) and np.array_equal(sb, sf)
    state = st0.copy()
    for t in range(L1 + L2):
        ot = orc.conv_update(state, x[..., t], w, bias, silu=True)
        assert np.array_equal(ot, full[..., t])
    assert np.array_equal(state, sf)
    # a call shorter than the state keeps the older state entries in order
    short, ss = orc.causal_conv1d(x[..., :1], w, bias, st0, silu=False)
    assert np.array_equal(ss, np.concatenate([st0[..., 1:], x[..., :1].astype(np.float64)], -1))


# ---------------------------------------------------------------------------
# 14. Backward: every gradient equals a central finite difference of the forward
#     oracle (pinned above) for the loss l = <dout, out> + <dh_last, h_last>, on
#     dyadic inputs where x +- 2^-10 is exact in fp32.
# ---------------------------------------------------------------------------
def check_bwd_finite_differences(orc):
    rng = np.random.default_rng(37)
    bt, dim, L, N = 2, 2, 5, 3
    eps = 2.0 ** -10

    def dy(shape, den=64, lo=-96, hi=96):
        return (rng.integers(lo, hi + 1, size=shape) / den).astype(np.float32)
    for with_z, sp in ((True, True), (False, False)):
        u, delta = dy((bt, dim, L)), dy((bt, dim, L), lo=-64, hi=32)
        z = dy((bt, dim, L)) if with_z else None
        B, C = dy((bt, N, L)), dy((bt, N, L))
        A = -(rng.integers(16, 128, size=(dim, N)) / 64).astype(np.float32)
        D = dy((dim,))
        bias = dy((dim,), lo=-32, hi=0)
        if not sp:       # raw dt must stay positive and modest
            delta = (rng.integers(4, 48, size=(bt, dim, L)) / 64).astype(np.float32)
            bias = np.zeros((dim,), np.float32)
        h0 = rng.standard_normal((bt, dim, N))
        dout = rng.standard_normal((bt, dim, L))
        dhl = rng.standard_normal((bt, dim, N))

        def loss(**kw):
            args = dict(u=u, delta=delta, A=A, B=B, C=C, D=D, z=z, bias=bias, h0=h0)
            args.update(kw)
            y, hl = orc.scan(args["u"], args["delta"], args["A"], args["B"], args["C"], args["D"], args["z"],
                             args["bias"], sp, args["h0"])
            return float(np.sum(dout * y) + np.sum(dhl * hl))
        g = orc.scan_bwd(u, delta, A, B, C, D, z, bias, sp, h0, dout, dhl)
        pairs = [("u", u, "du"), ("delta", delta, "ddelta"), ("B", B, "dB"), ("C", C, "dC"), ("A", A, "dA"),
                 ("D", D, "dD"), ("bias", bias, "ddelta_bias"), ("h0", h0, "dh0")]
        if with_z:
            pairs.append(("z", z, "dz"))
        for name, arr, gname in pairs:
            if name == "bias" and not sp:
                continue
            fd = np.zeros(arr.shape)
            for idx in np.ndindex(arr.shape):
                p_, m_ = arr.copy(), arr.copy()
                p_[idx] += eps
                m_[idx] -= eps
                fd[idx] = (loss(**{name: p_}) - loss(**{name: m_})) / (2 * eps)
            err = np.max(np.abs(fd - g[gname])) / max(1.0, float(np.max(np.abs(fd))))
            assert err < 2e-5, (name, with_z, err)


# ---------------------------------------------------------------------------
# 15. Mamba-2 SSM (the next row): the recurrence oracle against (a) the pinned
#     Mamba-1 oracle with every state of a head sharing its A, dt, B and C;
#     (b) the state space duality's quadratic (semi-separable matrix) form; and
#     (c) the chunked algorithm ([guide] section 6, "State Space Duality").
# ---------------------------------------------------------------------------
def _ssd_case(rng, bt=2, L=37, H=4, P=3, G=2, N=5, sp=True):
    x = rng.standard_normal((bt, L, H, P)).astype(np.float32)
    dt = (rng.standard_normal((bt, L, H)) * 0.5).astype(np.float32)
    A = -np.exp(rng.uniform(np.log(0.5), np.log(4.0), size=(H,))).astype(np.float32)
    B = rng.standard_normal((bt, L, G, N)).astype(np.float32)
    C = rng.standard_normal((bt, L, G, N)).astype(np.float32)
    D = rng.standard_normal((H,)).astype(np.float32)
    bias = (rng.uniform(-4, -2, size=(H,))).astype(np.float32)
    h0 = rng.standard_normal((bt, H, P, N))
    return x, dt, A, B, C, D, bias, h0


def check_ssd_matches_mamba1(orc):
    rng = np.random.default_rng(41)
    x, dt, A, B, C, D, bias, h0 = _ssd_case(rng)
    z = rng.standard_normal(x.shape).astype(np.float32)
    bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y, hl = orc.ssd_scan(x, dt, A, B, C, D, z, bias, True, h0)
    # channel (h, p) of Mamba-1: u = x[:, :, h, p], delta = dt[:, :, h], A_dn = A_h, B/C of the head's group
    for h in range(H):
        g = h // (H // G)
        u1 = np.ascontiguousarray(x[:, :, h, :].transpose(0, 2, 1))
        d1 = np.ascontiguousarray(np.repeat(dt[:, None, :, h], P, axis=1))
        z1 = np.ascontiguousarray(z[:, :, h, :].transpose(0, 2, 1))
        A1 = np.full((P, N), A[h], np.float32)
        B1 = np.ascontiguousarray(B[:, :, g, :].transpose(0, 2, 1))
        C1 = np.ascontiguousarray(C[:, :, g, :].transpose(0, 2, 1))
        y1, h1 = orc.scan(u1, d1, A1, B1, C1, np.full(P, D[h], np.float32), z1, np.full(P, bias[h], np.float32),
                          True, h0[:, h])
        assert _rel(y1.transpose(0, 2, 1), y[:, :, h, :]) < 1e-13
        assert _rel(h1, hl[:, h]) < 1e-13


def check_ssd_quadratic_and_chunked(orc):
    rng = np.random.default_rng(43)
    x, dt, A, B, C, D, bias, h0 = _ssd_case(rng, L=53)
    y, hl = orc.ssd_scan(x, dt, A, B, C, D, None, None, False, h0)       # raw dt: no softplus
    dt64 = dt.astype(np.float64)
    dtp = np.abs(dt64) + 0.01          # the forms below need the discretised dt itself
    y2, hl2 = orc.ssd_scan(x, dtp.astype(np.float32), A, B, C, D, None, None, False, h0)
    yq = forms.ssd_quadratic(x, dtp.astype(np.float32), A, B, C, D, h0)
    assert _rel(yq, y2) < 1e-11
    for q in (1, 7, 16, 64):
        yc, hc = forms.ssd_chunked(x, dtp.astype(np.float32), A, B, C, D, h0, chunk=q)
        assert _rel(yc, y2) < 1e-11 and _rel(hc, hl2) < 1e-11
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(hl))


# ---------------------------------------------------------------------------
# 16. Directional scans and the zero-order hold (the next row after Mamba-2):
#     (a) each traversal order equals the raster scan run on the inputs
#     rearranged by numpy (flip, transpose of the rows x cols image) with its
#     output rearranged back; (b) one zero-order-hold step equals the exact
#     solution of h' = A h + B u over the step (u held constant), taken from the
#     matrix exponential of the augmented 2 x 2 system ([guide] section 2,
#     "Discretization"), A = 0 included.
# ---------------------------------------------------------------------------
def _dir_case(rng, bt=2, dim=3, rows=5, cols=7, N=4):
    L = rows * cols
    u = rng.standard_normal((bt, dim, L)).astype(np.float32)
    delta = (rng.standard_normal((bt, dim, L)) * 0.5).astype(np.float32)
    z = rng.standard_normal((bt, dim, L)).astype(np.float32)
    A = -np.exp(rng.uniform(np.log(0.5), np.log(4.0), size=(dim, N))).astype(np.float32)
    B = rng.standard_normal((bt, N, L)).astype(np.float32)
    C = rng.standard_normal((bt, N, L)).astype(np.float32)
    D = rng.standard_normal((dim,)).astype(np.float32)
    bias = rng.uniform(-4, -1, size=(dim,)).astype(np.float32)
    h0 = rng.standard_normal((bt, dim, N))
    return u, delta, z, A, B, C, D, bias, h0


def check_scan_dir_orders(orc):
    rng = np.random.default_rng(47)
    rows, cols = 5, 7
    u, delta, z, A, B, C, D, bias, h0 = _dir_case(rng, rows=rows, cols=cols)
    bt, dim, L = u.shape

    def colmajor(a):   # raster (.., rows*cols) -> column-major sequence
        return np.ascontiguousarray(a.reshape(a.shape[:-1] + (rows, cols)).swapaxes(-1, -2).reshape(a.shape))

    def raster(a):     # inverse of colmajor
        return np.ascontiguousarray(a.reshape(a.shape[:-1] + (cols, rows)).swapaxes(-1, -2).reshape(a.shape))

    def flip(a):
        return np.ascontiguousarray(a[..., ::-1])

    forward = {1: (flip, flip), 2: (colmajor, raster), 3: (lambda a: flip(colmajor(a)), lambda a: raster(flip(a)))}
    for order, (to_seq, back) in forward.items():
        y, hl = orc.scan_dir(u, delta, A, B, C, D, z, bias, True, h0, order=order, rows=rows, cols=cols)
        y1, h1 = orc.scan(to_seq(u), to_seq(delta), A, to_seq(B), to_seq(C), D, to_seq(z), bias, True, h0)
        assert _rel(back(y1), y) < 1e-13, order
        assert _rel(h1, hl) < 1e-13, order
    y, hl = orc.scan_dir(u, delta, A, B, C, D, z, bias, True, h0, order=0)
    y1, h1 = orc.scan(u, delta, A, B, C, D, z, bias, True, h0)
    assert _rel(y1, y) == 0 and _rel(h1, hl) == 0


def check_scan_zoh_exact_step(orc):
    from scipy.linalg import expm
    rng = np.random.default_rng(53)
    bt, dim, N = 2, 3, 5
    u = rng.standard_normal((bt, dim, 1)).astype(np.float32)
    dt = np.exp(rng.uniform(np.log(0.05), np.log(1.5), size=(bt, dim, 1))).astype(np.float32)
    A = -np.exp(rng.uniform(np.log(0.3), np.log(4.0), size=(dim, N))).astype(np.float32)
    A[1, 2] = 0.0                                   # the A = 0 limit: dt * B
    B = rng.standard_normal((bt, N, 1)).astype(np.float32)
    C = rng.standard_normal((bt, N, 1)).astype(np.float32)
    h0 = rng.standard_normal((bt, dim, N))
    _, hl = orc.scan_dir(u, dt, A, B, C, None, None, None, False, h0, zoh=True)
    for b in range(bt):
        for d in range(dim):
            for n in range(N):
                # d/ds [h, 1] = [[A, B u], [0, 0]] [h, 1]  over s in [0, dt]
                M = np.array([[float(A[d, n]), float(B[b, n, 0]) * float(u[b, d, 0])], [0.0, 0.0]])
                e = expm(M * float(dt[b, d, 0])) @ np.array([h0[b, d, n], 1.0])
                assert abs(e[0] - hl[b, d, n]) <= 1e-12 * max(1.0, abs(e[0])), (b, d, n)
    # the simplified form differs from the hold wherever dt A is not small
    _, hs = orc.scan_dir(u, dt, A, B, C, None, None, None, False, h0, zoh=False)
    assert _rel(hs, hl) > 1e-3


ALL_CHECKS = [
    check_bruteforce_rational,
    check_symbolic_two_steps,
    check_exact_integer,
    check_softplus_silu,
    check_sm1_closed_form,
    check_sm1_literal_clamp_reading,
    check_lti_convolution,
    check_tree_scan,
    check_resume,
    check_decode_equals_prefill,
    check_linearity,
    check_limits,
    check_conv_impulse,
    check_conv_library,
    check_conv_resume_and_decode,
    check_bwd_finite_differences,
    check_ssd_matches_mamba1,
    check_ssd_quadratic_and_chunked,
    check_scan_dir_orders,
    check_scan_zoh_exact_step,
]
