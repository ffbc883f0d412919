"""GPU parity of the Mamba-2 SSD scan (ssm_ssd_scan_fwd, tcgen05 tensor cores) against
the fp64 oracle's multi-head recurrence, through the C ABI.

Tolerance. The inputs are bf16, so the bf16 bound of the scan applies: max|err| /
rms(oracle) <= 2e-3 for an fp32 y and for h_last; a bf16 y is checked elementwise
against 2e-3 rms plus half a bf16 ulp. The kernel's own error is far below it:
x, B and C enter the tensor cores exactly, the three computed operands (the
decay-masked C B^T, the carried state, the decay-weighted x) are split into bf16
high and low parts (about 2^-17 relative), dt and the decays are fp32."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from workloads.torch_io import ssd_to_torch, to_torch
from tests.parity import assert_state_close, assert_y_close, to_np

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def ssm():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import selective_state_space_121_b300 as m
    return m


def _inputs(cfg_name="ssd_tiny", **kw):
    cfg = W.SSD_CONFIGS[cfg_name]
    opts = {k: kw.pop(k) for k in ("has_D", "has_z", "h0") if k in kw}
    if opts:
        cfg = dataclasses.replace(cfg, **opts)
    return W.make_ssd_inputs(cfg, **kw)


def _oracle(inp, softplus=True, bias=True, dt_override=None):
    z = inp["z"]
    dt = inp["dt"].f32() if dt_override is None else dt_override
    return oracle.ssd_scan(inp["x"].f32(), dt, inp["A"], inp["B"].f32(), inp["C"].f32(), inp["D"],
                           None if z is None else z.f32(), inp["dt_bias"] if bias else None, softplus, inp["h0"])


def _run(ssm, inp, out_dtype=torch.float32, softplus=True, bias=True, dt=None, in_place=False):
    t = ssd_to_torch(inp)
    if dt is not None:
        t["dt"] = dt
    h_last = None
    if in_place:
        assert t["h0"] is not None
        h_last = t["h0"]
    y, hl = ssm.ssd_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["z"],
                             t["dt_bias"] if bias else None, softplus, t["h0"], out_dtype=out_dtype, h_last=h_last)
    torch.cuda.synchronize()
    assert ssm.device_status() == 0
    return y, hl


def _check(y, hl, ref, out_dtype, what="ssd"):
    yr, hr = ref
    assert_y_close(to_np(y), yr, TOL, out_dtype == torch.bfloat16, what)
    assert_state_close(to_np(hl), hr, TOL, what + " h_last")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["y_f32", "y_bf16"])
@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("G", [1, 2])
def test_ssd_parity(ssm, out_dtype, N, G):
    inp = _inputs(dstate=N, ngroups=G)
    y, hl = _run(ssm, inp, out_dtype)
    _check(y, hl, _oracle(inp), out_dtype)


@pytest.mark.parametrize("L", [1, 5, 127, 128, 129, 256, 1000])
def test_ssd_lengths(ssm, L):
    """Ragged chunk tails, exact chunk multiples and a single step."""
    inp = _inputs(seqlen=L, batch=1, nheads=3, ngroups=1)
    y, hl = _run(ssm, inp)
    _check(y, hl, _oracle(inp), torch.float32, f"L={L}")


@pytest.mark.parametrize("opts", [dict(has_z=False), dict(has_D=False), dict(h0="zero"),
                                  dict(has_z=False, has_D=False, h0="zero")],
                         ids=["no_z", "no_D", "no_h0", "bare"])
def test_ssd_options(ssm, opts):
    inp = _inputs(**opts)
    y, hl = _run(ssm, inp)
    _check(y, hl, _oracle(inp), torch.float32)


def test_ssd_no_bias_and_raw_dt(ssm):
    """Without dt_bias, and with softplus off on a positive dt (dt taken as given)."""
    inp = _inputs(seqlen=260)
    y, hl = _run(ssm, inp, bias=False)
    _check(y, hl, _oracle(inp, bias=False), torch.float32, "no bias")
    # positive raw dt: softplus(dt + bias) rounded to bf16, then passed with softplus off
    v = inp["dt"].f32().astype(np.float64) + inp["dt_bias"][None, None, :]
    dtp = np.where(v > 20, v, np.log1p(np.exp(v))).astype(np.float32)
    dt_t = W.Tensor(dtp, W.BF16)
    y, hl = _run(ssm, inp, softplus=False, bias=False, dt=to_torch(dt_t))
    _check(y, hl, _oracle(inp, softplus=False, bias=False, dt_override=dt_t.f32()), torch.float32, "raw dt")


def test_ssd_state_in_place_and_resume(ssm):
    """h_last written over h0, and two calls (L1 then L2 from the first's h_last) equal
    one call over L1 + L2."""
    inp = _inputs(seqlen=384, batch=1)
    t = ssd_to_torch(inp)
    h = t["h0"].clone()
    y_full, h_full = ssm.ssd_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["z"], t["dt_bias"],
                                      True, h, out_dtype=torch.float32)
    _check(y_full, h_full, _oracle(inp), torch.float32, "full")
    L1 = 200
    s1 = {k: t[k][:, :L1].contiguous() for k in ("x", "dt", "B", "C", "z")}
    s2 = {k: t[k][:, L1:].contiguous() for k in ("x", "dt", "B", "C", "z")}
    y1, _ = ssm.ssd_scan_fwd(s1["x"], s1["dt"], t["A"], s1["B"], s1["C"], t["D"], s1["z"], t["dt_bias"], True,
                             h, out_dtype=torch.float32, h_last=h)            # in place
    y2, h2 = ssm.ssd_scan_fwd(s2["x"], s2["dt"], t["A"], s2["B"], s2["C"], t["D"], s2["z"], t["dt_bias"], True,
                              h, out_dtype=torch.float32)
    torch.cuda.synchronize()
    _check(torch.cat([y1, y2], 1), h2, _oracle(inp), torch.float32, "resumed")


def test_ssd_empty(ssm):
    inp = _inputs(seqlen=4, batch=1)
    t = ssd_to_torch(inp)
    e = {k: t[k][:, :0].contiguous() for k in ("x", "dt", "B", "C", "z")}
    y, hl = ssm.ssd_scan_fwd(e["x"], e["dt"], t["A"], e["B"], e["C"], t["D"], e["z"], t["dt_bias"], True, t["h0"])
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert torch.equal(hl, t["h0"])


def test_ssd_deterministic(ssm):
    inp = _inputs()
    y1, h1 = _run(ssm, inp)
    y2, h2 = _run(ssm, inp)
    assert torch.equal(y1, y2) and torch.equal(h1, h2)


def test_ssd_full_size_sampled(ssm):
    """The (4, 4096, 80 heads x 64, d_state 64) bf16 workload the bench times; the oracle
    runs 8 sampled (batch, head) pairs over the whole sequence."""
    cfg = W.SSD_CONFIGS["ssd_5120"]
    inp = W.make_ssd_inputs(cfg)
    t = ssd_to_torch(inp)
    y, hl = ssm.ssd_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["z"], t["dt_bias"], True, t["h0"])
    torch.cuda.synchronize()
    assert ssm.device_status() == 0
    rng = np.random.default_rng(9)
    pairs = {(0, 0), (cfg.batch - 1, cfg.nheads - 1)} | {(int(rng.integers(cfg.batch)), int(rng.integers(cfg.nheads)))
                                                        for _ in range(6)}
    x, dt, z = inp["x"].f32(), inp["dt"].f32(), inp["z"].f32()
    Bv, Cv = inp["B"].f32(), inp["C"].f32()
    for b, h in sorted(pairs):
        g = h // (cfg.nheads // cfg.ngroups)
        yr, hr = oracle.ssd_scan(x[b:b + 1, :, h:h + 1], dt[b:b + 1, :, h:h + 1], inp["A"][h:h + 1],
                                 Bv[b:b + 1, :, g:g + 1], Cv[b:b + 1, :, g:g + 1], inp["D"][h:h + 1],
                                 z[b:b + 1, :, h:h + 1], inp["dt_bias"][h:h + 1], True, None)
        assert_y_close(to_np(y[b:b + 1, :, h:h + 1]), yr, TOL, True, f"(b={b}, h={h})")
        assert_state_close(to_np(hl[b:b + 1, h:h + 1]), hr, TOL, f"h_last (b={b}, h={h})")


# -- the work-balanced launch (a workspace, more sequences than SMs, not whole rounds) --
# (2, 300, 80 heads): 160 sequences of 3 chunks on 148 CTAs, runs of 3.2 chunks (the
# tail of one sequence and the head of the next); (3, 260, 100 heads), d_state 128,
# 2 groups: 300 sequences, runs of 6.1 chunks (a tail, whole sequences, a head).
BAL_CASES = [dict(batch=2, seqlen=300, nheads=80, ngroups=1, dstate=64),
             dict(batch=3, seqlen=260, nheads=100, ngroups=2, dstate=128)]


def _run_ws(ssm, inp, workspace, out_dtype=torch.float32):
    t = ssd_to_torch(inp)
    y, hl = ssm.ssd_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["z"], t["dt_bias"], True, t["h0"],
                             out_dtype=out_dtype, workspace=workspace)
    torch.cuda.synchronize()
    assert ssm.device_status() == 0
    return y, hl


@pytest.mark.parametrize("case", BAL_CASES, ids=["160seq", "300seq_N128"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["y_f32", "y_bf16"])
def test_ssd_balanced_matches_oracle(ssm, case, out_dtype):
    inp = _inputs(**case)
    y, hl = _run_ws(ssm, inp, "auto", out_dtype)
    _check(y, hl, _oracle(inp), out_dtype, "balanced")


@pytest.mark.parametrize("case", BAL_CASES, ids=["160seq", "300seq_N128"])
def test_ssd_balanced_bitwise_equals_plain(ssm, case):
    """The state crosses each split as the fp32 values in tensor memory and enters the
    next piece on the path h0 takes (split for G3, rescaled for G4): the same
    arithmetic as the one-sequence-per-CTA launch."""
    inp = _inputs(**case)
    y1, h1 = _run_ws(ssm, inp, "auto", torch.bfloat16)
    y2, h2 = _run_ws(ssm, inp, None, torch.bfloat16)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(h1.view(torch.int32), h2.view(torch.int32))


@pytest.mark.parametrize("L", [1, 129, 385], ids=["L1", "L129", "L385"])
def test_ssd_balanced_short_and_ragged(ssm, L):
    """The work-balanced launch with one-chunk sequences and one-step tail chunks."""
    inp = _inputs(batch=2, seqlen=L, nheads=80, ngroups=1, dstate=64)
    y, hl = _run_ws(ssm, inp, "auto", torch.float32)
    _check(y, hl, _oracle(inp), torch.float32, f"balanced L={L}")
