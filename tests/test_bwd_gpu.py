"""GPU parity of the selective-scan backward (ssm_scan_bwd) against the fp64 oracle's
backward (itself pinned by finite differences of the forward), through the C ABI.

Tolerance (the pages fix none for gradients; derived from the arithmetic). The
kernel recomputes the forward states in fp32 and carries the adjoint g = dl/dh in
fp32 backwards; over a channel's memory (up to ~1/(dt |A|) ~ 1e3 steps at the
recipe's dt >= 1e-3) the relative rounding of fp32 (6e-8 per step) accumulates to
~6e-5, so fp32 inputs are held to 2e-4 max|err| / rms per gradient tensor. bf16
inputs take the forward's SFU forms (dt to ~1e-4 relative), so their gradients
are held to the bf16 forward bound, 2e-3; a bf16 gradient output adds half a bf16
ulp elementwise. dB and dC are sums over channels accumulated with atomics (order
varies run to run), covered by the same bounds."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from workloads.torch_io import scan_to_torch
from tests.parity import assert_y_close, rel_err, to_np

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-4, "bf16": 2e-3}


@pytest.fixture(scope="module")
def ssm():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import selective_state_space_121_b300 as m
    return m


def _case(cfg_name, bt, dim, L, N, in_dtype, seed=0, with_z=True, with_D=True, with_bias=True, h0=True):
    cfg = W.CONFIGS[cfg_name]
    import dataclasses
    cfg = dataclasses.replace(cfg, in_dtype=in_dtype, has_z=with_z, has_D=with_D,
                              h0="normal" if h0 else "zero")
    inp = W.make_scan_inputs(cfg, batch=bt, dim=dim, seqlen=L, dstate=N)
    if N != cfg.dstate and cfg.A_kind == "s4d_real":
        inp["A"] = W.s4d_real_A(dim, N)
    if not with_bias:
        inp["delta_bias"] = None
    rng = np.random.default_rng(100 + seed)
    dout = rng.standard_normal((bt, dim, L)).astype(np.float32)
    dhl = rng.standard_normal((bt, dim, N)).astype(np.float32)
    return inp, dout, dhl


def _run(ssm, inp, dout, dhl, dout_dtype=torch.float32):
    t = scan_to_torch(inp)
    dt = torch.from_numpy(dout).to("cuda", dout_dtype)
    g = ssm.scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                     t["h0"], dout=dt, dh_last=torch.from_numpy(dhl).cuda())
    torch.cuda.synchronize()
    dout64 = to_np(dt)
    z = inp["z"]
    ref = oracle.scan_bwd(inp["u"].f32(), inp["delta"].f32(), inp["A"], inp["B"].f32(), inp["C"].f32(), inp["D"],
                          None if z is None else z.f32(), inp["delta_bias"], True, inp["h0"], dout64,
                          dhl.astype(np.float64))
    return g, ref


def _check(g, ref, in_dtype):
    tol = TOL[in_dtype]
    for k in ("du", "ddelta", "dz"):
        if ref[k] is None or g[k] is None:
            assert (ref[k] is None) == (g[k] is None), k
            continue
        assert_y_close(to_np(g[k]), ref[k], tol, g[k].dtype == torch.bfloat16, k)
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias", "dh0"):
        if g[k] is None:
            continue
        r = rel_err(to_np(g[k]), ref[k])
        assert r <= tol, f"{k}: max|err|/rms = {r:.3e} > {tol:.1e}"


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [16, 8, 4, 2, 1])
def test_bwd_parity_dstate(ssm, in_dtype, N):
    inp, dout, dhl = _case("mamba130m", 2, 40, 203, N, W.F32 if in_dtype == "f32" else W.BF16, seed=N)
    g, ref = _run(ssm, inp, dout, dhl)
    _check(g, ref, in_dtype)


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
def test_bwd_dout_other_width(ssm, in_dtype):
    """dout narrower (bf16 for fp32 inputs) or wider (fp32 for bf16 inputs) than the inputs."""
    inp, dout, dhl = _case("mamba130m", 2, 24, 77, 16, W.F32 if in_dtype == "f32" else W.BF16, seed=5)
    g, ref = _run(ssm, inp, dout, dhl, torch.bfloat16 if in_dtype == "f32" else torch.float32)
    _check(g, ref, in_dtype)


@pytest.mark.parametrize("opts", [dict(with_z=False), dict(with_D=False), dict(with_bias=False),
                                  dict(h0=False), dict(with_z=False, with_D=False, with_bias=False, h0=False)],
                         ids=["no_z", "no_D", "no_bias", "no_h0", "bare"])
def test_bwd_options(ssm, opts):
    inp, dout, dhl = _case("mamba130m", 2, 24, 96, 16, W.F32, seed=7, **opts)
    g, ref = _run(ssm, inp, dout, dhl)
    _check(g, ref, "f32")


@pytest.mark.parametrize("L", [1, 7, 8, 9, 64, 1000])
def test_bwd_lengths(ssm, L):
    inp, dout, dhl = _case("mamba130m", 1, 36, L, 16, W.BF16, seed=L)
    g, ref = _run(ssm, inp, dout, dhl, torch.bfloat16)
    _check(g, ref, "bf16")


def test_bwd_long_sequence(ssm):
    """A long fp32 sequence: the adjoint runs 4096 steps back through the checkpoints."""
    inp, dout, dhl = _case("tiny", 1, 16, 4096, 16, W.F32, seed=3)
    g, ref = _run(ssm, inp, dout, dhl)
    _check(g, ref, "f32")


def test_bwd_mamba130m_full_size(ssm):
    """The (8, 1536, 2048, 16) bf16 layer the bench times; every gradient against the
    oracle (dB and dC need every channel, so the oracle runs the whole problem)."""
    inp, dout, dhl = _case("mamba130m", 8, 1536, 2048, 16, W.BF16, seed=11)
    g, ref = _run(ssm, inp, dout, dhl, torch.bfloat16)
    _check(g, ref, "bf16")


def test_bwd_empty(ssm):
    """No time steps: every per-step gradient is empty, the summed ones are zero and
    dh0 is dh_last (the adjoint passes through zero steps unchanged)."""
    inp, dout, dhl = _case("mamba130m", 2, 40, 8, 16, W.BF16, seed=1)
    t = scan_to_torch(inp)
    e = {k: t[k][..., :0].contiguous() for k in ("u", "delta", "B", "C", "z")}   # zero steps
    g = ssm.scan_bwd(e["u"], e["delta"], t["A"], e["B"], e["C"], t["D"], e["z"], t["delta_bias"], True, t["h0"],
                     dout=torch.empty((2, 40, 0), dtype=torch.bfloat16, device="cuda"),
                     dh_last=torch.from_numpy(dhl).cuda())
    torch.cuda.synchronize()
    assert g["du"].numel() == 0 and g["dB"].numel() == 0
    for k in ("dA", "dD", "ddelta_bias"):
        assert torch.count_nonzero(g[k]).item() == 0, k
    assert torch.equal(g["dh0"].cpu(), torch.from_numpy(dhl))
