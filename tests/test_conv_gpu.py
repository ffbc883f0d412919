"""GPU parity of the causal depthwise conv1d (+ silu) and its decode update against
the fp64 oracle, through the C ABI.

Tolerance. Each output is a sum of at most five fp32 products and a bias, then a
silu, computed from the exact stored inputs: its error is a few fp32 roundings
plus the silu's (about 1e-6 relative on the bf16 path's SFU form), so the bound is
1e-5 max|err| / rms(oracle) for an fp32 output and, elementwise, 1e-5 rms plus half
a bf16 ulp for a bf16 output. The conv states are copies of inputs: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from workloads.torch_io import to_torch
from tests.parity import assert_y_close, to_np

pytestmark = pytest.mark.gpu

TOL = 1e-5
DT = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module")
def ssm():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import selective_state_space_121_b300 as m
    return m


def _cfg(in_dtype, out_dtype):
    return W.ConvConfig("t", 1, 1, 1, 4, W.BF16 if in_dtype == "bf16" else W.F32,
                        W.BF16 if out_dtype == "bf16" else W.F32, 6100)


def _run(ssm, inp, out_dtype, silu=True, use_bias=True, use_state=True, inplace=False):
    x = to_torch(inp["x"])
    w = to_torch(inp["weight"])
    b = to_torch(inp["bias"]) if use_bias else None
    st = to_torch(inp["conv_state"]) if use_state and inp["conv_state"] is not None else None
    if inplace:
        assert st is not None
        out, so = ssm.causal_conv1d_fwd(x, w, b, st, silu, out_dtype=DT[out_dtype], conv_state_out=st)
        assert so is st
    else:
        out, so = ssm.causal_conv1d_fwd(x, w, b, st, silu, out_dtype=DT[out_dtype])
    torch.cuda.synchronize()
    ref, rso = oracle.causal_conv1d(inp["x"].f32(), inp["weight"], inp["bias"] if use_bias else None,
                                    inp["conv_state"] if use_state else None, silu)
    return out, so, ref, rso


def _check(out, so, ref, rso, out_dtype, what="conv"):
    assert_y_close(to_np(out), ref, TOL, out_dtype == "bf16", what)
    assert np.array_equal(to_np(so), rso), f"{what}: conv state differs"


@pytest.mark.parametrize("dt", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32"), ("f32", "bf16")],
                         ids=lambda d: f"{d[0]}-{d[1]}")
@pytest.mark.parametrize("width", [1, 2, 3, 4])
@pytest.mark.parametrize("shape", [(2, 24, 1000), (1, 3, 4097), (3, 40, 257)], ids=str)
def test_conv_parity(ssm, dt, width, shape):
    bt, dim, L = shape
    inp = W.make_conv_inputs(_cfg(*dt), batch=bt, dim=dim, seqlen=L, width=width)
    _check(*_run(ssm, inp, dt[1]), dt[1])


@pytest.mark.parametrize("silu,use_bias,use_state", [(False, True, True), (True, False, False),
                                                     (False, False, False)])
def test_conv_options(ssm, silu, use_bias, use_state):
    inp = W.make_conv_inputs(_cfg("bf16", "f32"), batch=2, dim=16, seqlen=600, width=4)
    out, so, ref, rso = _run(ssm, inp, "f32", silu, use_bias, use_state)
    _check(out, so, ref, rso, "f32")


@pytest.mark.parametrize("L", [0, 1, 2, 3, 7, 255, 256, 257])
@pytest.mark.parametrize("dt", [("bf16", "bf16"), ("f32", "f32")], ids=lambda d: d[0])
def test_conv_short_and_ragged(ssm, L, dt):
    """Lengths below the state width (the outgoing state mixes old state and x), at and
    around a block edge, and rows that are not 16-byte multiples (scalar path)."""
    inp = W.make_conv_inputs(_cfg(*dt), batch=2, dim=5, seqlen=L, width=4)
    _check(*_run(ssm, inp, dt[1]), dt[1], f"conv L={L}")


def test_conv_in_place_state(ssm):
    inp = W.make_conv_inputs(_cfg("bf16", "bf16"), batch=2, dim=8, seqlen=2, width=4)
    _check(*_run(ssm, inp, "bf16", inplace=True), "bf16", "in place, L < width-1")
    inp = W.make_conv_inputs(_cfg("bf16", "bf16"), batch=1, dim=2, seqlen=9000, width=4)
    _check(*_run(ssm, inp, "bf16", inplace=True), "bf16", "in place, several segments")


def test_conv_empty(ssm):
    inp = W.make_conv_inputs(_cfg("bf16", "bf16"), batch=0, dim=4, seqlen=16, width=4)
    x = torch.empty((0, 4, 16), dtype=torch.bfloat16, device="cuda")
    out, so = ssm.causal_conv1d_fwd(x, to_torch(inp["weight"]), to_torch(inp["bias"]), None, True)
    torch.cuda.synchronize()
    assert out.shape == (0, 4, 16) and so.shape == (0, 4, 3)


def test_conv_update_matches_oracle_and_prefill(ssm):
    """T decode updates equal the oracle step by step, and together equal one prefill
    conv over the same T inputs from the same state (both on the GPU)."""
    T = 24
    inp = W.make_conv_inputs(W.CONV_CONFIGS["conv_decode"], batch=16, dim=320, seqlen=T)
    x = to_torch(inp["x"])
    w, b = to_torch(inp["weight"]), to_torch(inp["bias"])
    st = to_torch(inp["conv_state"]).clone()
    ost = inp["conv_state"].astype(np.float64).copy()
    outs = []
    for t in range(T):
        xt = x[..., t].contiguous()
        o = ssm.causal_conv1d_update(st, xt, w, b, True)
        outs.append(o)
        ref = oracle.conv_update(ost, inp["x"].f32()[..., t], inp["weight"], inp["bias"], True)
        torch.cuda.synchronize()
        assert_y_close(to_np(o), ref, TOL, True, f"update t={t}")
    assert np.array_equal(to_np(st), ost)
    pre, pso = ssm.causal_conv1d_fwd(x, w, b, to_torch(inp["conv_state"]), True)
    torch.cuda.synchronize()
    assert torch.equal(torch.stack(outs, -1), pre)
    assert torch.equal(pso, st)


@pytest.mark.parametrize("width", [1, 2, 3])
def test_conv_update_widths(ssm, width):
    inp = W.make_conv_inputs(_cfg("f32", "f32"), batch=3, dim=70, seqlen=5, width=width)
    x = to_torch(inp["x"])
    w, b = to_torch(inp["weight"]), to_torch(inp["bias"])
    st = to_torch(inp["conv_state"]).clone()
    ost = inp["conv_state"].astype(np.float64).copy()
    for t in range(5):
        o = ssm.causal_conv1d_update(st, x[..., t].contiguous(), w, b, True)
        ref = oracle.conv_update(ost, inp["x"].f32()[..., t], inp["weight"], inp["bias"], True)
        torch.cuda.synchronize()
        assert_y_close(to_np(o), ref, TOL, False, f"update w={width} t={t}")
    assert np.array_equal(to_np(st), ost)


def test_conv_full_size_sampled(ssm):
    """The (8, 1536, 2048) bf16 conv feeding the Mamba-130M-shaped scan, in the launch
    configuration the bench times; the oracle checks 48 sampled rows in full."""
    cfg = W.CONV_CONFIGS["conv_mamba130m"]
    inp = W.make_conv_inputs(cfg)
    out, so = ssm.causal_conv1d_fwd(to_torch(inp["x"]), to_torch(inp["weight"]), to_torch(inp["bias"]),
                                    to_torch(inp["conv_state"]), True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows = sorted({(0, 0), (cfg.batch - 1, cfg.dim - 1)} |
                  {(int(rng.integers(cfg.batch)), int(rng.integers(cfg.dim))) for _ in range(46)})
    for b, d in rows:
        ref, rso = oracle.causal_conv1d(inp["x"].rows_f32((b, np.array([d])))[None], inp["weight"][[d]],
                                        inp["bias"][[d]], inp["conv_state"][b, [d]][None], True)
        assert_y_close(to_np(out[b, d]), ref[0, 0], TOL, True, f"row ({b}, {d})")
        assert np.array_equal(to_np(so[b, d]), rso[0, 0])
