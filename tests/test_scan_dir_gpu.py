"""GPU parity of the directional scans and the zero-order-hold input matrix
(ssm_scan_fwd_dir) against the fp64 oracle's oracle_scan_dir, through the C ABI.

Tolerances are the scan's (max|err| / rms(oracle)): 1e-5 for fp32 inputs, 2e-3 for
bf16 inputs on an fp32 y and for h_last, and elementwise 2e-3 rms plus half a bf16
ulp for a bf16 y. The zero-order-hold factor (exp(dt A) - 1) / A comes from the
decay the kernel already forms: exactly as expm1 on the fp32 path, as a - 1 from
the SFU exponential on the bf16 path (about 2e-4 relative at dt |A| = 1e-3,
inside the bf16 bound)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from workloads.torch_io import scan_to_torch
from tests.parity import assert_state_close, assert_y_close, to_np

pytestmark = pytest.mark.gpu

ORDERS = ["raster", "reverse", "columns", "columns_reverse"]


@pytest.fixture(scope="module")
def ssm():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import selective_state_space_121_b300 as m
    return m


def _inputs(in_dtype, batch, dim, rows, cols, N, h0=True, seed_cfg="mamba130m"):
    cfg = dataclasses.replace(W.CONFIGS[seed_cfg], in_dtype=in_dtype, h0="normal" if h0 else "zero")
    inp = W.make_scan_inputs(cfg, batch=batch, dim=dim, seqlen=rows * cols, dstate=N)
    if N != cfg.dstate:
        inp["A"] = W.s4d_real_A(dim, N)
    return inp


def _run(ssm, inp, order, rows, cols, zoh, out_dtype=torch.float32):
    t = scan_to_torch(inp)
    y, hl = ssm.scan_fwd_dir(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                             t["h0"], order=order, rows=rows, cols=cols, zoh=zoh, out_dtype=out_dtype)
    torch.cuda.synchronize()
    z = inp["z"]
    ref = oracle.scan_dir(inp["u"].f32(), inp["delta"].f32(), inp["A"], inp["B"].f32(), inp["C"].f32(), inp["D"],
                          None if z is None else z.f32(), inp["delta_bias"], True, inp["h0"],
                          order=W_ORDER[order], rows=rows, cols=cols, zoh=zoh)
    return y, hl, ref


W_ORDER = {name: i for i, name in enumerate(ORDERS)}


def _check(y, hl, ref, tol, out_bf16, what):
    assert_y_close(to_np(y), ref[0], tol, out_bf16, what)
    assert_state_close(to_np(hl), ref[1], tol, what + " h_last")


@pytest.mark.parametrize("zoh", [False, True], ids=["dtB", "zoh"])
@pytest.mark.parametrize("in_dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("order", ORDERS)
@pytest.mark.parametrize("N", [1, 4, 16])
def test_dir_parity(ssm, order, in_dtype, zoh, N):
    rows, cols = 23, 29                        # 667 steps: three 256-step chunks, the last ragged
    inp = _inputs(in_dtype, 2, 40, rows, cols, N)
    y, hl, ref = _run(ssm, inp, order, rows, cols, zoh)
    _check(y, hl, ref, 1e-5 if in_dtype == W.F32 else 2e-3, False, f"{order} zoh={zoh}")


@pytest.mark.parametrize("order", ORDERS)
def test_dir_bf16_out(ssm, order):
    inp = _inputs(W.BF16, 2, 24, 16, 20, 16)
    y, hl, ref = _run(ssm, inp, order, 16, 20, True, out_dtype=torch.bfloat16)
    _check(y, hl, ref, 2e-3, True, order)


def test_zoh_zero_A_limit(ssm):
    """Channels with A = 0 take the limit dt * B of the hold."""
    inp = _inputs(W.F32, 2, 16, 7, 9, 4)
    inp["A"] = inp["A"].copy()
    inp["A"][::3, 1] = 0.0
    y, hl, ref = _run(ssm, inp, "columns", 7, 9, True)
    _check(y, hl, ref, 1e-5, False, "A = 0")


@pytest.mark.parametrize("rows,cols", [(1, 37), (37, 1), (1, 1), (256, 1), (2, 128)])
@pytest.mark.parametrize("order", ["columns", "columns_reverse"])
def test_dir_degenerate_grids(ssm, rows, cols, order):
    """A single row or column (the column order is then the raster or its transpose),
    one step, and chunk-sized grids."""
    inp = _inputs(W.F32, 1, 9, rows, cols, 8)
    y, hl, ref = _run(ssm, inp, order, rows, cols, False)
    _check(y, hl, ref, 1e-5, False, f"{order} {rows}x{cols}")


def test_dir_empty(ssm):
    inp = _inputs(W.BF16, 2, 8, 1, 4, 16)
    t = scan_to_torch(inp)
    e = {k: t[k][..., :0].contiguous() for k in ("u", "delta", "B", "C", "z")}
    y, hl = ssm.scan_fwd_dir(e["u"], e["delta"], t["A"], e["B"], e["C"], t["D"], e["z"], t["delta_bias"], True,
                             t["h0"], order="reverse")
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.equal(hl, t["h0"])


def test_dir_raster_matches_forward_scan(ssm):
    """The raster order is the forward scan: same kernel arithmetic as the warp-scan
    algorithm of ssm_scan_fwd_algo, so the outputs agree to rounding."""
    inp = _inputs(W.BF16, 2, 16, 12, 40, 16)
    t = scan_to_torch(inp)
    y1, h1 = ssm.scan_fwd_dir(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                              t["h0"], order="raster", out_dtype=torch.float32)
    y2, h2 = ssm.scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True, t["h0"],
                          algo="warpscan", out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.allclose(y1, y2, rtol=1e-5, atol=1e-5) and torch.allclose(h1, h2, rtol=1e-5, atol=1e-5)


def test_vmamba56_four_directions_sampled(ssm):
    """The (8, 192, 56 x 56, 16) bf16 image workload the bench times, all four
    directions; the oracle checks 12 sampled channels of each in full."""
    cfg = W.CONFIGS["vmamba56"]
    rows, cols = W.IMAGE_GRIDS["vmamba56"]
    inp = W.make_scan_inputs(cfg)
    t = scan_to_torch(inp)
    rng = np.random.default_rng(17)
    chans = sorted({(0, 0), (cfg.batch - 1, cfg.dim - 1)} |
                   {(int(rng.integers(cfg.batch)), int(rng.integers(cfg.dim))) for _ in range(10)})
    u32, d32, z32 = inp["u"].f32(), inp["delta"].f32(), inp["z"].f32()
    B32, C32 = inp["B"].f32(), inp["C"].f32()
    for order in ORDERS:
        y, hl = ssm.scan_fwd_dir(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                                 None, order=order, rows=rows, cols=cols, out_dtype=torch.float32)
        torch.cuda.synchronize()
        for b, d in chans:
            sl = (slice(b, b + 1), slice(d, d + 1))
            ref = oracle.scan_dir(u32[sl], d32[sl], inp["A"][d:d + 1], B32[b:b + 1], C32[b:b + 1],
                                  inp["D"][d:d + 1], z32[sl], inp["delta_bias"][d:d + 1], True, None,
                                  order=W_ORDER[order], rows=rows, cols=cols)
            assert_y_close(to_np(y[sl]), ref[0], 2e-3, False, f"{order} ({b}, {d})")
            assert_state_close(to_np(hl[sl]), ref[1], 2e-3, f"{order} h_last ({b}, {d})")


@pytest.mark.parametrize("order", ORDERS)
@pytest.mark.parametrize("shape", [(5, 1000, 25, 40), (1, 128, 100, 200)], ids=["serial", "lookback"])
def test_dir_prefill_algorithms(ssm, order, shape):
    """With a workspace, every walk of bf16 inputs with 16-byte aligned rows runs on
    the prefill's own algorithms: the time-serial scan (5,000 channels, work-balanced)
    and the look-back (128 channels, 20,000 steps, ~79 segments of 256 steps); the
    reversed walks mirror every bulk copy, the column walks scan transposed copies.
    Against the oracle, with h0, y in fp32."""
    bt, dim, rows, cols = shape
    inp = _inputs(W.BF16, bt, dim, rows, cols, 16)
    y, hl, ref = _run(ssm, inp, order, rows, cols, False)
    _check(y, hl, ref, 2e-3, False, f"{order} {shape}")
    # and the same outputs as the warp-scan form, to the prefill's tolerance
    t = scan_to_torch(inp)
    y2, h2 = ssm.scan_fwd_dir(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                              t["h0"], order=order, rows=rows, cols=cols, out_dtype=torch.float32, workspace=None)
    torch.cuda.synchronize()
    scale = y2.pow(2).mean().sqrt().item()
    assert (y - y2).abs().max().item() <= 2e-3 * scale


@pytest.mark.parametrize("order", ORDERS)
@pytest.mark.parametrize("case", [
    dict(in_dtype=W.BF16, N=16, rows=7, cols=143, h0=True),    # L = 1001: unaligned rows, reversed walks fall back
    dict(in_dtype=W.F32, N=16, rows=13, cols=37, h0=False),    # fp32: no bulk copies, reversed walks fall back
    dict(in_dtype=W.BF16, N=8, rows=24, cols=40, h0=True),     # d_state 8
], ids=["bf16_L1001", "f32", "N8"])
def test_dir_prefill_algorithms_edges(ssm, order, case):
    """Every order with a workspace on shapes that take the time-serial kernel (5,000
    channels), where the prefill paths apply and where they must fall back to the
    warp scan; against the oracle."""
    rows, cols = case["rows"], case["cols"]
    inp = _inputs(case["in_dtype"], 5, 1000, rows, cols, case["N"], h0=case["h0"])
    y, hl, ref = _run(ssm, inp, order, rows, cols, False)
    _check(y, hl, ref, 1e-5 if case["in_dtype"] == W.F32 else 2e-3, False, f"{order} {case}")
