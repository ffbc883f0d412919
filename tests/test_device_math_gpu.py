"""The device math helpers behind the scan's softplus, decays and gate, each held to
its stated error bound over a dense grid of its domain against numpy fp64 (through
the ssm_test_math hook of the C ABI). The scan's parity runs check them only
indirectly; these bounds are the ones their comments in common.cuh state:
  * exp (argument-error feedback on the SFU ex2): a few fp32 ulp, for x <= 88;
  * log1p on [0, 1] (fitted degree-8 polynomial): under 2e-7 relative;
  * expm1 (Cody-Waite reduction, Taylor polynomial): a few ulp relative;
  * accurate softplus and silu (fp32 inputs): a few 1e-7 relative;
  * SFU softplus log2(1 + 2^x) (bf16 inputs): the rounding of 1 + 2^x costs up to
    2^-24 absolute in dt, the SFU log2 about 2^-22 absolute, so the bound is
    absolute 4e-7 plus 4e-7 relative (about 1e-4 relative at dt = 1e-3);
  * SFU silu z / (1 + 2^(-z log2 e)): a few ulp of ex2 and rcp (1e-6 relative) plus
    the fp32 rounding of the exponent z log2 e, |z| 2^-24 absolute in it, which is
    |z| 2^-24 ln 2 log2 e = |z| 6e-8 relative in the result."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import selective_state_space_121_b300 as m
    return m


def _eval(ssm, fn, x64):
    x32 = x64.astype(np.float32)
    y = ssm.test_math(fn, torch.from_numpy(x32).cuda()).cpu().numpy().astype(np.float64)
    return x32.astype(np.float64), y


def _softplus64(x):
    return np.where(x > 20.0, x, np.log1p(np.exp(np.minimum(x, 20.0))))


def _silu64(x):
    return x / (1.0 + np.exp(-x))


def test_exp(ssm):
    x, y = _eval(ssm, "exp", np.linspace(-87.0, 88.0, 1 << 21))
    ref = np.exp(x)
    rel = np.abs(y - ref) / ref
    assert rel.max() <= 3.0e-7, rel.max()


def test_log1p_unit_interval(ssm):
    x, y = _eval(ssm, "log1p01", np.concatenate([np.linspace(0.0, 1.0, 1 << 20), np.geomspace(1e-30, 1e-3, 4096)]))
    ref = np.log1p(x)
    nz = ref > 0
    assert np.all(y[~nz] == 0.0)
    rel = np.abs(y[nz] - ref[nz]) / ref[nz]
    assert rel.max() <= 2.0e-7, rel.max()


def test_expm1(ssm):
    grid = np.concatenate([np.linspace(-88.0, 88.0, 1 << 21), np.geomspace(1e-30, 1.0, 8192),
                           -np.geomspace(1e-30, 1.0, 8192)])
    x, y = _eval(ssm, "expm1", grid)
    ref = np.expm1(x)
    nz = ref != 0
    rel = np.abs(y[nz] - ref[nz]) / np.abs(ref[nz])
    assert rel.max() <= 4.0e-7, rel.max()


def test_softplus_accurate(ssm):
    x, y = _eval(ssm, "softplus", np.linspace(-60.0, 60.0, 1 << 21))
    ref = _softplus64(x)
    rel = np.abs(y - ref) / ref
    assert rel.max() <= 5.0e-7, rel.max()


def test_silu_accurate(ssm):
    x, y = _eval(ssm, "silu", np.linspace(-80.0, 80.0, 1 << 21))
    ref = _silu64(x)
    nz = ref != 0
    rel = np.abs(y[nz] - ref[nz]) / np.abs(ref[nz])
    assert rel.max() <= 5.0e-7, rel.max()


def test_softplus_sfu(ssm):
    x, y = _eval(ssm, "softplus_sfu", np.linspace(-30.0, 60.0, 1 << 21))
    ref = _softplus64(x)
    err = np.abs(y - ref)
    assert np.all(err <= 4e-7 + 4e-7 * ref), float(np.max(err - 4e-7 * ref))


def test_silu_sfu(ssm):
    x, y = _eval(ssm, "silu_sfu", np.linspace(-80.0, 80.0, 1 << 21))
    ref = _silu64(x)
    nz = ref != 0
    rel = np.abs(y[nz] - ref[nz]) / np.abs(ref[nz])
    bound = 1e-6 + 6e-8 * np.abs(x[nz])
    assert np.all(rel <= bound), float(np.max(rel - bound))
