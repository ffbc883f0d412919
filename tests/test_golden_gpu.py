"""The GPU path on the stored worked cases of tests/golden/ (every algorithm, fp32
and bf16 storage of the same exactly representable inputs), through the C ABI."""
import numpy as np
import pytest
import torch

from tests import golden_io
from tests.parity import assert_state_close, assert_y_close, to_np

pytestmark = pytest.mark.gpu

ALGOS = ["thread", "warpscan", "lookback", "auto"]


@pytest.fixture(scope="module")
def ssm():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import selective_state_space_121_b300 as m
    return m


def _dev(a, dtype=torch.float32):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_golden_scan(ssm, algo, dt):
    tin = torch.float32 if dt == "f32" else torch.bfloat16
    for name in ("exact_integer", "gated_small"):
        fx = golden_io.load(name)
        i = fx["inputs"]
        y, h = ssm.scan_fwd(_dev(i["u"], tin), _dev(i["delta"], tin), _dev(i["A"]), _dev(i["B"], tin),
                            _dev(i["C"], tin), _dev(i["D"]), _dev(i["z"], tin), _dev(i["delta_bias"]),
                            fx["softplus"], _dev(i["h0"]), out_dtype=torch.float32, algo=algo)
        torch.cuda.synchronize()
        if name == "exact_integer":
            assert np.array_equal(to_np(y), fx["expected"]["y"])
            assert np.array_equal(to_np(h), fx["expected"]["h_last"])
        else:
            tol = 1e-5 if dt == "f32" else 2e-3
            assert_y_close(to_np(y), fx["expected"]["y"], tol, False)
            assert_state_close(to_np(h), fx["expected"]["h_last"], tol)


def test_golden_scalar(ssm):
    fx = golden_io.load("scalar_small")
    i = fx["inputs"]
    y, h = ssm.scalar_scan_fwd(_dev(i["u"]), _dev(i["delta"]), _dev(i["A"][:, 0]), _dev(i["B"][:, 0]),
                               _dev(i["C"][:, 0]), None, None, _dev(i["delta_bias"]), fx["softplus"],
                               _dev(i["h0"][:, :, 0]))
    torch.cuda.synchronize()
    assert_y_close(to_np(y), fx["expected"]["y"], 1e-5, False)
    assert_state_close(to_np(h), fx["expected"]["h_last"][:, :, 0], 1e-5)
