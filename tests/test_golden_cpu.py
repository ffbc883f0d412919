"""The oracle reproduces the stored worked cases of tests/golden/, and the exact
integer case equals its closed form h = h0 + cumsum(B * u) (decay factors all 1)."""
import numpy as np
import pytest

import oracle
from tests import golden_io


@pytest.mark.parametrize("name", golden_io.NAMES)
def test_oracle_reproduces_golden(name):
    fx = golden_io.load(name)
    i = fx["inputs"]
    y, h = oracle.scan(i["u"], i["delta"], i["A"], i["B"], i["C"], i["D"], i["z"], i["delta_bias"],
                       fx["softplus"], None if i["h0"] is None else i["h0"].astype(np.float64))
    np.testing.assert_allclose(y, fx["expected"]["y"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(h, fx["expected"]["h_last"], rtol=1e-14, atol=1e-14)


def test_exact_integer_closed_form():
    fx = golden_io.load("exact_integer")
    i = fx["inputs"]
    u, B, C, D, h0 = (i[k].astype(np.float64) for k in ("u", "B", "C", "D", "h0"))
    # h[b,d,n,t] = h0[b,d,n] + sum_{s<=t} B[b,n,s] u[b,d,s]
    h = h0[:, :, :, None] + np.cumsum(B[:, None, :, :] * u[:, :, None, :], axis=-1)
    y = np.einsum("bdnt,bnt->bdt", h, C) + D[None, :, None] * u
    assert np.array_equal(y, fx["expected"]["y"])
    assert np.array_equal(h[..., -1], fx["expected"]["h_last"])
