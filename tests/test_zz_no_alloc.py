"""The allocation-free look-back entry point, ssm_scan_fwd_lookback_static.

Some callers cannot allocate device memory or hand the library a workspace: a
plugin running inside a host application that owns every device allocation, or a
latency-critical path that must not call cudaMalloc (which can synchronise the
device). For them the library runs its look-back scan on a fixed 4 MiB scratch
array of its own. These tests call that entry point through the C ABI and check
that two calls in a row (different sizes, so the second one meets what the first
left in the shared array) match the workspace entry point within the parity
tolerance for bf16 inputs and meet the fp64 oracle's 2e-3 bound themselves, and
that a problem needing more scratch is refused before anything is launched. The
file name makes pytest collect it last."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from workloads.torch_io import scan_to_torch
from tests.parity import TOL_BF16, assert_state_close, assert_y_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import selective_state_space_121_b300 as m
    return m


def test_static_scratch_matches_workspace_entry_point(ssm):
    for dim, L in ((8, 6000), (12, 9001)):
        inp = W.make_scan_inputs(W.CONFIGS["long"], batch=1, dim=dim, seqlen=L)
        t = scan_to_torch(inp)
        args = (t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True, None)
        # the several look-back segments these sizes cut time into use the scratch
        assert ssm.workspace_size(1, dim, L, 16) > 16
        y_ref, h_ref = ssm.scan_fwd(*args, out_dtype=torch.float32, algo="lookback")
        y = torch.empty((1, dim, L), dtype=torch.float32, device="cuda")
        h = torch.empty((1, dim, 16), dtype=torch.float32, device="cuda")
        assert ssm.scan_fwd_lookback_static(*args, y=y, h_last=h) == 0
        torch.cuda.synchronize()
        assert_y_close(to_np(y), to_np(y_ref), TOL_BF16, False)
        assert_state_close(to_np(h), to_np(h_ref), TOL_BF16)
        # and against the oracle on a sample of the channels
        chans = [(0, 0), (0, dim // 2), (0, dim - 1)]
        ref = oracle.scan_inputs(inp, chans)
        for (b, d) in chans:
            yr, hr = ref[(b, d)]
            assert_y_close(to_np(y[b, d]), yr, TOL_BF16, False, f"y channel {d}")
            assert_state_close(to_np(h[b, d]), hr, TOL_BF16, f"h_last channel {d}")


def test_static_scratch_refuses_oversized_problem(ssm):
    batch, dim, L, N = 1, 16384, 1 << 17, 16
    assert ssm.workspace_size(batch, dim, L, N) > ssm.STATIC_SCRATCH_BYTES
    fake = 0x10000   # never dereferenced: the size check comes before any CUDA call
    rc = ssm._lib.ssm_scan_fwd_lookback_static(fake, fake * 2, fake * 3, fake * 4, fake * 5, None, None, None, 1,
                                               None, fake * 6, None, batch, dim, L, N, 1, 1, None)
    assert rc == ssm.SSM_ERR_SCRATCH_LIMIT
    assert ssm.status_string(rc).startswith("SSM_ERR_SCRATCH_LIMIT")
