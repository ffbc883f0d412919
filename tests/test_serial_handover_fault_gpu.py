"""The state hand-over of the work-balanced time-serial scan is bounded: when a
ticket withholds the state it would publish, the next ticket's wait gives up after
its poll budget, records the failure (ssm_device_status reports
SSM_ERR_WAIT_TIMEOUT), continues from a zero state and the kernel finishes. Nothing
faults or hangs; the context stays usable and a normal run afterwards matches the
oracle."""
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_state_close, assert_y_close, to_np, tol_for
from workloads.torch_io import scan_to_torch

pytestmark = pytest.mark.gpu


def test_withheld_handover_is_reported_and_context_survives():
    assert torch.cuda.is_available()
    import selective_state_space_121_b300 as ssm
    # 160 channel groups of 32 on 148 CTAs: every run is a tail and a head
    inp = W.make_scan_inputs(W.CONFIGS["mamba130m"], batch=5, dim=1000, seqlen=1000)
    t = scan_to_torch(inp)
    ws = ssm.alloc_workspace(5, 1000, 1000, 16)
    assert ssm.device_status(clear=True) == 0
    y = torch.empty_like(t["u"])
    rc = ssm.run_serial_handover_timeout_test(t["u"], t["delta"], t["A"], t["B"], t["C"], y, ws,
                                              drop_ticket=7, spin_limit=2000)
    assert rc == 0
    torch.cuda.synchronize()
    assert ssm.device_status(clear=True) == ssm.SSM_ERR_WAIT_TIMEOUT
    # a normal balanced run on the same context and workspace runs clean afterwards
    y2, h2 = ssm.scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                          t["h0"], out_dtype=torch.float32, algo="thread", workspace=ws)
    torch.cuda.synchronize()
    assert ssm.device_status(clear=True) == 0
    yr, hr = oracle.scan_inputs(inp)
    tol = tol_for(inp["cfg"].in_dtype)
    assert_y_close(to_np(y2), yr, tol, False)
    assert_state_close(to_np(h2), hr, tol)
