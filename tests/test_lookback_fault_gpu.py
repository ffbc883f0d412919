"""The look-back wait is bounded: when a segment never publishes, the next one gives
up after its poll budget, records SSM_ERR_LOOKBACK_TIMEOUT in the workspace status
word, and the kernel finishes. Nothing faults or hangs; the context stays usable."""
import pytest
import torch

import workloads as W
from workloads.torch_io import scan_to_torch

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_context_survives():
    assert torch.cuda.is_available()
    import selective_state_space_121_b300 as ssm
    inp = W.make_scan_inputs(W.CONFIGS["long"], batch=1, dim=8, seqlen=8192)
    t = scan_to_torch(inp)
    ws = ssm.alloc_workspace(1, 8, 8192, 16)
    y = torch.empty_like(t["u"])
    rc = ssm.run_lookback_timeout_test(t["u"], t["delta"], t["A"], t["B"], t["C"], y, ws, drop_segment=1,
                                       spin_limit=2000)
    assert rc == 0
    assert ssm.query_status(ws) == ssm.SSM_ERR_LOOKBACK_TIMEOUT
    # a normal look-back scan on the same context and workspace runs clean afterwards
    y2, h2 = ssm.scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                          None, algo="lookback", workspace=ws)
    assert ssm.query_status(ws) == 0
    y3, _ = ssm.scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                         None, algo="warpscan")
    torch.cuda.synchronize()
    assert (y2.float() - y3.float()).abs().max().item() <= 2e-2 * y3.float().pow(2).mean().sqrt().item()
