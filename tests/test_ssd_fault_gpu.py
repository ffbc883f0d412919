"""The SSD kernel's pipeline waits are bounded. With one compute-side arrival
withheld (a test hook: compute warp 0 skips its first "w o x ready" arrive), the
control warp's wait for it runs out after a short poll budget. The kernel records
the wait's source line, raises its abort flag so every other wait gives up, lets
the tensor core and the copies in flight finish, frees tensor memory and returns.
Nothing faults or hangs: the failure is a wait that nothing completes, and the
context stays usable. A normal SSD run afterwards matches the fp64 oracle."""
import pytest
import torch

from tests.test_ssd_gpu import TOL, _check, _inputs, _oracle, _run, ssm  # noqa: F401  (fixture)
from workloads.torch_io import ssd_to_torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N", [64, 128])
def test_withheld_arrival_is_reported_and_context_survives(ssm, N):
    inp = _inputs(dstate=N, ngroups=1)
    t = ssd_to_torch(inp)
    assert ssm.device_status(clear=True) == 0
    y = torch.empty(t["x"].shape, dtype=torch.bfloat16, device=t["x"].device)
    rc = ssm.run_ssd_wait_fault_test(t["x"], t["dt"], t["A"], t["B"], t["C"], y, wait_limit=1 << 14,
                                     withhold_arrive=True)
    assert rc == 0
    torch.cuda.synchronize()
    assert ssm.device_status(clear=True) == ssm.SSM_ERR_WAIT_TIMEOUT
    assert ssm.device_status(clear=True) == 0   # the record was cleared
    # the same short budget with nothing withheld completes without a record
    rc = ssm.run_ssd_wait_fault_test(t["x"], t["dt"], t["A"], t["B"], t["C"], y, wait_limit=1 << 20,
                                     withhold_arrive=False)
    assert rc == 0
    assert ssm.device_status(clear=True) == 0
    # and a normal run on the same context matches the oracle
    yn, hl = _run(ssm, inp)
    _check(yn, hl, _oracle(inp), torch.float32, f"after the fault, N={N}")


def test_wait_budget_is_validated(ssm):
    inp = _inputs()
    t = ssd_to_torch(inp)
    y = torch.empty(t["x"].shape, dtype=torch.bfloat16, device=t["x"].device)
    for bad in (0, -1, 1 << 31):
        assert ssm.run_ssd_wait_fault_test(t["x"], t["dt"], t["A"], t["B"], t["C"], y, wait_limit=bad,
                                           withhold_arrive=False) == ssm.SSM_ERR_DIM


def test_withheld_state_handover_is_reported_and_context_survives(ssm):
    """Work-balanced launch (160 sequences on 148 CTAs): ticket 5 withholds the state
    it would publish for ticket 6, whose hand-over wait then runs out after the short
    budget. The kernel records it, drains and returns; a normal balanced run on the
    same context afterwards matches the oracle."""
    inp = _inputs(batch=2, seqlen=300, nheads=80, ngroups=1, dstate=64)
    t = ssd_to_torch(inp)
    ws = torch.empty(ssm.ssd_workspace_size(2, 80, 64), dtype=torch.uint8, device=t["x"].device)
    assert ssm.device_status(clear=True) == 0
    y = torch.empty(t["x"].shape, dtype=torch.bfloat16, device=t["x"].device)
    rc = ssm.run_ssd_wait_fault_test(t["x"], t["dt"], t["A"], t["B"], t["C"], y, wait_limit=1 << 16,
                                     withhold_arrive=False, workspace=ws, drop_ticket=5)
    assert rc == 0
    torch.cuda.synchronize()
    assert ssm.device_status(clear=True) == ssm.SSM_ERR_WAIT_TIMEOUT
    yn, hl = _run(ssm, inp)
    _check(yn, hl, _oracle(inp), torch.float32, "after the withheld hand-over")
