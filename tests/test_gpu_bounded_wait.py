"""The bounded waits of the bulk-copy kernels, exercised without a fault: a GPU thread waits on an
mbarrier that nothing completes (a flag that nothing sets), gives up after the limit, records
GQ_ERR_TIMEOUT (5) in the workspace status word, and the context stays usable (a fused
allreduce-mean afterwards matches the same call made before)."""
import pytest

from gpu_common import gq_module

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    return gq_module()


@pytest.mark.parametrize("limit_ms", [20, 200])
def test_wait_gives_up_and_reports(gq, limit_ms):
    import torch
    from allreduce_compatible_gradient_gb300 import workloads
    x = workloads.device_inputs("normal", 4, 1 << 20, seed=2)
    ws = gq.gq_workspace()
    before = gq.gq_allreduce_mean(x, 2, 2, gq.EXP, 4, 1, 0, ws=ws)
    assert gq.gq_get_status(ws) == 0
    status, waited_ns = gq.gq_selftest_wait_timeout(limit_ms * 1_000_000, ws=ws)
    assert status == 5 and gq.gq_status_string(status) == "device wait timed out"
    assert limit_ms * 1e6 <= waited_ns < limit_ms * 1e6 + 1e9  # gave up soon after the limit
    assert gq.gq_get_status(ws) == 0  # reading the status cleared it
    after = gq.gq_allreduce_mean(x, 2, 2, gq.EXP, 4, 1, 0, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(before, after)
    assert gq.gq_get_status(ws) == 0


def test_selftest_argument_checks(gq):
    import torch
    ws = gq.gq_workspace()
    with pytest.raises(gq.GQError):
        gq.gq_selftest_wait_timeout(10, ws=ws)  # below 1 us
    with pytest.raises(gq.GQError):
        gq.gq_selftest_wait_timeout(5_000_000_000, ws=ws)  # above 4 s
    with pytest.raises(gq.GQError):
        gq.gq_selftest_wait_timeout(1_000_000, ws=torch.empty(16, dtype=torch.uint8, device="cuda"))
