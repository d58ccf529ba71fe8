"""GPU parity of the Global-E allreduce with re-rounding at every hop, through the C ABI.

gq_exp_combine against the oracle's step (bit-exact codes), and gq_exp_allreduce (tree and
ring) on gq_quantize's code matrix against the oracle's tree / ring on the oracle's codes
(bit-exact reduced codes; dequantised mean within 1e-6 * N).
"""
import numpy as np
import pytest

from gpu_common import EXP, gq_module, to_device
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    return gq_module()


@pytest.fixture(scope="module")
def oracle_mod():
    from oracle import gq_oracle
    gq_oracle.lib()
    return gq_oracle


@pytest.mark.parametrize("d", [1, 15, 16, 17, 1003, 65541])
def test_combine_matches_oracle(gq, oracle_mod, d):
    import torch
    rng = np.random.default_rng(d)
    a = rng.integers(-20, 21, d).astype(np.int8)
    b = rng.integers(-20, 21, d).astype(np.int8)
    a[: d // 3] = 0
    for sid in (oracle_mod.exp_tree_stream(1, 0), oracle_mod.exp_tree_stream(4, 7),
                oracle_mod.exp_ring_stream(3, 2)):
        got = gq.gq_exp_combine(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(),
                                0xABCDEF0123, 17, sid).cpu().numpy()
        np.testing.assert_array_equal(got, oracle_mod.exp_combine(a, b, 0xABCDEF0123, 17, sid))


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("s", [4, 8])
@pytest.mark.parametrize("n,d", [(1, 100), (2, 1001), (3, 4099), (5, 333), (8, 20000), (16, 777)])
def test_allreduce_matches_oracle(gq, oracle_mod, order, s, n, d):
    import torch
    x = workloads.host_inputs("normal", n, d, seed=n + d)
    norm32 = np.float32(oracle_mod.global_norm(x, 2, 2))
    ocodes, rc = oracle_mod.quantize(x, norm32, EXP, s, 21, 3)
    if order == 0:
        root = oracle_mod.exp_tree_allreduce(ocodes, 21, 3)
    else:
        root = oracle_mod.exp_ring_allreduce(ocodes, d, 21, 3)
    units = oracle_mod.exp_units(root).astype(np.float64)
    want = float(norm32) * units * 2.0 ** -(s - 1) / n
    norm = torch.tensor([float(norm32)], device="cuda")
    codes = gq.gq_quantize(to_device(x), norm, EXP, s, 21, 3)
    root_g = torch.empty(d, dtype=torch.int8, device="cuda")
    out = gq.gq_exp_allreduce(codes, s, n, d, order, norm, 21, 3, root_codes=root_g)
    np.testing.assert_array_equal(root_g.cpu().numpy(), root)
    assert np.abs(out.cpu().numpy().astype(np.float64) - want).max() <= 1e-6 * float(norm32)


def test_allreduce_argument_checks(gq):
    import torch
    codes = torch.zeros(65 * 32, dtype=torch.uint8, device="cuda")
    norm = torch.ones(1, device="cuda")
    with pytest.raises(gq.GQError) as e:
        gq.gq_exp_allreduce(codes, 4, 65, 32, 0, norm, 1, 1)   # more workers than the kernel holds
    assert e.value.status == 1
    with pytest.raises(gq.GQError) as e:
        gq.gq_exp_allreduce(codes, 4, 4, 32, 2, norm, 1, 1)    # no such order
    assert e.value.status == 1
    with pytest.raises(gq.GQError) as e:
        gq.gq_exp_allreduce(codes, 25, 4, 32, 0, norm, 1, 1)   # s beyond Global-E's range
    assert e.value.status == 2
