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


@pytest.mark.parametrize("lim", [24, 25, 30, 31, 62])
def test_combine_code_ranges(gq, oracle_mod, lim):
    """The three arithmetic paths of the combine kernel: codes up to |k| = 24 through the table of
    splits, up to 30 in 32 bits, larger (extended codes of earlier hops) in 64 bits; a thread's 16
    coordinates take the table only if all of them fit, so groups of each kind sit side by side."""
    import torch
    d = 70_003
    rng = np.random.default_rng(lim)
    a = rng.integers(-12, 13, d).astype(np.int8)
    b = rng.integers(-12, 13, d).astype(np.int8)
    big = rng.random(d) < 0.02  # about a quarter of the 16-coordinate groups hold a large code
    a[big] = rng.integers(-lim, lim + 1, int(big.sum())).astype(np.int8)
    b[: 64] = lim  # the largest magnitude at both signs in the first groups
    b[64: 128] = -lim
    sid = oracle_mod.exp_ring_stream(2, 5)
    got = gq.gq_exp_combine(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), 77, 3,
                            sid).cpu().numpy()
    np.testing.assert_array_equal(got, oracle_mod.exp_combine(a, b, 77, 3, sid))


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


@pytest.mark.parametrize("j0", [0, 16, 4096, 812_512])
def test_combine_with_column_base(gq, oracle_mod, j0):
    """gq_exp_combine on a window whose first element is coordinate j0 of the whole vector (a ring
    chunk): the random words are those of the global coordinates."""
    import torch
    rng = np.random.default_rng(j0 + 1)
    d = 1000 + j0 % 37
    a = rng.integers(-12, 13, d).astype(np.int8)
    b = rng.integers(-12, 13, d).astype(np.int8)
    sid = gq.gq_exp_ring_stream(3, 2)
    got = gq.gq_exp_combine(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), 5, 6, sid,
                            j0=j0).cpu().numpy()
    np.testing.assert_array_equal(got, oracle_mod.exp_combine(a, b, 5, 6, sid, j0=j0))


def test_combine_rejects_unaligned_base(gq):
    import torch
    a = torch.zeros(64, dtype=torch.int8, device="cuda")
    with pytest.raises(gq.GQError):
        gq.gq_exp_combine(a, a, 1, 1, 0, j0=4)


@pytest.mark.parametrize("s", [4, 8])
@pytest.mark.parametrize("out16", [False, True])
def test_exp_dequantize_matches_oracle(gq, oracle_mod, s, out16):
    import torch
    rng = np.random.default_rng(s)
    d, n = 4099, 5
    codes = rng.integers(-20, 21, d).astype(np.int8)  # extended codes, as a reduction leaves them
    norm = torch.tensor([3.25], device="cuda")
    odt = torch.bfloat16 if out16 else torch.float32
    got = gq.gq_exp_dequantize(torch.from_numpy(codes).cuda(), norm, s, n, out_dtype=odt)
    want, rc = oracle_mod.dequantize(oracle_mod.exp_units(codes), 3.25, 1, s, n)
    assert rc == 0
    g = got.float().cpu().numpy().astype(np.float64)
    # out = fp32(scale) * 2^m exactly: relative error of the rounded scale only (plus bf16)
    tol = np.abs(want) * (2.0 ** -23 + (2.0 ** -8 if out16 else 0.0))
    assert np.all(np.abs(g - want) <= tol)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("s,bits", [(4, 4), (4, 8), (8, 8)])
def test_quantize_codes_with_worker_offset(gq, oracle_mod, dtype, s, bits):
    """One rank's codes (rows worker0 ..) as int8 or int4, equal to the oracle's rows of the
    stacked matrix."""
    import torch
    from allreduce_compatible_gradient_gb300 import workloads
    from gpu_common import unpack_codes
    n, d = 5, 1003
    x = workloads.host_inputs("normal", n, d, seed=4, dtype=dtype)
    norm32 = float(np.float32(oracle_mod.global_norm(x, 0, 0)))
    want, rc = oracle_mod.quantize(x, norm32, 1, s, 9, 3)
    assert rc == 0
    xd = __import__("gpu_common").to_device(x)
    norm = torch.tensor([norm32], device="cuda")
    for r0, m in [(0, 2), (2, 3)]:
        got = gq.gq_quantize_codes(xd[r0:r0 + m].clone(), norm, gq.EXP, s, 9, 3, worker0=r0,
                                   code_bits=bits).cpu().numpy()
        if bits == 8:
            pitch = gq.gq_code_pitch(d)
            rows = got.view(np.int8).reshape(m, pitch)[:, :d]
        else:
            rows = unpack_codes(got, gq.EXP, s, m, d)
        np.testing.assert_array_equal(rows, want[r0:r0 + m])
