"""GPU parity: every step of the CUDA path against the CPU oracle, through the C ABI.

Bars (from the method's definitions and the library's documented precision):
  * codes and integer sums: bit-exact whenever both sides use the same fp32 norm (always for the
    max norm; for the l2 forms the oracle's norm is fed to the GPU);
  * l2 norms: relative 1e-6 of the oracle's fp64 norm; the max norm exactly;
  * dequantised mean: |out - oracle| <= 1e-6 * N.
Shapes span several 256-thread blocks and ragged tails (d not a multiple of 4, 8 or 32).
"""
import numpy as np
import pytest

from gpu_common import EXP, INF, LINEAR, gq_module, to_device, to_host, unpack_codes
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu

ORDERS = [(2, 2), (2, INF), (INF, 2), (INF, INF)]
SHAPES = [(1, 1), (2, 3), (3, 17), (4, 67), (5, 1000), (8, 4099), (3, 65536 + 24), (16, 2053)]
SCHEMES = [(LINEAR, 1), (LINEAR, 7), (LINEAR, 15), (LINEAR, 127), (EXP, 1), (EXP, 4), (EXP, 8),
           (EXP, 24)]


@pytest.fixture(scope="module")
def gq():
    return gq_module()


@pytest.fixture(scope="module")
def oracle_mod():
    from oracle import gq_oracle
    gq_oracle.lib()
    return gq_oracle


def _inputs(n, d, dtype, seed):
    dist = "student_t3" if dtype == "bf16" else "normal"
    return workloads.host_inputs(dist, n, d, seed=seed, dtype=dtype)


def _norm_tol(q, p):
    return 0.0 if (q, p) == (INF, INF) else 1e-6


# ---------------------------------------------------------------------------------------------
# Philox: library device stream == oracle
# ---------------------------------------------------------------------------------------------

def test_philox_matches_oracle(gq, oracle_mod):
    import torch
    rng = np.random.default_rng(1)
    ck = rng.integers(0, 2**32, size=(4096, 6), dtype=np.uint64).astype(np.uint32)
    ck[0] = 0
    ck[1] = 0xFFFFFFFF
    out = gq.gq_philox4x32_10(torch.from_numpy(ck.view(np.int32)).cuda())
    got = out.cpu().numpy().view(np.uint32)
    for t in range(ck.shape[0]):
        np.testing.assert_array_equal(got[t], oracle_mod.philox4x32_10(ck[t, :4], ck[t, 4:]))


# ---------------------------------------------------------------------------------------------
# Step 1: norm
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,d", SHAPES)
@pytest.mark.parametrize("q,p", ORDERS)
def test_norm(gq, oracle_mod, dtype, n, d, q, p):
    x = _inputs(n, d, dtype, seed=n * 1000 + d)
    want = oracle_mod.global_norm(x, q, p)
    got = float(gq.gq_global_norm(to_device(x), q, p).item())
    if (q, p) == (INF, INF):
        assert got == float(np.float32(want))
    else:
        assert got == pytest.approx(want, rel=1e-6)


@pytest.mark.parametrize("scale", [1e-30, 1e-20, 1e20, 1e30, 3e38])
@pytest.mark.parametrize("q,p", ORDERS)
def test_norm_extreme_magnitudes(gq, oracle_mod, scale, q, p):
    # squares of these values leave the fp32 range: the scaled sums must still be accurate
    x = (workloads.host_inputs("normal", 3, 999, seed=5) * np.float32(scale / 4)).astype(np.float32)
    want = oracle_mod.global_norm(x, q, p)
    got = float(gq.gq_global_norm(to_device(x), q, p).item())
    if not np.isfinite(np.float32(want)):
        assert not np.isfinite(got)
    else:
        assert got == pytest.approx(want, rel=1e-6)


@pytest.mark.parametrize("q,p", ORDERS)
def test_norm_subnormal_and_mixed(gq, oracle_mod, q, p):
    rng = np.random.default_rng(3)
    x = np.zeros((4, 333), dtype=np.float32)
    x[:, ::3] = (rng.standard_normal((4, 111)) * 1e-40).astype(np.float32)   # subnormal
    x[1, 7] = 1e-38
    want = oracle_mod.global_norm(x, q, p)
    got = float(gq.gq_global_norm(to_device(x), q, p).item())
    assert got == pytest.approx(want, rel=1e-6)
    x[2, 100] = 1e25   # huge next to subnormals
    want = oracle_mod.global_norm(x, q, p)
    got = float(gq.gq_global_norm(to_device(x), q, p).item())
    assert got == pytest.approx(want, rel=1e-6)


def test_norm_zero_and_nonfinite(gq):
    import torch
    ws = gq.gq_workspace()
    for q, p in ORDERS:
        z = torch.zeros((3, 77), device="cuda")
        assert float(gq.gq_global_norm(z, q, p, ws=ws).item()) == 0.0
        assert gq.gq_get_status(ws) == 0
        for bad in (float("nan"), float("inf"), float("-inf")):
            x = torch.randn((3, 77), device="cuda")
            x[1, 40] = bad
            nrm = float(gq.gq_global_norm(x, q, p, ws=ws).item())
            assert not np.isfinite(nrm)
            assert gq.gq_get_status(ws) == 4          # GQ_ERR_NONFINITE, then cleared
            assert gq.gq_get_status(ws) == 0


# ---------------------------------------------------------------------------------------------
# Steps 2-4 unfused, with the oracle's fp32 norm fed to the GPU
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,d", SHAPES)
@pytest.mark.parametrize("scheme,s", SCHEMES)
def test_quantize_reduce_dequantize(gq, oracle_mod, dtype, n, d, scheme, s):
    import torch
    if scheme == EXP and n * 2 ** (s - 1) >= 2**24:
        pytest.skip("sum range")
    x = _inputs(n, d, dtype, seed=7 * n + d + s)
    q, p = ORDERS[(n + d + s) % 4]
    ref = oracle_mod.allreduce_mean(x, q, p, scheme, s, 0xDEADBEEF12345678, 99)
    norm = torch.tensor([ref["norm32"]], dtype=torch.float32, device="cuda")
    xg = to_device(x)
    codes = gq.gq_quantize(xg, norm, scheme, s, 0xDEADBEEF12345678, 99)
    got = unpack_codes(codes.cpu().numpy(), scheme, s, n, d)
    np.testing.assert_array_equal(got, ref["codes"])
    sums = gq.gq_reduce_codes(codes, scheme, s, n, d)
    np.testing.assert_array_equal(sums.cpu().numpy().astype(np.int64), ref["sums"])
    out = gq.gq_dequantize(sums, norm, scheme, s, n).cpu().numpy().astype(np.float64)
    assert np.abs(out - ref["out"]).max() <= 1e-6 * float(ref["norm32"])


# ---------------------------------------------------------------------------------------------
# Fused path
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,d", SHAPES)
@pytest.mark.parametrize("scheme,s", [(LINEAR, 15), (LINEAR, 127), (EXP, 4), (EXP, 8)])
def test_fused_max_norm_bit_exact(gq, oracle_mod, dtype, n, d, scheme, s):
    import torch
    x = _inputs(n, d, dtype, seed=11 * n + d)
    ref = oracle_mod.allreduce_mean(x, INF, INF, scheme, s, 7, 3)
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    codes = torch.empty(gq.gq_code_bytes(scheme, s, n, d), dtype=torch.uint8, device="cuda")
    out = gq.gq_allreduce_mean(to_device(x), INF, INF, scheme, s, 7, 3, norm=norm, codes=codes)
    assert float(norm.item()) == float(ref["norm32"])
    np.testing.assert_array_equal(unpack_codes(codes.cpu().numpy(), scheme, s, n, d), ref["codes"])
    got = out.cpu().numpy().astype(np.float64)
    assert np.abs(got - ref["out"]).max() <= 1e-6 * float(ref["norm32"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("q,p", ORDERS)
@pytest.mark.parametrize("scheme,s", [(LINEAR, 7), (EXP, 8)])
def test_fused_with_oracle_norm(gq, oracle_mod, dtype, q, p, scheme, s):
    import torch
    n, d = 6, 5001
    x = _inputs(n, d, dtype, seed=17)
    ref = oracle_mod.allreduce_mean(x, q, p, scheme, s, 5, 6)
    norm = torch.tensor([ref["norm32"]], dtype=torch.float32, device="cuda")
    codes = torch.empty(gq.gq_code_bytes(scheme, s, n, d), dtype=torch.uint8, device="cuda")
    out = gq.gq_allreduce_mean_with_norm(to_device(x), norm, scheme, s, 5, 6, codes=codes)
    np.testing.assert_array_equal(unpack_codes(codes.cpu().numpy(), scheme, s, n, d), ref["codes"])
    got = out.cpu().numpy().astype(np.float64)
    assert np.abs(got - ref["out"]).max() <= 1e-6 * float(ref["norm32"])


@pytest.mark.parametrize("q,p", ORDERS)
def test_fused_equals_unfused(gq, q, p):
    import torch
    n, d = 5, 12347
    x = to_device(_inputs(n, d, "f32", seed=23))
    for scheme, s in [(LINEAR, 5), (EXP, 6), (LINEAR, 100), (EXP, 12)]:
        norm_f = torch.empty(1, dtype=torch.float32, device="cuda")
        codes_f = torch.empty(gq.gq_code_bytes(scheme, s, n, d), dtype=torch.uint8, device="cuda")
        out_f = gq.gq_allreduce_mean(x, q, p, scheme, s, 9, 10, norm=norm_f, codes=codes_f)
        norm_u = gq.gq_global_norm(x, q, p)
        codes_u = gq.gq_quantize(x, norm_u, scheme, s, 9, 10)
        out_u = gq.gq_dequantize(gq.gq_reduce_codes(codes_u, scheme, s, n, d), norm_u, scheme, s, n)
        assert torch.equal(norm_f, norm_u)
        assert torch.equal(codes_f, codes_u)
        assert torch.equal(out_f, out_u)
        out_nc = gq.gq_allreduce_mean(x, q, p, scheme, s, 9, 10)   # no codes, no norm out
        assert torch.equal(out_nc, out_u)


def test_deterministic(gq):
    import torch
    x = to_device(_inputs(8, 100003, "f32", seed=1))
    for q, p in ORDERS:
        a = gq.gq_allreduce_mean(x, q, p, EXP, 8, 1, 2)
        b = gq.gq_allreduce_mean(x, q, p, EXP, 8, 1, 2)
        assert torch.equal(a, b)
        na, nb = gq.gq_global_norm(x, q, p), gq.gq_global_norm(x, q, p)
        assert torch.equal(na, nb)


def test_zero_and_nonfinite_inputs(gq):
    import torch
    n, d = 3, 1001
    ws = gq.gq_workspace()
    for scheme, s in [(LINEAR, 7), (EXP, 4), (LINEAR, 20)]:
        codes = torch.full((gq.gq_code_bytes(scheme, s, n, d),), 0x55, dtype=torch.uint8,
                           device="cuda")
        out = torch.full((d,), 3.0, device="cuda")
        gq.gq_allreduce_mean(torch.zeros((n, d), device="cuda"), 2, 2, scheme, s, 1, 1, out=out,
                             codes=codes, ws=ws)
        assert not out.any() and not codes.any()
        assert gq.gq_get_status(ws) == 0
        x = torch.randn((n, d), device="cuda")
        x[2, 500] = float("nan")
        codes.fill_(0x55)
        out.fill_(3.0)
        gq.gq_allreduce_mean(x, INF, INF, scheme, s, 1, 1, out=out, codes=codes, ws=ws)
        assert not out.any() and not codes.any()
        assert gq.gq_get_status(ws) == 4


def test_saturation_and_nan_under_supplied_norm(gq, oracle_mod):
    import torch
    x = np.array([[np.nan, 1.0, np.inf, -2.0, 0.5, -0.0, 3.0, 1e-45]], dtype=np.float32)
    for scheme, s in [(LINEAR, 5), (EXP, 5)]:
        want, rc = oracle_mod.quantize(x, np.float32(2.0), scheme, s, 1, 1)
        norm = torch.tensor([2.0], device="cuda")
        codes = gq.gq_quantize(to_device(x), norm, scheme, s, 1, 1)
        np.testing.assert_array_equal(unpack_codes(codes.cpu().numpy(), scheme, s, 1, 8), want)


def test_argument_errors(gq):
    import torch
    x = torch.randn((4, 64), device="cuda")
    norm = torch.ones(1, device="cuda")
    with pytest.raises(gq.GQError) as e:
        gq.gq_quantize(x, norm, LINEAR, 128, 1, 1)
    assert e.value.status == 2
    with pytest.raises(gq.GQError) as e:
        gq.gq_quantize(x, norm, EXP, 25, 1, 1)
    assert e.value.status == 2
    with pytest.raises(gq.GQError) as e:
        gq.gq_quantize(torch.randn((163840, 1), device="cuda"), norm, LINEAR, 127, 1, 1)  # n s >= 2^24
    assert e.value.status == 3
    with pytest.raises(gq.GQError) as e:
        gq.gq_quantize(torch.randn((4, 8), device="cuda"), norm, EXP, 23, 1, 1)  # 4 * 2^22 = 2^24
    assert e.value.status == 3
    with pytest.raises(gq.GQError) as e:
        gq.gq_global_norm(x, 1, 2)
    assert e.value.status == 1
    ws_small = torch.zeros(100, dtype=torch.uint8, device="cuda")
    with pytest.raises(gq.GQError) as e:
        gq.gq_global_norm(x, 2, 2, ws=ws_small)
    assert e.value.status == 7
    xm = torch.randn(4 * 64 + 1, device="cuda")[1:].view(4, 64)   # 4-byte offset: misaligned
    with pytest.raises(gq.GQError) as e:
        gq.gq_global_norm(xm, 2, 2)
    assert e.value.status == 1
