"""GPU parity of the 16-bit outputs (bf16, fp16) of the dequantised mean.

The 16-bit output is defined as the fp32 output rounded to nearest even, so it is checked
  * bit for bit against the fp32 output of the same call converted on the host (torch's CPU
    conversion, round to nearest even), for the fused call, the unfused dequantisation and the
    segmented form, on ragged shapes;
  * against the oracle's fp64 mean: |out16 - exact| <= 1e-6 N + half a 16-bit ulp of the value;
  * fp16 past 65504 becomes infinite (IEEE rounding), bf16 keeps the fp32 range.
"""
import numpy as np
import pytest

from gpu_common import EXP, INF, LINEAR, gq_module, to_device, to_host
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1), (3, 17), (5, 1000), (8, 4099), (3, 65536 + 24)]


@pytest.fixture(scope="module")
def gq():
    return gq_module()


@pytest.fixture(scope="module")
def oracle_mod():
    from oracle import gq_oracle
    gq_oracle.lib()
    return gq_oracle


def _t16(name):
    import torch
    return {"bf16": torch.bfloat16, "f16": torch.float16}[name]


def _half_ulp(name, v):
    """Half a unit in the last place of the 16-bit format at |v| (normal range), or of its
    smallest subnormal step."""
    mant, emin = (8, -126) if name == "bf16" else (11, -14)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** emin)))
    return 2.0 ** (e - mant)


@pytest.mark.parametrize("out16", ["bf16", "f16"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,d", SHAPES)
@pytest.mark.parametrize("scheme,s", [(LINEAR, 7), (LINEAR, 127), (EXP, 8)])
def test_fused_out16(gq, oracle_mod, out16, dtype, n, d, scheme, s):
    import torch
    x = workloads.host_inputs("normal", n, d, seed=n + d, dtype=dtype)
    xd = to_device(x)
    seed, step = 3, 17
    o32 = gq.gq_allreduce_mean(xd, INF, INF, scheme, s, seed, step)
    o16 = gq.gq_allreduce_mean(xd, INF, INF, scheme, s, seed, step, out_dtype=_t16(out16))
    torch.cuda.synchronize()
    assert o16.dtype == _t16(out16)
    assert torch.equal(o16.cpu(), o32.cpu().to(_t16(out16)))
    res = oracle_mod.allreduce_mean(x, INF, INF, scheme, s, seed, step)
    assert res["rc"] == 0
    want = res["out"]
    got = o16.cpu().float().numpy().astype(np.float64)
    tol = 1e-6 * res["norm32"] + _half_ulp(out16, want) * (1 + 1e-6)
    assert np.all(np.abs(got - want) <= tol)


@pytest.mark.parametrize("out16", ["bf16", "f16"])
@pytest.mark.parametrize("scheme,s", [(LINEAR, 15), (EXP, 4)])
def test_dequantize_out16(gq, out16, scheme, s):
    import torch
    n, d = 6, 4099
    x = to_device(workloads.host_inputs("normal", n, d, seed=9))
    norm = gq.gq_global_norm(x, INF, INF)
    codes = gq.gq_quantize(x, norm, scheme, s, 1, 2)
    sums = gq.gq_reduce_codes(codes, scheme, s, n, d)
    o32 = gq.gq_dequantize(sums, norm, scheme, s, n)
    o16 = gq.gq_dequantize(sums, norm, scheme, s, n, out_dtype=_t16(out16))
    torch.cuda.synchronize()
    assert torch.equal(o16.cpu(), o32.cpu().to(_t16(out16)))


@pytest.mark.parametrize("out16", ["bf16", "f16"])
def test_segments_out16(gq, out16):
    import torch
    sizes = [1, 3, 17, 4099, 1000, 65536 + 24, 8, 2053]
    segs = workloads.segment_tensors(5, sizes, seed=2)
    o32 = gq.gq_allreduce_mean_segments(segs, 2, 2, EXP, 8, 4, 5)
    o16 = gq.gq_allreduce_mean_segments(segs, 2, 2, EXP, 8, 4, 5, out_dtype=_t16(out16))
    torch.cuda.synchronize()
    for a, b in zip(o32, o16):
        assert torch.equal(b.cpu(), a.cpu().to(_t16(out16)))


def test_f16_overflow_is_infinite(gq):
    import torch
    x = torch.tensor([[1e5, -3e4, 70000.0, 1.0]], device="cuda")
    o32 = gq.gq_allreduce_mean(x, INF, INF, LINEAR, 127, 0, 0)
    o16 = gq.gq_allreduce_mean(x, INF, INF, LINEAR, 127, 0, 0, out_dtype=torch.float16)
    ob = gq.gq_allreduce_mean(x, INF, INF, LINEAR, 127, 0, 0, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(o16.cpu(), o32.cpu().to(torch.float16))
    assert torch.isinf(o16[0]).item() and torch.isinf(o16[2]).item()
    assert torch.isfinite(ob).all().item()


def test_out_type_errors(gq):
    import torch
    x = torch.ones(2, 8, device="cuda")
    with pytest.raises(TypeError):
        gq.gq_allreduce_mean(x, INF, INF, EXP, 8, 0, 0, out_dtype=torch.float64)
    sums = torch.zeros(8, dtype=torch.int32, device="cuda")
    norm = torch.ones(1, device="cuda")
    out = torch.empty(8, device="cuda")
    rc = gq.lib().gq_dequantize_to(sums.data_ptr(), norm.data_ptr(), EXP, 8, 2, 8, out.data_ptr(),
                                   7, None)
    assert rc == 1  # GQ_ERR_INVALID: no such output type
