"""GPU parity of the 16-bit-uniform rounding mode (scheme | GQ_ROUND_U16) against the oracle's mode
(gqo_quantize_u16_cols), through every quantise kernel: codes bit for bit, integer sums read back
from the mean bit for bit, the mean within 1e-6 N.

Inputs put thousands of decisions on the mode's own boundary: under a max norm of 1 (an anchor
element |x| = 1) the fraction F is set exactly to H - 1, H (a tie, which stays down) or H + 1 for
the element's high half H (Global-E: |x| = 2^e (1 + F 2^-16) or F 2^-16 2^-(s-1); Global-L with
s a power of two: |x| = (m + F 2^-16) / s), on random levels.  The kernels decide these with the
16.16 estimate alone (no exact path), so they must compute exactly the mode's F.
"""
import numpy as np
import pytest

import boundary_inputs as bi
from gpu_common import EXP, INF, LINEAR, gq_module, to_device, unpack_codes

pytestmark = pytest.mark.gpu

U16 = 16
SEED, STEP = 7, 9


@pytest.fixture(scope="module")
def gq():
    return gq_module()


def u16_matrix(n, d, scheme, s, rng, dtype="f32", step=STEP, count=3000):
    """Max norm 1 (anchor), background noise below it, `count` elements with F = H - 1, H, H + 1."""
    x = bi.background(n, d, rng, 0.2, dtype)
    np.clip(x, -1.0, 1.0, out=x)
    R = bi.words(n, d, SEED, step)
    pos = rng.choice(n * d, size=count, replace=False)
    for p in pos[1:]:
        i, j = divmod(int(p), d)
        H = int(R[i, j]) >> 16
        F = min(0xFFFF, max(0, H + int(rng.integers(-1, 2))))
        if scheme == EXP:
            m = int(rng.integers(0, s))
            v = (F / 2.0**16) * 2.0 ** -(s - 1) if m == 0 else 2.0 ** (m - s) * (1 + F / 2.0**16)
        else:
            m = int(rng.integers(0, s))
            v = (m + F / 2.0**16) / s
        x[i, j] = np.float32(v) * (1.0 if rng.random() < 0.5 else -1.0)
    x.ravel()[int(pos[0])] = 1.0
    if dtype == "bf16":  # exactly representable only where F has few bits; still a valid input
        x = (bi._bf16_bits(x.ravel()).astype(np.uint32) << 16).view(np.float32).reshape(n, d)
        x.ravel()[int(pos[0])] = 1.0
    return bi.to_dtype(x, dtype)


def _sums(out, N32, scheme, s, n):
    sc = float(np.float32(float(N32) / (n * s))) if scheme == LINEAR else float(
        np.float32(np.ldexp(float(N32), -(s - 1)) / n))
    return np.rint(out.astype(np.float64) / sc).astype(np.int64)


def _check(oracle, xh, N32, scheme, s, out, codes_u8=None, step=STEP, worker0=0):
    n, d = xh.shape
    if worker0:
        full = np.ascontiguousarray(np.concatenate([np.zeros((worker0, d), xh.dtype), xh]))
        ref_codes, rc = oracle.quantize_u16(full, N32, scheme, s, SEED, step)
        ref_codes = ref_codes[worker0:]
    else:
        ref_codes, rc = oracle.quantize_u16(xh, N32, scheme, s, SEED, step)
    assert rc == 0
    sums = oracle.reduce_codes(ref_codes, scheme, s)
    if out is not None:
        ref_out, _ = oracle.dequantize(sums, N32, scheme, s, n)
        got = out.cpu().numpy()
        np.testing.assert_array_equal(_sums(got, N32, scheme, s, n), sums)
        assert np.abs(got.astype(np.float64) - ref_out).max() <= 1e-6 * float(N32)
    if codes_u8 is not None:
        got = unpack_codes(codes_u8.cpu().numpy(), scheme, s, n, d)
        bad = np.argwhere(got != ref_codes)
        assert len(bad) == 0, "%d codes differ, first %s" % (len(bad), bad[:4].tolist())
    return ref_codes, sums


SCHEMES = [(LINEAR, 4), (LINEAR, 64), (EXP, 8), (EXP, 4)]


@pytest.mark.parametrize("n,d,dtype", [(8, 1 << 20, "f32"), (8, 1 << 21, "bf16"),
                                       (5, (1 << 18) + 3, "f32"), (4, 65_536, "f32")])
@pytest.mark.parametrize("scheme,s", SCHEMES)
def test_fused(gq, oracle, n, d, dtype, scheme, s):
    """Bulk-copy kernel (large aligned), direct loads (ragged), single launch (small)."""
    import torch
    rng = np.random.default_rng(d + s + scheme)
    xh = u16_matrix(n, d, scheme, s, rng, dtype)
    x = to_device(xh)
    ws = gq.gq_workspace()
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    out = gq.gq_allreduce_mean(x, INF, INF, scheme | U16, s, SEED, STEP, norm=norm, ws=ws)
    codes = torch.empty(gq.gq_code_bytes(scheme, s, n, d), dtype=torch.uint8, device="cuda")
    out2 = gq.gq_allreduce_mean(x, INF, INF, scheme | U16, s, SEED, STEP, codes=codes, ws=ws)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    N32 = np.float32(norm.item())
    assert N32 == np.float32(1.0)
    _check(oracle, xh, N32, scheme, s, out)
    _check(oracle, xh, N32, scheme, s, out2, codes)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scheme,s", [(EXP, 8), (LINEAR, 7)])
def test_compacting_consumer(gq, oracle, dtype, scheme, s):
    """The (2, 2) norm: the compacting consumer's light test uses the mode's own bound (H >= F
    for every element of a row-group)."""
    import torch
    from allreduce_compatible_gradient_gb300 import workloads
    from gpu_common import to_host
    n, d = 8, (1 << 20) if dtype == "f32" else (1 << 21)
    x = workloads.device_inputs("student_t3", n, d, seed=5, dtype=dtype)
    ws = gq.gq_workspace()
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    out = gq.gq_allreduce_mean(x, 2, 2, scheme | U16, s, SEED, STEP, norm=norm, ws=ws)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    xh = to_host(x)
    N32 = np.float32(norm.item())
    assert float(N32) == pytest.approx(oracle.global_norm(xh, 2, 2), rel=1e-6)
    _check(oracle, xh, N32, scheme, s, out)


@pytest.mark.parametrize("scheme,s", [(LINEAR, 4), (EXP, 8)])
def test_supplied_norm_and_codes(gq, oracle, scheme, s):
    """gq_allreduce_mean_with_norm and gq_quantize (direct loads, untrusted norm: |x| above N
    saturates, NaN gives 0) and the exact mode for a norm outside [2^-100, 2^100]."""
    import torch
    n, d = 4, 100_003
    rng = np.random.default_rng(s)
    xh = u16_matrix(n, d, scheme, s, rng)
    xh[0, :5] = [2.0, -3.0, np.nan, 1.0, -1.0]
    x = to_device(xh)
    for N in (1.0, 0.8, 2.0**-110):
        norm = torch.tensor([N], dtype=torch.float32, device="cuda")
        out = gq.gq_allreduce_mean_with_norm(x, norm, scheme | U16, s, SEED, STEP)
        codes = gq.gq_quantize(x, norm, scheme | U16, s, SEED, STEP)
        torch.cuda.synchronize()
        _check(oracle, xh, np.float32(N), scheme, s, out, codes)


def test_segments_and_rank_shares(gq, oracle):
    import torch
    scheme, s = EXP, 4
    sizes = [400_000, 1003, 263_168, 65_536]
    hosts = [u16_matrix(4, sz, scheme, s, np.random.default_rng(sz), step=(STEP << 16) | l)
             for l, sz in enumerate(sizes)]
    xs = [to_device(h) for h in hosts]
    ws = gq.gq_workspace()
    norms = torch.empty(len(sizes), dtype=torch.float32, device="cuda")
    outs = gq.gq_allreduce_mean_segments(xs, INF, INF, scheme | U16, s, SEED, STEP, norms=norms,
                                         ws=ws)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    for l, (h, o) in enumerate(zip(hosts, outs)):
        _check(oracle, h, np.float32(norms[l].item()), scheme, s, o, step=(STEP << 16) | l)
    # one rank's rows 3 .. 4 of a stacked matrix: sums and codes with a worker offset
    h = u16_matrix(2, 1 << 20, LINEAR, 4, np.random.default_rng(2))
    x = to_device(h)
    norm = torch.tensor([1.0], dtype=torch.float32, device="cuda")
    sums = gq.gq_quantize_sum(x, norm, LINEAR | U16, 4, SEED, STEP, worker0=3, ws=ws)
    codes = gq.gq_quantize_codes(x, norm, LINEAR | U16, 4, SEED, STEP, worker0=3, ws=ws)
    torch.cuda.synchronize()
    ref_codes, ref_sums = _check(oracle, h, np.float32(1.0), LINEAR, 4, None, worker0=3)
    np.testing.assert_array_equal(sums.cpu().numpy().astype(np.int64), ref_sums)
    np.testing.assert_array_equal(unpack_codes(codes.cpu().numpy(), EXP, 8, 2, 1 << 20), ref_codes)
