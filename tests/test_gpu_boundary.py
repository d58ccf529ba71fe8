"""GPU parity on inputs that put the rounding decision on its boundary, through every quantise
kernel (tests/boundary_inputs.py builds them on the CPU from the oracle alone).

Round up iff r < T (Global-Q operator: unbiased rounding between adjacent levels; this project's
random word r and threshold T = floor(P(up) 2^32)).  The kernels decide most elements from a
16.16 fixed-point estimate and the high half of r, and take the exact path (correctly rounded
quotient, full word) when the estimate is within the certainty window.  Here thousands of
elements per matrix have T - r = 0 (a tie, which stays down), +-1, or near +-1..4 x 2^16 (the
window's edges), on random levels; the Global-L_127 case also holds elements whose estimate is
more than one unit low (the window's margin).  Every kernel's codes must equal the oracle's bit
for bit, its code sums (read back exactly from the dequantised mean) too, and its mean within
1e-6 N:
  * the fused call, two passes, bulk-copy quantise kernel (fp32 and bf16; max norm; and the
    (2, 2) norm under Global-E, which takes the compacting consumer), with and without codes;
  * the fused call on unaligned rows (direct-load kernel);
  * the single launch (matrix held in shared memory);
  * a supplied norm (gq_allreduce_mean_with_norm, gq_quantize): also |x| equal to and above N;
  * the segmented form (bulk-copy ring over segments, and the direct-load segment kernel);
  * one rank's sums and codes with a worker offset (bulk-copy one-row and two-row forms, and the
    direct-load kernel without a workspace).
"""
import numpy as np
import pytest

import boundary_inputs as bi
from gpu_common import EXP, INF, LINEAR, gq_module, to_device, unpack_codes

pytestmark = pytest.mark.gpu

SEED, STEP = 3, 5
WORST_N = 0.48058903


@pytest.fixture(scope="module")
def gq():
    return gq_module()


def _scale(N32: float, scheme: int, s: int, n: int) -> float:
    """The fp32 dequantisation scale, as the library states it (computed in fp64)."""
    if scheme == LINEAR:
        return float(np.float32(float(N32) / (n * s)))
    return float(np.float32(np.ldexp(float(N32), -(s - 1)) / n))


def _sums_from_out(out: np.ndarray, N32: float, scheme: int, s: int, n: int) -> np.ndarray:
    """Integer sums S from out = fp32(scale S): exact while |S| < 2^23."""
    sc = _scale(N32, scheme, s, n)
    if sc == 0.0:
        return np.zeros(out.shape, dtype=np.int64)
    return np.rint(out.astype(np.float64) / sc).astype(np.int64)


def _oracle(oracle, xh, N32, scheme, s, worker0=0, step=STEP):
    """Codes (rows worker0 ..), sums and mean of the oracle for the rows of xh."""
    if worker0:
        pad = np.zeros((worker0, xh.shape[1]), dtype=xh.dtype)
        full = np.ascontiguousarray(np.concatenate([pad, xh]))
        codes, rc = oracle.quantize(full, N32, scheme, s, SEED, step)
        codes = codes[worker0:]
    else:
        codes, rc = oracle.quantize(xh, N32, scheme, s, SEED, step)
    assert rc == 0
    sums = oracle.reduce_codes(codes, scheme, s)
    out, rc = oracle.dequantize(sums, N32, scheme, s, xh.shape[0])
    return codes, sums, out


def _compare_out(out_gpu, N32, scheme, s, n, sums, ref_out):
    got = out_gpu.cpu().numpy()
    np.testing.assert_array_equal(_sums_from_out(got, N32, scheme, s, n), sums)
    assert np.abs(got.astype(np.float64) - ref_out).max() <= 1e-6 * float(N32)


def _compare_codes(codes_gpu, scheme, s, n, d, ref_codes):
    got = unpack_codes(codes_gpu.cpu().numpy(), scheme, s, n, d)
    mism = np.argwhere(got != ref_codes)
    assert len(mism) == 0, "%d codes differ, first at %s" % (len(mism), mism[:5].tolist())


def _max_case(scheme, s, dtype, n, d, count=4096, seed=1):
    rng = np.random.default_rng(seed + 7 * s + (dtype == "bf16"))
    if scheme == LINEAR and s == 127 and dtype == "f32":
        return bi.max_norm_matrix(n, d, scheme, s, SEED, STEP, count, rng, dtype, N=WORST_N,
                                  worst=256)
    return bi.max_norm_matrix(n, d, scheme, s, SEED, STEP, count, rng, dtype)


SCHEMES = [(LINEAR, 127), (LINEAR, 7), (EXP, 8), (EXP, 4)]


def _fused(gq, oracle, xh, q, p, scheme, s, expect_launches):
    import torch
    n, d = xh.shape
    x = to_device(xh)
    assert gq.gq_fused_launches(x.dtype, n, d) == expect_launches
    ws = gq.gq_workspace()
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    out = gq.gq_allreduce_mean(x, q, p, scheme, s, SEED, STEP, norm=norm, ws=ws)
    codes = torch.empty(gq.gq_code_bytes(scheme, s, n, d), dtype=torch.uint8, device="cuda")
    norm2 = torch.empty(1, dtype=torch.float32, device="cuda")
    out2 = gq.gq_allreduce_mean(x, q, p, scheme, s, SEED, STEP, norm=norm2, codes=codes, ws=ws)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    N32 = np.float32(norm.item())
    want64 = oracle.global_norm(xh, q, p)
    if (q, p) == (INF, INF):
        assert N32 == np.float32(want64)
    else:
        assert float(N32) == pytest.approx(want64, rel=1e-6)
    ref_codes, sums, ref_out = _oracle(oracle, xh, N32, scheme, s)
    _compare_out(out, N32, scheme, s, n, sums, ref_out)
    N2 = np.float32(norm2.item())
    if N2 != N32:  # the single launch may split an l2 sum differently from the two-pass form
        ref_codes, sums, ref_out = _oracle(oracle, xh, N2, scheme, s)
    _compare_codes(codes, scheme, s, n, d, ref_codes)
    _compare_out(out2, N2, scheme, s, n, sums, ref_out)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scheme,s", SCHEMES)
def test_fused_bulk_copy_max_norm(gq, oracle, dtype, scheme, s):
    n, d = 8, (1 << 20) if dtype == "f32" else (1 << 21)
    xh, info = _max_case(scheme, s, dtype, n, d)
    _fused(gq, oracle, xh, INF, INF, scheme, s, 2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scheme,s", [(EXP, 8), (EXP, 4), (LINEAR, 7), (LINEAR, 127)])
def test_fused_bulk_copy_l2(gq, oracle, dtype, scheme, s):
    """The (2, 2) norm: the compacting consumer (row-groups whose elements all round down are
    settled by one comparison; the rest are queued and decided a warp at a time)."""
    n, d = 8, (1 << 20) if dtype == "f32" else (1 << 21)
    rng = np.random.default_rng(40 + s + scheme)
    xh, info = bi.l2_norm_matrix(n, d, scheme, s, SEED, STEP, 4096, rng, dtype)
    _fused(gq, oracle, xh, 2, 2, scheme, s, 2)


@pytest.mark.parametrize("scheme,s", SCHEMES)
def test_fused_direct_load_unaligned(gq, oracle, scheme, s):
    n, d = 5, (1 << 18) + 3  # rows not 16-byte aligned: direct loads
    xh, _ = _max_case(scheme, s, "f32", n, d, count=2048)
    _fused(gq, oracle, xh, INF, INF, scheme, s, 2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scheme,s", SCHEMES)
def test_single_launch(gq, oracle, dtype, scheme, s):
    import torch
    n, d = 4, 65536
    xh, _ = _max_case(scheme, s, dtype, n, d, count=2048)
    x = to_device(xh)
    assert gq.gq_fused_launches(x.dtype, n, d) == 1
    ws = gq.gq_workspace()
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    out = gq.gq_allreduce_mean(x, INF, INF, scheme, s, SEED, STEP, norm=norm, ws=ws)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    N32 = np.float32(norm.item())
    assert N32 == np.float32(oracle.global_norm(xh, INF, INF))
    _, sums, ref_out = _oracle(oracle, xh, N32, scheme, s)
    _compare_out(out, N32, scheme, s, n, sums, ref_out)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scheme,s", SCHEMES)
def test_supplied_norm(gq, oracle, dtype, scheme, s):
    """gq_allreduce_mean_with_norm and gq_quantize (no workspace: direct loads; the norm is not
    trusted, so |x| above N saturates at the top level)."""
    import torch
    n, d = 6, 200_000
    rng = np.random.default_rng(60 + s)
    N = 0.7431
    xh, info = bi.supplied_norm_matrix(n, d, scheme, s, SEED, STEP, 3072, rng, N, dtype)
    x = to_device(xh)
    N32 = np.float32(info["N"])
    norm = torch.tensor([float(N32)], dtype=torch.float32, device="cuda")
    out = gq.gq_allreduce_mean_with_norm(x, norm, scheme, s, SEED, STEP)
    codes = gq.gq_quantize(x, norm, scheme, s, SEED, STEP)
    torch.cuda.synchronize()
    ref_codes, sums, ref_out = _oracle(oracle, xh, N32, scheme, s)
    _compare_out(out, N32, scheme, s, n, sums, ref_out)
    _compare_codes(codes, scheme, s, n, d, ref_codes)


@pytest.mark.parametrize("big", [True, False])
@pytest.mark.parametrize("scheme,s", [(LINEAR, 127), (EXP, 8)])
def test_segments(gq, oracle, big, scheme, s):
    """Segment l draws with step (step << 16) | l; each segment has its own max norm."""
    import torch
    n = 4
    sizes = [400_000, 263_168, 310_000] if big else [5003, 65536, 1 << 14]
    hosts, xs = [], []
    for l, d in enumerate(sizes):
        rng = np.random.default_rng(80 + l + 10 * s)
        xh, _ = bi.max_norm_matrix(n, d, scheme, s, SEED, (STEP << 16) | l, 1024, rng,
                                   N=0.5 + l)
        hosts.append(xh)
        xs.append(to_device(xh))
    ws = gq.gq_workspace()
    norms = torch.empty(len(sizes), dtype=torch.float32, device="cuda")
    outs = gq.gq_allreduce_mean_segments(xs, INF, INF, scheme, s, SEED, STEP, norms=norms, ws=ws)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    for l, (xh, out) in enumerate(zip(hosts, outs)):
        N32 = np.float32(norms[l].item())
        assert N32 == np.float32(oracle.global_norm(xh, INF, INF))
        _, sums, ref_out = _oracle(oracle, xh, N32, scheme, s, step=(STEP << 16) | l)
        _compare_out(out, N32, scheme, s, n, sums, ref_out)


@pytest.mark.parametrize("m,with_ws", [(1, True), (2, True), (3, False)])
@pytest.mark.parametrize("scheme,s", [(LINEAR, 15), (EXP, 4)])
def test_rank_sums_and_codes(gq, oracle, m, with_ws, scheme, s):
    """One rank's rows (workers 5 ..): integer code sums and codes, against the oracle's rows 5 ..
    of the stacked matrix; with a workspace, large aligned rows take the bulk-copy kernel (one
    row at a time for a single worker)."""
    import torch
    worker0 = 5
    d = 1 << 20
    rng = np.random.default_rng(90 + m + s)
    xh, _ = bi.max_norm_matrix(m, d, scheme, s, SEED, STEP, 3072, rng, worker0=worker0)
    x = to_device(xh)
    N32 = np.float32(oracle.global_norm(xh, INF, INF))
    norm = torch.tensor([float(N32)], dtype=torch.float32, device="cuda")
    ws = gq.gq_workspace() if with_ws else None
    sums = gq.gq_quantize_sum(x, norm, scheme, s, SEED, STEP, worker0=worker0, ws=ws)
    codes = gq.gq_quantize_codes(x, norm, scheme, s, SEED, STEP, worker0=worker0, ws=ws)
    torch.cuda.synchronize()
    if ws is not None:
        assert gq.gq_get_status(ws) == 0
    ref_codes, ref_sums, _ = _oracle(oracle, xh, N32, scheme, s, worker0=worker0)
    np.testing.assert_array_equal(sums.cpu().numpy().astype(np.int64), ref_sums)
    got = unpack_codes(codes.cpu().numpy(), EXP, 8, m, d)  # int8 codes whatever s is
    np.testing.assert_array_equal(got, ref_codes)
