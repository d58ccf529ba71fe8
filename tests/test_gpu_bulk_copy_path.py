"""GPU parity of the fused path's bulk-copy kernel (quantize_tma_kernel).

The fused call takes that kernel for 16-byte aligned rows with at least one 3840-column chunk
per SM (d >= 583,680 on 152 SMs).  At such sizes, with ragged last groups, odd worker counts,
one worker, both dtypes, both schemes and every code width, the fused result (out and codes)
must equal the unfused chain (norm, quantise, sum, dequantise: the direct-load kernels, pinned
to the oracle elsewhere) bit for bit, and sampled column windows (first, last, seeded interior)
must match the oracle: codes bit-exact, out within 1e-6 N.  The workspace status stays 0 (no
bounded wait gave up).
"""
import numpy as np
import pytest

from gpu_common import EXP, INF, LINEAR, gq_module, to_device, to_host, unpack_codes
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu

CASES = [
    # n, d, dtype, scheme, s, with codes
    (5, 600_004, "f32", LINEAR, 7, True),     # d % 8 = 4: the last group is half full
    (5, 600_004, "f32", EXP, 8, False),
    (8, 1_000_000, "f32", LINEAR, 127, True),
    (1, 700_000, "f32", EXP, 4, True),        # one worker: stages of one row
    (2, 800_000, "f32", LINEAR, 7, True),     # two workers: stages of two rows, twice as many
    (2, 1_310_720, "bf16", EXP, 8, False),
    (7, 640_000, "f32", LINEAR, 15, False),
    (3, 600_000, "bf16", EXP, 4, True),
    (8, 655_360, "bf16", LINEAR, 15, False),
    (6, 1_200_008, "bf16", EXP, 8, True),
]


@pytest.fixture(scope="module")
def gq():
    return gq_module()


@pytest.fixture(scope="module")
def oracle_mod():
    from oracle import gq_oracle
    gq_oracle.lib()
    return gq_oracle


def _windows(d, seed):
    rng = np.random.default_rng(seed)
    starts = {0, d - 1003}
    while len(starts) < 5:
        starts.add(int(rng.integers(0, d - 1003)) // 32 * 32)
    return sorted((s0, min(d, s0 + 1003)) for s0 in starts)


@pytest.mark.parametrize("n,d,dtype,scheme,s,with_codes", CASES)
def test_bulk_copy_path(gq, oracle_mod, n, d, dtype, scheme, s, with_codes):
    import torch
    x = workloads.device_inputs("normal" if dtype == "f32" else "student_t3", n, d, seed=d + n,
                                dtype=dtype)
    seed, step = 21, 5
    ws = gq.gq_workspace()
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    cb = gq.gq_code_bytes(scheme, s, n, d)
    codes = torch.empty(cb, dtype=torch.uint8, device="cuda") if with_codes else None
    out = gq.gq_allreduce_mean(x, INF, INF, scheme, s, seed, step, norm=norm, codes=codes, ws=ws)
    # the unfused chain
    n2 = gq.gq_global_norm(x, INF, INF)
    c2 = gq.gq_quantize(x, n2, scheme, s, seed, step)
    sums = gq.gq_reduce_codes(c2, scheme, s, n, d)
    ref = gq.gq_dequantize(sums, n2, scheme, s, n)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    assert torch.equal(norm, n2)
    assert torch.equal(out, ref)
    if with_codes:
        assert torch.equal(codes, c2)

    # sampled windows against the oracle
    xh = to_host(x)
    norm32 = float(norm.item())
    assert norm32 == float(np.float32(oracle_mod.global_norm(xh, INF, INF)))
    out_h = out.cpu().numpy().astype(np.float64)
    bits = gq.gq_code_bits(scheme, s)
    pitch = gq.gq_code_pitch(d)
    codes_h = c2.cpu().numpy().reshape(n, pitch * bits // 8)
    for j0, j1 in _windows(d, seed=d):
        ref_codes, rc = oracle_mod.quantize(xh, norm32, scheme, s, seed, step, j0, j1)
        assert rc == 0
        ref_out, rc = oracle_mod.dequantize(oracle_mod.reduce_codes(ref_codes, scheme, s), norm32,
                                            scheme, s, n)
        assert rc == 0
        a0 = j0 // 32 * 32
        a1 = min(pitch, (j1 + 31) // 32 * 32)
        win = unpack_codes(np.ascontiguousarray(codes_h[:, a0 * bits // 8:a1 * bits // 8]).ravel(),
                           scheme, s, n, a1 - a0, check_padding=False)
        np.testing.assert_array_equal(win[:, j0 - a0:j1 - a0], ref_codes)
        assert np.abs(out_h[j0:j1] - ref_out).max() <= 1e-6 * norm32


def test_bulk_copy_path_l2_norm_and_zero(gq):
    """(2,2) norm through the bulk-copy path equals the unfused chain with the same norm; an
    all-zero problem gives zeros and status 0."""
    import torch
    n, d = 4, 800_000
    x = workloads.device_inputs("normal", n, d, seed=3)
    ws = gq.gq_workspace()
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    out = gq.gq_allreduce_mean(x, 2, 2, EXP, 8, 1, 1, norm=norm, ws=ws)
    ref = gq.gq_allreduce_mean_with_norm(x, norm, EXP, 8, 1, 1)
    z = torch.zeros(n, d, device="cuda")
    outz = gq.gq_allreduce_mean(z, 2, 2, LINEAR, 15, 1, 1, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.count_nonzero(outz) == 0
    assert gq.gq_get_status(ws) == 0


@pytest.mark.parametrize("dtype,scheme,s,with_codes", [("f32", EXP, 8, True), ("f32", LINEAR, 127, False),
                                                    ("bf16", EXP, 4, False), ("bf16", LINEAR, 15, True)])
def test_with_norm_workspace(gq, oracle_mod, dtype, scheme, s, with_codes):
    """gq_allreduce_mean_with_norm_ws and gq_quantize_ws (the bulk-copy kernel under a supplied,
    untrusted norm) equal gq_allreduce_mean_with_norm and gq_quantize (direct loads) bit for bit,
    codes too, on values above the norm, a NaN and zero blocks; and the oracle on windows."""
    import torch
    from gpu_common import to_host, unpack_codes
    n, d = 5, 1_048_576
    x = workloads.device_inputs("laplace_block_sparse", n, d, seed=11, dtype=dtype)
    x[1, 5] = float("nan")
    norm = gq.gq_global_norm(x[2:], 0, 0) * 0.5  # half the maximum of rows 2..: many |x| above N
    ws = gq.gq_workspace()
    cb = gq.gq_code_bytes(scheme, s, n, d)
    c1 = torch.empty(cb, dtype=torch.uint8, device="cuda") if with_codes else None
    c2 = torch.empty(cb, dtype=torch.uint8, device="cuda") if with_codes else None
    got = gq.gq_allreduce_mean_with_norm_ws(x, norm, scheme, s, 6, 7, ws, codes=c1)
    ref = gq.gq_allreduce_mean_with_norm(x, norm, scheme, s, 6, 7, codes=c2)
    q1 = gq.gq_quantize_ws(x, norm, scheme, s, 6, 7, ws)   # codes alone, both kernels
    q2 = gq.gq_quantize(x, norm, scheme, s, 6, 7)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    assert torch.equal(got, ref)
    assert torch.equal(q1, q2)
    if with_codes:
        assert torch.equal(c1, c2)
        assert torch.equal(q1, c1)
    xh = to_host(x)
    N32 = np.float32(norm.item())
    out_h = got.cpu().numpy().astype(np.float64)
    allc = unpack_codes(c1.cpu().numpy(), scheme, s, n, d) if with_codes else None
    for j0, j1 in _windows(d, 3):
        xw = np.ascontiguousarray(xh[:, j0:j1])
        codes, rc = oracle_mod.quantize_cols(xw, j0, N32, scheme, s, 6, 7)
        assert rc == 0
        sums = oracle_mod.reduce_codes(codes, scheme, s)
        want, _ = oracle_mod.dequantize(sums, N32, scheme, s, n)
        assert np.abs(out_h[j0:j1] - want).max() <= 1e-6 * float(N32)
        if with_codes:
            np.testing.assert_array_equal(allc[:, j0:j1], codes)


COMPACT_CASES = [
    # n, d, dtype, scheme, s, (q, p)
    (1, 700_000, "f32", EXP, 8, (2, 2)),       # one worker: stages of one row
    (2, 900_000, "bf16", EXP, 8, (2, 2)),      # two workers: stages of two rows
    (2, 800_004, "f32", LINEAR, 15, (2, 2)),
    (3, 600_004, "f32", LINEAR, 7, (2, 2)),    # ragged last group
    (5, 640_000, "bf16", EXP, 4, (2, 2)),
    (8, 1_000_000, "f32", EXP, 21, (2, 2)),    # the largest s for 8 workers
    (13, 655_360, "bf16", LINEAR, 127, (2, 2)),
    (33, 600_000, "f32", EXP, 8, (INF, 2)),
    (6, 1_200_008, "bf16", EXP, 8, (INF, 2)),
]


@pytest.mark.parametrize("n,d,dtype,scheme,s,qp", COMPACT_CASES)
def test_compacting_consumer(gq, oracle_mod, n, d, dtype, scheme, s, qp):
    """Norms with p = 2 take the compacting consumer (row-groups that certainly round down are
    settled at once, the rest queued per warp and decided a warp at a time): its mean equals the
    direct-load kernel's given the same norm bit for bit, and the oracle's on sampled windows.
    Heavy-tailed inputs, so that some row-groups of most warps are queued."""
    import torch
    x = workloads.device_inputs("student_t3", n, d, seed=d + n, dtype=dtype)
    q, p = qp
    seed, step = 21, 6
    ws = gq.gq_workspace()
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    out = gq.gq_allreduce_mean(x, q, p, scheme, s, seed, step, norm=norm, ws=ws)
    ref = gq.gq_allreduce_mean_with_norm(x, norm, scheme, s, seed, step)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    assert torch.equal(out, ref)
    xh = to_host(x)
    norm32 = float(norm.item())
    assert norm32 == pytest.approx(oracle_mod.global_norm(xh, q, p), rel=1e-6)
    out_h = out.cpu().numpy().astype(np.float64)
    for j0, j1 in _windows(d, seed=d + 1):
        ref_codes, rc = oracle_mod.quantize(xh, norm32, scheme, s, seed, step, j0, j1)
        assert rc == 0
        ref_out, rc = oracle_mod.dequantize(oracle_mod.reduce_codes(ref_codes, scheme, s), norm32,
                                            scheme, s, n)
        assert np.abs(out_h[j0:j1] - ref_out).max() <= 1e-6 * norm32


@pytest.mark.parametrize("dtype,scheme,s,qp", [("f32", EXP, 4, (2, INF)), ("f32", LINEAR, 127, (INF, INF)),
                                               ("bf16", EXP, 8, (INF, INF)), ("f32", EXP, 8, (2, 2))])
def test_zero_blocks(gq, dtype, scheme, s, qp):
    """Block-sparse inputs (half of the 4096-coordinate blocks zero for every worker, as in sparse
    layers), with signed zeros, single non-zero elements in zero blocks and a worker whose rows
    are zero in another pattern: rows that are zero across a warp skip their random words; the
    result equals the direct-load kernel's bit for bit."""
    import torch
    n, d = 7, 1_048_576
    x = workloads.device_inputs("laplace_block_sparse", n, d, seed=5, dtype=dtype)
    flat = x.view(-1)
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    idx = torch.randint(0, n * d, (64,), generator=g, device="cuda")
    flat[idx[:32]] = -0.0
    flat[idx[32:]] = 3e-3
    x[3, : d // 2] = 0
    q, p = qp
    ws = gq.gq_workspace()
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    out = gq.gq_allreduce_mean(x, q, p, scheme, s, 4, 2, norm=norm, ws=ws)
    ref = gq.gq_allreduce_mean_with_norm(x, norm, scheme, s, 4, 2)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    assert torch.equal(out, ref)
    assert torch.count_nonzero(out) > 0
