"""gq_allreduce_mean_noalloc: the allreduce-mean for callers that cannot allocate device memory.

Some callers have no way to get a workspace buffer at the point where they quantise: code that
runs inside a framework's caching allocator or communication hook (which may not call back into
the allocator) or a process whose device memory is planned in full ahead of time.  For them the
library keeps the scratch in a fixed array of its own device memory.  These tests call that entry
point through the C ABI, two calls in a row on every shape, and check each result:
  * against the oracle: the norm (exact for the max norm, 1e-6 for the l2 forms), every code bit
    for bit, the integer sums read back from the mean exactly and the mean within 1e-6 N, on
    every coordinate;
  * against the regular gq_allreduce_mean, which takes the same kernels: norm, codes and mean
    bit for bit;
on 16-byte aligned rows large enough for the bulk-copy quantise kernel, ragged rows (direct
loads), a small problem without codes (the single launch), with and without a code output.  The
refusal rule for problems whose norm step needs more block partials than the fixed array holds is
checked through the block-count query.  Nothing here depends on what ran before in the process,
so the file passes alone in a fresh process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

CASES = [
    # n, d, dtype, q, p, scheme, s, with codes
    (8, 1 << 20, "f32", 0, 0, 0, 127, False),   # bulk-copy kernel
    (8, 1 << 20, "bf16", 2, 2, 1, 8, False),    # bulk-copy kernel, compacting consumer
    (8, 1 << 20, "f32", 2, 0, 1, 4, True),      # bulk-copy kernel with codes
    (8, 300_007, "f32", 0, 2, 0, 15, True),     # ragged rows: direct loads
    (8, 300_007, "bf16", 2, 2, 1, 8, False),
    (4, 65_536, "f32", 2, 2, 0, 7, False),      # the single launch
    (4, 65_536, "bf16", 0, 0, 1, 4, True),      # with codes: two launches
]


def _gq():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from allreduce_compatible_gradient_gb300 import _build

    _build.build_library()
    import allreduce_compatible_gradient_gb300 as gq

    gq.lib()
    return torch, gq


def _oracle_check(oracle, xh, N32, scheme, s, seed, step, out, codes_u8, n, d):
    from gpu_common import unpack_codes

    ref_codes, rc = oracle.quantize(xh, N32, scheme, s, seed, step)
    assert rc == 0
    sums = oracle.reduce_codes(ref_codes, scheme, s)
    ref_out, rc = oracle.dequantize(sums, N32, scheme, s, n)
    got = out.astype(np.float64)
    scale = float(np.float32(float(N32) / (n * s))) if scheme == 0 else float(
        np.float32(np.ldexp(float(N32), -(s - 1)) / n))
    np.testing.assert_array_equal(np.rint(got / scale).astype(np.int64), sums)
    assert np.abs(got - ref_out).max() <= 1e-6 * float(N32)
    if codes_u8 is not None:
        np.testing.assert_array_equal(unpack_codes(codes_u8, scheme, s, n, d), ref_codes)


@pytest.mark.parametrize("n,d,dtype,q,p,scheme,s,with_codes", CASES)
def test_noalloc_against_oracle_and_allreduce_mean(oracle, n, d, dtype, q, p, scheme, s,
                                                   with_codes):
    torch, gq = _gq()
    from allreduce_compatible_gradient_gb300 import workloads
    from gpu_common import to_host

    lib = gq.lib()
    x = workloads.device_inputs("student_t3" if dtype == "bf16" else "normal", n, d, seed=3,
                                dtype=dtype)
    xh = to_host(x)
    dt = 0 if dtype == "f32" else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    nbytes = gq.gq_code_bytes(scheme, s, n, d)
    want64 = oracle.global_norm(xh, q, p)
    for step in (11, 12):  # two calls in a row share the fixed scratch
        out = torch.empty(d, dtype=torch.float32, device="cuda")
        norm = torch.empty(1, dtype=torch.float32, device="cuda")
        codes = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if with_codes else None
        rc = lib.gq_allreduce_mean_noalloc(
            ctypes.c_void_p(x.data_ptr()), dt, n, d, q, p, scheme, s, 5, step,
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(norm.data_ptr()),
            ctypes.c_void_p(codes.data_ptr()) if with_codes else None, stream)
        assert rc == 0, gq.gq_status_string(rc)
        ref_norm = torch.empty(1, dtype=torch.float32, device="cuda")
        ref_codes = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if with_codes else None
        ref = gq.gq_allreduce_mean(x, q, p, scheme, s, 5, step, norm=ref_norm, codes=ref_codes)
        torch.cuda.synchronize()
        N32 = np.float32(norm.item())
        if (q, p) == (0, 0):
            assert N32 == np.float32(want64)
        else:
            assert float(N32) == pytest.approx(want64, rel=1e-6)
        assert N32 == np.float32(ref_norm.item())
        assert torch.equal(out, ref)
        if with_codes:
            assert torch.equal(codes, ref_codes)
        _oracle_check(oracle, xh, N32, scheme, s, 5, step, out.cpu().numpy(),
                      codes.cpu().numpy() if with_codes else None, n, d)


def test_noalloc_block_rule():
    """The fixed scratch holds gq_noalloc_max_blocks() norm partials; the call is refused with
    GQ_ERR_WORKSPACE exactly when gq_norm_blocks exceeds it.  On this GPU every size stays within
    it (the norm step's grid is at most a few waves of the SM count), so the refusal itself cannot
    be reached: the rule is pinned through the two queries."""
    torch, gq = _gq()
    assert gq.gq_noalloc_max_blocks() == 1024
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for dt in (gq.F32, gq.BF16):
        for q, p in ((0, 0), (2, 2), (2, 0), (0, 2)):
            for n, d in ((1, 1), (3, 1000), (8, 1 << 20), (16, 350_000_000), (64, 1 << 28)):
                b = gq.gq_norm_blocks(dt, n, d, q, p)
                assert 1 <= b <= gq.gq_noalloc_max_blocks()
                assert b <= 4 * sms
    assert gq.gq_norm_blocks(gq.F32, 0, 10, 2, 2) == 0
    assert gq.gq_norm_blocks(gq.F32, 4, 10, 3, 2) == 0


def test_noalloc_argument_checks():
    torch, gq = _gq()
    lib = gq.lib()
    x = torch.randn((4, 64), device="cuda")
    out = torch.empty(64, device="cuda")
    rc = lib.gq_allreduce_mean_noalloc(ctypes.c_void_p(x.data_ptr()), 0, 4, 64, 1, 2, 0, 5, 1, 1,
                                       ctypes.c_void_p(out.data_ptr()), None, None, None)
    assert rc == 1  # bad norm order
    rc = lib.gq_allreduce_mean_noalloc(ctypes.c_void_p(x.data_ptr()), 0, 4, 64, 2, 2, 0, 200, 1, 1,
                                       ctypes.c_void_p(out.data_ptr()), None, None, None)
    assert rc == 2  # unsupported s
