"""gq_allreduce_mean_noalloc: the allreduce-mean for callers that cannot allocate device memory.

Some callers have no way to get a workspace buffer at the point where they quantise: code that
runs inside a framework's caching allocator or communication hook (which may not call back into
the allocator) or a process whose device memory is planned in full ahead of time.  For them the
library keeps the norm step's scratch in a fixed array of its own device memory.  This test calls
that entry point through the C ABI twice in a row and checks each result against the regular
gq_allreduce_mean (same tolerance as the other parity tests: the norm and the codes identical, the
dequantised mean within 1e-6 * N).  It does not depend on what ran before it in the process, so it
passes alone in a fresh process and after the rest of the suite.
"""
import ctypes

import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("q,p,scheme,s", [(0, 0, 0, 127), (2, 2, 1, 8), (2, 0, 1, 4),
                                          (0, 2, 0, 15)])
def test_noalloc_matches_allreduce_mean(dtype, q, p, scheme, s):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from allreduce_compatible_gradient_gb300 import _build, workloads

    _build.build_library()
    import allreduce_compatible_gradient_gb300 as gq

    lib = gq.lib()
    n, d = 8, 300_007  # several blocks per SM wave and a ragged tail
    x = workloads.device_inputs("student_t3" if dtype == "bf16" else "normal", n, d, seed=3,
                                dtype=dtype)
    dt = 0 if dtype == "f32" else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    nbytes = gq.gq_code_bytes(scheme, s, n, d)
    for step in (11, 12):  # two calls in a row share the fixed scratch
        out = torch.empty(d, dtype=torch.float32, device="cuda")
        norm = torch.empty(1, dtype=torch.float32, device="cuda")
        codes = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        rc = lib.gq_allreduce_mean_noalloc(
            ctypes.c_void_p(x.data_ptr()), dt, n, d, q, p, scheme, s, 5, step,
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(norm.data_ptr()),
            ctypes.c_void_p(codes.data_ptr()), stream)
        assert rc == 0, gq.gq_status_string(rc)
        ref_norm = torch.empty(1, dtype=torch.float32, device="cuda")
        ref_codes = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        ref = gq.gq_allreduce_mean(x, q, p, scheme, s, 5, step, norm=ref_norm, codes=ref_codes)
        torch.cuda.synchronize()
        assert float(norm.item()) == float(ref_norm.item())
        assert torch.equal(codes, ref_codes)
        N = float(ref_norm.item())
        err = (out.double() - ref.double()).abs().max().item()
        assert err <= 1e-6 * N


def test_noalloc_argument_checks():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from allreduce_compatible_gradient_gb300 import _build

    _build.build_library()
    import allreduce_compatible_gradient_gb300 as gq

    lib = gq.lib()
    x = torch.randn((4, 64), device="cuda")
    out = torch.empty(64, device="cuda")
    rc = lib.gq_allreduce_mean_noalloc(ctypes.c_void_p(x.data_ptr()), 0, 4, 64, 1, 2, 0, 5, 1, 1,
                                       ctypes.c_void_p(out.data_ptr()), None, None, None)
    assert rc == 1  # bad norm order
    rc = lib.gq_allreduce_mean_noalloc(ctypes.c_void_p(x.data_ptr()), 0, 4, 64, 2, 2, 0, 200, 1, 1,
                                       ctypes.c_void_p(out.data_ptr()), None, None, None)
    assert rc == 2  # unsupported s
