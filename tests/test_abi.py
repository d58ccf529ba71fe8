"""The C ABI on a machine without a GPU: the library loads, exports every entry point that
include/gq.h declares, and its host-only functions and argument checks behave as documented
(none of these calls reaches the GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gq_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from allreduce_compatible_gradient_gb300 import _build
    path = _build.build_library()
    return ctypes.CDLL(path)


def test_header_declares_the_pipeline():
    names = declared_functions()
    for want in ("gq_global_norm", "gq_quantize", "gq_reduce_codes", "gq_dequantize",
                 "gq_allreduce_mean", "gq_get_status", "gq_workspace_bytes"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_entry_point():
    import allreduce_compatible_gradient_gb300 as gq
    for name in declared_functions():
        if name == "gq_workspace_init":
            continue  # wrapped by gq_workspace()
        assert hasattr(gq, name), name


def test_host_only_functions():
    import allreduce_compatible_gradient_gb300 as gq
    assert gq.gq_abi_version() == 1
    assert gq.gq_workspace_bytes(8, 10**9) == 256 + 8 * 4096 + 3 * 4 * 256
    assert [gq.gq_code_bits(0, s) for s in (0, 1, 7, 8, 127, 128)] == [0, 4, 4, 8, 8, 0]
    assert [gq.gq_code_bits(1, s) for s in (0, 1, 7, 8, 24, 25)] == [0, 4, 4, 8, 8, 0]
    assert gq.gq_code_bits(2, 5) == 0
    assert [gq.gq_code_pitch(d) for d in (0, 1, 32, 33, 25_557_032)] == [0, 32, 32, 64, 25_557_056]
    assert gq.gq_code_bytes(0, 127, 8, 25_557_032) == 8 * 25_557_056
    assert gq.gq_code_bytes(1, 4, 16, 350_000_000) == 16 * 350_000_000 // 2
    assert gq.gq_code_bytes(1, 4, 3, 33) == 3 * 64 // 2
    assert gq.gq_status_string(0) == "ok"
    assert gq.gq_status_string(4) == "non-finite norm"
    assert gq.gq_status_string(99) == "unknown status"


def test_fused_launch_count_query():
    """One launch for small aligned problems without a code output, two otherwise (far from the
    size boundary, which depends on the SM count); 0 for invalid arguments."""
    import allreduce_compatible_gradient_gb300 as gq
    assert gq.gq_fused_launches(gq.F32, 4, 65_536) == 1
    assert gq.gq_fused_launches(gq.BF16, 8, 1 << 20) == 1
    assert gq.gq_fused_launches(gq.F32, 4, 65_536, with_codes=True) == 2
    assert gq.gq_fused_launches(gq.F32, 4, 65_538) == 2   # rows not 16-byte aligned
    assert gq.gq_fused_launches(gq.BF16, 4, 65_540) == 2  # (8 bf16 per 16 bytes)
    assert gq.gq_fused_launches(gq.F32, 8, 25_557_032) == 2
    assert gq.gq_fused_launches(gq.F32, 1 << 20, 8) == 2
    assert gq.gq_fused_launches(gq.F16, 4, 64) == 0      # not a gradient type
    assert gq.gq_fused_launches(gq.F32, 0, 64) == 0
    assert gq.gq_fused_launches(gq.F32, 4, 0) == 0


def test_fused_launch_rule_matches_its_documentation():
    """The size rule gq.h states for the single launch, n * 8 * ceil(ceil(d / 8) / SMs) * bytes
    <= 204,800 with 16-byte aligned rows and no code output, over a grid of shapes (152 SMs: the
    count the library assumes where no GPU answers)."""
    import torch
    import allreduce_compatible_gradient_gb300 as gq
    if torch.cuda.is_available():
        pytest.skip("the SM count of a present GPU decides; checked on the GPU by the resident tests")
    for dtype, elt in ((gq.F32, 4), (gq.BF16, 2)):
        for n in (1, 2, 3, 8, 16, 64, 257):
            for d in (1, 4, 8, 12, 1000, 65_536, 65_540, 972_800, 972_808, 5_187_456, 7_782_400,
                      7_782_408, 40_000_000):
                groups = -(-d // 8)
                gpb = -(-groups // 152)
                want = 1 if (d % (16 // elt) == 0 and n * 8 * gpb * elt <= 204_800) else 2
                assert gq.gq_fused_launches(dtype, n, d) == want, (dtype, n, d)
                assert gq.gq_fused_launches(dtype, n, d, with_codes=True) == 2


def test_argument_checks_return_before_any_device_call(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("fake pointers: run only where no GPU can be reached")
    vp, i64, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
    lib.gq_global_norm.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_int, vp, vp,
                                   ctypes.c_size_t, vp]
    lib.gq_quantize.argtypes = [vp, ctypes.c_int, i64, i64, vp, ctypes.c_int, ctypes.c_int, u64,
                                u64, vp, vp]
    fake = vp(1 << 20)  # aligned, never dereferenced: every call below fails its checks first
    ws_bytes = 256 + 8 * 4096
    assert lib.gq_global_norm(None, 0, 2, 2, 2, 2, fake, fake, ws_bytes, None) == 1
    assert lib.gq_global_norm(vp((1 << 20) + 4), 0, 2, 2, 2, 2, fake, fake, ws_bytes, None) == 1
    assert lib.gq_global_norm(fake, 0, 0, 2, 2, 2, fake, fake, ws_bytes, None) == 1
    assert lib.gq_global_norm(fake, 0, 2, 1 << 34, 2, 2, fake, fake, ws_bytes, None) == 1
    assert lib.gq_global_norm(fake, 2, 2, 2, 2, 2, fake, fake, ws_bytes, None) == 1
    assert lib.gq_global_norm(fake, 0, 2, 2, 1, 2, fake, fake, ws_bytes, None) == 1
    assert lib.gq_global_norm(fake, 0, 2, 2, 2, 2, fake, fake, 100, None) == 7
    assert lib.gq_global_norm(fake, 0, 2, 2, 2, 2, fake, None, ws_bytes, None) == 7
    assert lib.gq_quantize(fake, 0, 2, 2, fake, 0, 0, 1, 1, fake, None) == 2
    assert lib.gq_quantize(fake, 0, 2, 2, fake, 0, 128, 1, 1, fake, None) == 2
    assert lib.gq_quantize(fake, 0, 2, 2, fake, 1, 25, 1, 1, fake, None) == 2
    assert lib.gq_quantize(fake, 0, 2, 2, fake, 7, 5, 1, 1, fake, None) == 1
    assert lib.gq_quantize(fake, 0, 163840, 2, fake, 0, 127, 1, 1, fake, None) == 3
    assert lib.gq_quantize(fake, 0, 4, 2, fake, 1, 23, 1, 1, fake, None) == 3
    assert lib.gq_quantize(fake, 0, 2, 2, None, 0, 5, 1, 1, fake, None) == 1


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    from allreduce_compatible_gradient_gb300 import _binding
    monkeypatch.setattr(_binding, "_LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(ImportError):
        _binding.lib()


def test_argument_checks_of_the_bucket_and_rank_entry_points(lib):
    """gq_allreduce_mean_segments, gq_quantize_sum, gq_norm_partial / gq_norm_finish and the
    *_to output-type entry points refuse bad arguments before any device call."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("fake pointers: run only where no GPU can be reached")
    vp, i64, u64, ci, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_size_t
    lib.gq_allreduce_mean_segments.argtypes = [i64, vp, vp, ci, i64, ci, ci, ci, ci, u64, u64, vp,
                                               ci, vp, vp, sz, vp]
    lib.gq_quantize_sum.argtypes = [vp, ci, i64, i64, i64, vp, ci, ci, u64, u64, vp, ci, vp, sz,
                                    vp]
    lib.gq_dequantize_sums.argtypes = [vp, ci, vp, ci, ci, i64, i64, vp, ci, vp]
    lib.gq_norm_partial.argtypes = [vp, ci, i64, i64, ci, ci, vp, vp, sz, vp]
    lib.gq_norm_finish.argtypes = [vp, ci, ci, vp, vp]
    lib.gq_dequantize_to.argtypes = [vp, vp, ci, ci, i64, i64, vp, ci, vp]
    lib.gq_allreduce_mean_to.argtypes = [vp, ci, i64, i64, ci, ci, ci, ci, u64, u64, vp, ci, vp,
                                         vp, vp, sz, vp]
    fake = 1 << 20
    ws_bytes = lib.gq_workspace_bytes(1, 1)
    P = ctypes.c_void_p * 2
    D = ctypes.c_int64 * 2
    grads, outs, ds = P(fake, fake + 4096), P(fake, fake + 4096), D(100, 200)

    def seg(nseg=2, g=grads, d=ds, n=4, q=0, p=0, scheme=1, s=8, step=1, o=outs, odt=0,
            ws=fake, wsb=ws_bytes):
        return lib.gq_allreduce_mean_segments(nseg, g, d, 0, n, q, p, scheme, s, 1, step, o, odt,
                                              None, vp(ws) if ws else None, wsb, None)
    assert seg(nseg=0) == 1
    assert seg(nseg=65537) == 1
    assert seg(step=1 << 48) == 1
    assert seg(odt=3) == 1
    assert seg(g=P(fake, fake + 4)) == 1                # unaligned second segment
    assert seg(o=P(fake, fake + 8)) == 1                # unaligned second output
    assert seg(d=D(100, 0)) == 1
    assert seg(q=1) == 1
    assert seg(s=25) == 2
    assert seg(n=1 << 17) == 3                          # n 2^(s-1) >= 2^24
    assert seg(ws=0) == 7
    assert seg(wsb=100) == 7

    def qsum(m=2, w0=0, scheme=1, s=8, out=fake, st=0, ws=None, wsb=0):
        return lib.gq_quantize_sum(vp(fake), 0, m, 64, w0, vp(fake), scheme, s, 1, 1,
                                   vp(out) if out else None, st, vp(ws) if ws else None, wsb, None)
    assert qsum(w0=-1) == 1
    assert qsum(w0=(1 << 31) - 1) == 1
    assert qsum(out=0) == 1
    assert qsum(out=fake + 4) == 1
    assert qsum(st=2) == 1
    assert qsum(s=0) == 2
    assert qsum(m=2, s=24) == 3
    assert qsum(m=2, s=8, st=1) == 3        # int8 sums: 2 workers x 2^7 units exceed 127
    assert qsum(m=8, scheme=0, s=16, st=1) == 3
    assert qsum(ws=fake, wsb=8) == 7
    assert lib.gq_dequantize_sums(vp(fake), 1, vp(fake), 0, 15, 9, 64, vp(fake), 0, None) == 3
    assert lib.gq_dequantize_sums(vp(fake), 2, vp(fake), 0, 15, 2, 64, vp(fake), 0, None) == 1

    assert lib.gq_norm_partial(vp(fake), 0, 2, 64, 2, 0, vp(fake), vp(fake), ws_bytes, None) == 2
    assert lib.gq_norm_partial(vp(fake), 0, 2, 64, 0, 2, vp(fake), vp(fake), ws_bytes, None) == 2
    assert lib.gq_norm_partial(vp(fake), 0, 2, 64, 2, 2, None, vp(fake), ws_bytes, None) == 1
    assert lib.gq_norm_partial(vp(fake), 0, 2, 64, 2, 2, vp(fake), vp(fake), 8, None) == 7
    assert lib.gq_norm_finish(vp(fake), 2, 0, vp(fake), None) == 2
    assert lib.gq_norm_finish(None, 2, 2, vp(fake), None) == 1
    assert lib.gq_norm_finish(vp(fake), 3, 2, vp(fake), None) == 1

    assert lib.gq_dequantize_to(vp(fake), vp(fake), 1, 8, 2, 64, vp(fake), 3, None) == 1
    assert lib.gq_dequantize_to(vp(fake), vp(fake), 1, 8, 2, 64, vp(fake + 2), 1, None) == 1
    assert lib.gq_allreduce_mean_to(vp(fake), 0, 2, 64, 0, 0, 1, 8, 1, 1, vp(fake), -1, None,
                                    None, vp(fake), ws_bytes, None) == 1
