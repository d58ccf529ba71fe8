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
    assert gq.gq_workspace_bytes(8, 10**9) == 256 + 8 * 4096 + 2 * 4 * 256
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
