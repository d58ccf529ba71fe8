"""Helpers for the GPU parity tests: build/load the library, move inputs, unpack codes.

Unpacking follows the documented code layout (include/gq.h): signed level indices, int8 when
s > 7 else two's-complement int4 nibbles with element 2m in the low nibble of byte m, rows of
round_up(d, 32) elements.
"""
import numpy as np
import pytest

LINEAR, EXP = 0, 1
INF = 0


def gq_module():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from allreduce_compatible_gradient_gb300 import _build

    _build.build_library()
    import allreduce_compatible_gradient_gb300 as gq

    gq.lib()
    return gq


def code_bits(scheme, s):
    return 4 if s <= 7 else 8


def pitch(d):
    return (d + 31) // 32 * 32


def unpack_codes(codes_u8: np.ndarray, scheme, s, n, d, check_padding=True) -> np.ndarray:
    P = pitch(d)
    if code_bits(scheme, s) == 8:
        full = codes_u8.view(np.int8).reshape(n, P)
    else:
        b = codes_u8.reshape(n, P // 2)
        lo = (b & 0xF).astype(np.int16)
        hi = (b >> 4).astype(np.int16)
        full = np.empty((n, P), dtype=np.int16)
        full[:, 0::2] = (lo ^ 8) - 8
        full[:, 1::2] = (hi ^ 8) - 8
        full = full.astype(np.int8)
    if check_padding:
        assert not full[:, d:].any(), "padding codes must be zero"
    return np.ascontiguousarray(full[:, :d])


def to_device(x: np.ndarray):
    import torch

    if x.dtype == np.uint16:  # bf16 bit patterns
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(x).cuda()


def to_host(t) -> np.ndarray:
    import torch

    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()
