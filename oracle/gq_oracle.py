"""ctypes loader and numpy wrappers for the C oracle in gq_oracle.c.

TEST INFRASTRUCTURE ONLY: imported by the test suite, by ``__graft_entry__.smoke()`` and by the
CPU-baseline leg of ``bench.py``.  The library under ``allreduce_compatible_gradient_gb300``
never imports this module and shares no code with it.

The oracle is plain single-threaded C (see gq_oracle.c for the method and its citations).  This
module compiles it with gcc the first time it is needed (or when the source is newer than the
shared object) and exposes numpy-level helpers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gq_oracle.c")
_LIB = os.path.join(_HERE, "libgq_oracle.so")
_lock = threading.Lock()
_lib = None

# Same meanings as the library's values, written out independently.
OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_NONFINITE = 0, 1, 2, 4
F32, BF16 = 0, 1
LINEAR, EXP = 0, 1
INF = 0  # norm order code for l-infinity


def build(force: bool = False) -> str:
    """Compile gq_oracle.c into libgq_oracle.so next to it; return the path."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + ".tmp.%d" % os.getpid()
            cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                   "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        # GQ_ORACLE_LIB points the pin tests at a deliberately broken copy of the oracle
        # (tests/test_oracle_mutants.py), to show that the pins catch planted mistakes.
        path = os.environ.get("GQ_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        i64, u64, u32, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32
        vp = ctypes.c_void_p
        L.gqo_abi_version.restype = ctypes.c_int
        L.gqo_philox4x32_10.argtypes = [vp, vp, vp]
        L.gqo_philox4x32_10.restype = None
        L.gqo_philox_word.argtypes = [u64, u64, i64, i64]
        L.gqo_philox_word.restype = u32
        L.gqo_philox_words.argtypes = [u64, u64, i64, i64, i64, vp]
        L.gqo_philox_words.restype = ctypes.c_int
        L.gqo_global_norm.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_int]
        L.gqo_global_norm.restype = ctypes.c_double
        L.gqo_level_split.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(i32), ctypes.POINTER(u32)]
        L.gqo_level_split.restype = ctypes.c_int
        L.gqo_quantize.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, ctypes.c_float,
                                   ctypes.c_int, ctypes.c_int, u64, u64, vp]
        L.gqo_quantize.restype = ctypes.c_int
        L.gqo_quantize_cols.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, ctypes.c_float,
                                        ctypes.c_int, ctypes.c_int, u64, u64, vp]
        L.gqo_quantize_cols.restype = ctypes.c_int
        L.gqo_level_split_u16.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_int,
                                          ctypes.c_int, ctypes.POINTER(i32), ctypes.POINTER(u32)]
        L.gqo_level_split_u16.restype = ctypes.c_int
        L.gqo_quantize_u16_cols.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, ctypes.c_float,
                                            ctypes.c_int, ctypes.c_int, u64, u64, vp]
        L.gqo_quantize_u16_cols.restype = ctypes.c_int
        L.gqo_reduce_codes.argtypes = [vp, ctypes.c_int, ctypes.c_int, i64, i64, vp]
        L.gqo_reduce_codes.restype = ctypes.c_int
        L.gqo_dequantize.argtypes = [vp, ctypes.c_float, ctypes.c_int, ctypes.c_int, i64, i64, vp]
        L.gqo_dequantize.restype = ctypes.c_int
        L.gqo_allreduce_mean.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, u64, u64, i64, i64,
                                         ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_float), vp, vp, vp]
        L.gqo_allreduce_mean.restype = ctypes.c_int
        L.gqo_exp_split_units.argtypes = [i64, ctypes.POINTER(i32), ctypes.POINTER(u32)]
        L.gqo_exp_split_units.restype = ctypes.c_int
        L.gqo_exp_tree_stream.argtypes = [ctypes.c_int, i64]
        L.gqo_exp_tree_stream.restype = i64
        L.gqo_exp_ring_stream.argtypes = [i64, i64]
        L.gqo_exp_ring_stream.restype = i64
        L.gqo_exp_combine.argtypes = [vp, vp, i64, i64, u64, u64, i64, vp]
        L.gqo_exp_combine.restype = ctypes.c_int
        L.gqo_exp_tree_allreduce.argtypes = [vp, i64, i64, i64, u64, u64, vp]
        L.gqo_exp_tree_allreduce.restype = ctypes.c_int
        L.gqo_exp_ring_allreduce.argtypes = [vp, i64, i64, i64, i64, u64, u64, vp]
        L.gqo_exp_ring_allreduce.restype = ctypes.c_int
        _lib = L
    return _lib


# ----------------------------------------------------------------------------------------------
# numpy-level helpers
# ----------------------------------------------------------------------------------------------

def _grads(x: np.ndarray):
    """(pointer, dtype code, n, d) for a C-contiguous n x d float32 or bf16-as-uint16 array."""
    if x.ndim != 2:
        raise ValueError("gradients must be an n x d array")
    if not x.flags.c_contiguous:
        raise ValueError("gradients must be C-contiguous")
    if x.dtype == np.float32:
        code = F32
    elif x.dtype == np.uint16:
        code = BF16  # bf16 bit patterns
    else:
        raise TypeError("gradients must be float32 or bf16 bits (uint16)")
    return x.ctypes.data, code, x.shape[0], x.shape[1]


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    lib().gqo_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def philox_word(seed: int, step: int, i: int, j: int) -> int:
    return int(lib().gqo_philox_word(seed, step, i, j))


def philox_words(seed: int, step: int, i: int, j0: int, w: int) -> np.ndarray:
    """The words philox_word(seed, step, i, j) for j = j0 .. j0 + w - 1 (uint32 array)."""
    out = np.zeros(w, dtype=np.uint32)
    rc = lib().gqo_philox_words(seed, step, i, j0, w, out.ctypes.data)
    if rc != OK:
        raise ValueError("gqo_philox_words returned %d" % rc)
    return out


def global_norm(x: np.ndarray, q: int, p: int) -> float:
    ptr, code, n, d = _grads(x)
    return float(lib().gqo_global_norm(ptr, code, n, d, q, p))


def level_split(absx: float, norm: float, scheme: int, s: int):
    lo = ctypes.c_int32()
    T = ctypes.c_uint32()
    rc = lib().gqo_level_split(absx, norm, scheme, s, ctypes.byref(lo), ctypes.byref(T))
    if rc != OK:
        raise ValueError("gqo_level_split returned %d" % rc)
    return int(lo.value), int(T.value)


def quantize(x: np.ndarray, norm32: float, scheme: int, s: int, seed: int, step: int,
             j0: int = 0, j1: int | None = None):
    """Signed level-index codes, n x (j1 - j0) int8, and the return code."""
    ptr, code, n, d = _grads(x)
    j1 = d if j1 is None else j1
    codes = np.zeros((n, j1 - j0), dtype=np.int8)
    rc = lib().gqo_quantize(ptr, code, n, d, j0, j1, float(norm32), scheme, s, seed, step,
                            codes.ctypes.data)
    return codes, rc


def quantize_cols(xw: np.ndarray, j0: int, norm32: float, scheme: int, s: int, seed: int,
                  step: int):
    """Codes of the columns j0 .. j0 + w - 1 of a larger matrix, given only those columns (an
    n x w array): the random words are keyed by the columns' global indices."""
    ptr, code, n, w = _grads(xw)
    codes = np.zeros((n, w), dtype=np.int8)
    rc = lib().gqo_quantize_cols(ptr, code, n, w, j0, w, float(norm32), scheme, s, seed, step,
                                 codes.ctypes.data)
    return codes, rc


USE_EXACT = 8  # gqo_level_split_u16: the norm is out of the mode's range, the exact mode applies


def level_split_u16(absx: float, norm: float, scheme: int, s: int):
    """(lower level, F) of the 16-bit-uniform mode, or None where the exact mode applies."""
    lo = ctypes.c_int32()
    F = ctypes.c_uint32()
    rc = lib().gqo_level_split_u16(absx, norm, scheme, s, ctypes.byref(lo), ctypes.byref(F))
    if rc == USE_EXACT:
        return None
    if rc != OK:
        raise ValueError("gqo_level_split_u16 returned %d" % rc)
    return int(lo.value), int(F.value)


def quantize_u16(x: np.ndarray, norm32: float, scheme: int, s: int, seed: int, step: int,
                 j0: int = 0, j1: int | None = None):
    """Codes of the 16-bit-uniform mode for the window [j0, j1) of x, and the return code."""
    ptr, code, n, d = _grads(x)
    j1 = d if j1 is None else j1
    esize = 2 if code == BF16 else 4
    codes = np.zeros((n, j1 - j0), dtype=np.int8)
    rc = lib().gqo_quantize_u16_cols(ptr + j0 * esize, code, n, d, j0, j1 - j0, float(norm32),
                                     scheme, s, seed, step, codes.ctypes.data)
    return codes, rc


def quantize_u16_cols(xw: np.ndarray, j0: int, norm32: float, scheme: int, s: int, seed: int,
                      step: int):
    """quantize_u16 on the columns j0 .. j0 + w - 1 of a larger matrix, given alone."""
    ptr, code, n, w = _grads(xw)
    codes = np.zeros((n, w), dtype=np.int8)
    rc = lib().gqo_quantize_u16_cols(ptr, code, n, w, j0, w, float(norm32), scheme, s, seed,
                                     step, codes.ctypes.data)
    return codes, rc


def reduce_codes(codes: np.ndarray, scheme: int, s: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    n, w = codes.shape
    sums = np.zeros(w, dtype=np.int64)
    rc = lib().gqo_reduce_codes(codes.ctypes.data, scheme, s, n, w, sums.ctypes.data)
    if rc != OK:
        raise ValueError("gqo_reduce_codes returned %d" % rc)
    return sums


def dequantize(sums: np.ndarray, norm32: float, scheme: int, s: int, n: int):
    sums = np.ascontiguousarray(sums, dtype=np.int64)
    out = np.zeros(sums.shape[0], dtype=np.float64)
    rc = lib().gqo_dequantize(sums.ctypes.data, float(norm32), scheme, s, n, sums.shape[0],
                              out.ctypes.data)
    return out, rc


def allreduce_mean(x: np.ndarray, q: int, p: int, scheme: int, s: int, seed: int, step: int,
                   j0: int = 0, j1: int | None = None) -> dict:
    """Whole pipeline on window [j0, j1): dict with norm64, norm32, codes, sums, out, rc."""
    ptr, code, n, d = _grads(x)
    j1 = d if j1 is None else j1
    w = j1 - j0
    n64 = ctypes.c_double()
    n32 = ctypes.c_float()
    codes = np.zeros((n, w), dtype=np.int8)
    sums = np.zeros(w, dtype=np.int64)
    out = np.zeros(w, dtype=np.float64)
    rc = lib().gqo_allreduce_mean(ptr, code, n, d, q, p, scheme, s, seed, step, j0, j1,
                                  ctypes.byref(n64), ctypes.byref(n32), codes.ctypes.data,
                                  sums.ctypes.data, out.ctypes.data)
    return {"norm64": n64.value, "norm32": np.float32(n32.value), "codes": codes, "sums": sums,
            "out": out, "rc": rc}


# ---- Global-E allreduce with re-rounding at every hop ------------------------------------------

def exp_units(codes) -> np.ndarray:
    """Value of extended Global-E codes in units of 2^-(s-1): sign * 2^(|k|-1), 0 for k = 0."""
    c = np.asarray(codes, dtype=np.int64)
    k = np.abs(c)
    u = np.where(k > 0, np.left_shift(np.int64(1), np.maximum(k - 1, 0)), 0)
    return np.sign(c) * u


def exp_split_units(t: int):
    lo = ctypes.c_int32()
    T = ctypes.c_uint32()
    lib().gqo_exp_split_units(int(t), ctypes.byref(lo), ctypes.byref(T))
    return int(lo.value), int(T.value)


def exp_tree_stream(level: int, m: int) -> int:
    return int(lib().gqo_exp_tree_stream(level, m))


def exp_ring_stream(h: int, c: int) -> int:
    return int(lib().gqo_exp_ring_stream(h, c))


def exp_combine(a, b, seed: int, step: int, stream_id: int, j0: int = 0) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.int8)
    b = np.ascontiguousarray(b, dtype=np.int8)
    out = np.zeros(a.shape[0], dtype=np.int8)
    rc = lib().gqo_exp_combine(a.ctypes.data, b.ctypes.data, a.shape[0], j0, seed, step,
                               stream_id, out.ctypes.data)
    if rc != OK:
        raise ValueError("gqo_exp_combine returned %d" % rc)
    return out


def exp_tree_allreduce(codes, seed: int, step: int, j0: int = 0) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    n, w = codes.shape
    root = np.zeros(w, dtype=np.int8)
    rc = lib().gqo_exp_tree_allreduce(codes.ctypes.data, n, w, j0, seed, step, root.ctypes.data)
    if rc != OK:
        raise ValueError("gqo_exp_tree_allreduce returned %d" % rc)
    return root


def exp_ring_allreduce(codes, d: int, seed: int, step: int, j0: int = 0) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    n, w = codes.shape
    root = np.zeros(w, dtype=np.int8)
    rc = lib().gqo_exp_ring_allreduce(codes.ctypes.data, n, d, w, j0, seed, step,
                                      root.ctypes.data)
    if rc != OK:
        raise ValueError("gqo_exp_ring_allreduce returned %d" % rc)
    return root
