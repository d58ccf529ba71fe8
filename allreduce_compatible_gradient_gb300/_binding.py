"""ctypes binding over libgq.so (include/gq.h).  Argument marshalling only: every step of the
pipeline runs in the library's CUDA kernels.  Output tensors that the caller does not pass are
allocated here with torch (the library itself allocates nothing)."""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# GQ_LIBRARY selects another build of the same library (the debug build with bounds checks)
_LIB_PATH = os.environ.get("GQ_LIBRARY") or os.path.join(_PKG, "libgq.so")

F32, BF16, F16 = 0, 1, 2
SUM_I32, SUM_I8 = 0, 1
LINEAR, EXP = 0, 1
ROUND_U16 = 16  # added to a scheme: the 16-bit-uniform rounding mode
NORM_INF, NORM_L2 = 0, 2
ORDER_TREE, ORDER_RING = 0, 1

_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libgq.so (built by ``__graft_entry__.build()``); fail loudly if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError("libgq.so is not built (%s): run `python -c \"import __graft_entry__ as g; "
                          "g.build()\"` first; there is no fallback path" % _LIB_PATH)
    L = ctypes.CDLL(_LIB_PATH)
    i64, u64, vp, ci = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int
    sz = ctypes.c_size_t
    sig = {
        "gq_abi_version": (ci, []),
        "gq_workspace_bytes": (sz, [i64, i64]),
        "gq_workspace_init": (ci, [vp, sz, vp]),
        "gq_code_bits": (ci, [ci, ci]),
        "gq_code_pitch": (i64, [i64]),
        "gq_fused_launches": (ci, [ci, i64, i64, ci]),
        "gq_norm_blocks": (i64, [ci, i64, i64, ci, ci]),
        "gq_noalloc_max_blocks": (i64, []),
        "gq_code_bytes": (sz, [ci, ci, i64, i64]),
        "gq_global_norm": (ci, [vp, ci, i64, i64, ci, ci, vp, vp, sz, vp]),
        "gq_quantize": (ci, [vp, ci, i64, i64, vp, ci, ci, u64, u64, vp, vp]),
        "gq_quantize_ws": (ci, [vp, ci, i64, i64, vp, ci, ci, u64, u64, vp, vp, sz, vp]),
        "gq_reduce_codes": (ci, [vp, ci, ci, i64, i64, vp, vp]),
        "gq_dequantize": (ci, [vp, vp, ci, ci, i64, i64, vp, vp]),
        "gq_allreduce_mean": (ci, [vp, ci, i64, i64, ci, ci, ci, ci, u64, u64, vp, vp, vp, vp, sz,
                                   vp]),
        "gq_allreduce_mean_with_norm": (ci, [vp, ci, i64, i64, vp, ci, ci, u64, u64, vp, vp, vp]),
        "gq_allreduce_mean_with_norm_ws": (ci, [vp, ci, i64, i64, vp, ci, ci, u64, u64, vp, vp, vp,
                                                sz, vp]),
        "gq_allreduce_mean_noalloc": (ci, [vp, ci, i64, i64, ci, ci, ci, ci, u64, u64, vp, vp, vp,
                                           vp]),
        "gq_philox4x32_10": (ci, [vp, vp, i64, vp]),
        "gq_allreduce_mean_segments": (ci, [i64, vp, vp, ci, i64, ci, ci, ci, ci, u64, u64, vp,
                                            ci, vp, vp, sz, vp]),
        "gq_dequantize_to": (ci, [vp, vp, ci, ci, i64, i64, vp, ci, vp]),
        "gq_allreduce_mean_to": (ci, [vp, ci, i64, i64, ci, ci, ci, ci, u64, u64, vp, ci, vp, vp,
                                      vp, sz, vp]),
        "gq_norm_partial": (ci, [vp, ci, i64, i64, ci, ci, vp, vp, sz, vp]),
        "gq_norm_finish": (ci, [vp, ci, ci, vp, vp]),
        "gq_quantize_sum": (ci, [vp, ci, i64, i64, i64, vp, ci, ci, u64, u64, vp, ci, vp, sz, vp]),
        "gq_dequantize_sums": (ci, [vp, ci, vp, ci, ci, i64, i64, vp, ci, vp]),
        "gq_exp_tree_stream": (ctypes.c_uint32, [ci, i64]),
        "gq_exp_ring_stream": (ctypes.c_uint32, [i64, i64]),
        "gq_exp_combine": (ci, [vp, vp, i64, i64, u64, u64, ctypes.c_uint32, vp, vp]),
        "gq_exp_allreduce": (ci, [vp, ci, i64, i64, ci, vp, u64, u64, vp, vp, vp]),
        "gq_get_status": (ci, [vp, vp]),
        "gq_selftest_wait_timeout": (ci, [vp, sz, u64, vp, vp]),
        "gq_quantize_codes": (ci, [vp, ci, i64, i64, i64, vp, ci, ci, u64, u64, vp, ci, vp, sz, vp]),
        "gq_exp_dequantize": (ci, [vp, i64, vp, ci, i64, vp, ci, vp]),
        "gq_status_string": (ctypes.c_char_p, [ci]),
        "gq_debug_status": (ci, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


class GQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, gq_status_string(status), status))


def gq_status_string(status: int) -> str:
    return lib().gq_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != 0:
        raise GQError(status, where)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("gradients must be float32 or bfloat16, got %s" % t.dtype)


def _grads(t: torch.Tensor):
    if t.dim() != 2 or not t.is_cuda or not t.is_contiguous():
        raise ValueError("gradients must be a contiguous n x d CUDA tensor")
    return _dtype_code(t), t.shape[0], t.shape[1]


# ---- sizes ---------------------------------------------------------------------------------

def gq_abi_version() -> int:
    return lib().gq_abi_version()


def gq_workspace_bytes(n: int = 1, d: int = 1) -> int:
    return lib().gq_workspace_bytes(n, d)


def gq_code_bits(scheme: int, s: int) -> int:
    return lib().gq_code_bits(scheme, s)


def gq_code_pitch(d: int) -> int:
    return lib().gq_code_pitch(d)


def gq_fused_launches(dtype, n: int, d: int, with_codes: bool = False) -> int:
    """1 if gq_allreduce_mean runs as one launch for this problem, 2 if as two, 0 if invalid;
    dtype: torch.float32 / torch.bfloat16 or F32 / BF16."""
    code = {torch.float32: F32, torch.bfloat16: BF16}.get(dtype, dtype)
    return lib().gq_fused_launches(int(code), n, d, 1 if with_codes else 0)


def gq_debug_status() -> int:
    """The first failed bounds check of a debug build (its source line), 0 for none, -1 in a
    normal build."""
    return lib().gq_debug_status()


def gq_norm_blocks(dtype, n: int, d: int, q: int, p: int) -> int:
    """Blocks the norm step of an n x d problem launches on the current device (0 if invalid)."""
    code = {torch.float32: F32, torch.bfloat16: BF16}.get(dtype, dtype)
    return lib().gq_norm_blocks(int(code), n, d, q, p)


def gq_noalloc_max_blocks() -> int:
    """Most norm-step blocks gq_allreduce_mean_noalloc's fixed scratch holds."""
    return lib().gq_noalloc_max_blocks()


def gq_code_bytes(scheme: int, s: int, n: int, d: int) -> int:
    return lib().gq_code_bytes(scheme, s, n, d)


def gq_workspace(device=None, stream=None) -> torch.Tensor:
    """A zero-initialised workspace tensor (uint8) for the norm step."""
    nb = gq_workspace_bytes()
    ws = torch.empty(nb, dtype=torch.uint8, device=device or "cuda")
    _check(lib().gq_workspace_init(_p(ws), nb, _stream(stream)), "gq_workspace_init")
    return ws


# ---- the pipeline --------------------------------------------------------------------------

def gq_global_norm(grads, q, p, norm=None, ws=None, stream=None) -> torch.Tensor:
    dt, n, d = _grads(grads)
    norm = torch.empty(1, dtype=torch.float32, device=grads.device) if norm is None else norm
    ws = gq_workspace(grads.device, stream) if ws is None else ws
    _check(lib().gq_global_norm(_p(grads), dt, n, d, q, p, _p(norm), _p(ws), ws.numel(),
                                _stream(stream)), "gq_global_norm")
    return norm


def gq_quantize(grads, norm, scheme, s, seed, step, codes=None, ws=None,
                stream=None) -> torch.Tensor:
    """Step 2 with a supplied device norm; a workspace (ws) lets large problems take the
    bulk-copy kernel (gq_quantize_ws)."""
    dt, n, d = _grads(grads)
    if codes is None:
        codes = torch.empty(gq_code_bytes(scheme, s, n, d), dtype=torch.uint8, device=grads.device)
    if ws is None:
        _check(lib().gq_quantize(_p(grads), dt, n, d, _p(norm), scheme, s, seed, step, _p(codes),
                                 _stream(stream)), "gq_quantize")
    else:
        _check(lib().gq_quantize_ws(_p(grads), dt, n, d, _p(norm), scheme, s, seed, step,
                                    _p(codes), _p(ws), ws.numel(), _stream(stream)),
               "gq_quantize_ws")
    return codes


def gq_quantize_ws(grads, norm, scheme, s, seed, step, ws, codes=None,
                   stream=None) -> torch.Tensor:
    """gq_quantize with a workspace (the bulk-copy kernel for large problems)."""
    return gq_quantize(grads, norm, scheme, s, seed, step, codes=codes, ws=ws, stream=stream)


def gq_reduce_codes(codes, scheme, s, n, d, sums=None, stream=None) -> torch.Tensor:
    if sums is None:
        sums = torch.empty(d, dtype=torch.int32, device=codes.device)
    _check(lib().gq_reduce_codes(_p(codes), scheme, s, n, d, _p(sums), _stream(stream)),
           "gq_reduce_codes")
    return sums


_OUT_TYPES = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}


def _out_code(out: torch.Tensor) -> int:
    if out.dtype not in _OUT_TYPES or not out.is_cuda or not out.is_contiguous():
        raise TypeError("outputs must be contiguous float32, bfloat16 or float16 CUDA tensors")
    return _OUT_TYPES[out.dtype]


def gq_dequantize(sums, norm, scheme, s, n, out=None, stream=None,
                  out_dtype=torch.float32) -> torch.Tensor:
    """Dequantised mean into out (float32, bfloat16 or float16; a new tensor of out_dtype when
    out is None)."""
    d = sums.numel()
    if out is None:
        out = torch.empty(d, dtype=out_dtype, device=sums.device)
    _check(lib().gq_dequantize_to(_p(sums), _p(norm), scheme, s, n, d, _p(out), _out_code(out),
                                  _stream(stream)), "gq_dequantize_to")
    return out


def gq_allreduce_mean(grads, q, p, scheme, s, seed, step, out=None, norm=None, codes=None,
                      ws=None, stream=None, out_dtype=torch.float32) -> torch.Tensor:
    """Fused pipeline; out is float32, bfloat16 or float16 (a new tensor of out_dtype when
    None)."""
    dt, n, d = _grads(grads)
    if out is None:
        out = torch.empty(d, dtype=out_dtype, device=grads.device)
    ws = gq_workspace(grads.device, stream) if ws is None else ws
    _check(lib().gq_allreduce_mean_to(_p(grads), dt, n, d, q, p, scheme, s, seed, step, _p(out),
                                      _out_code(out), _p(norm), _p(codes), _p(ws), ws.numel(),
                                      _stream(stream)), "gq_allreduce_mean_to")
    return out


def gq_dequantize_to(sums, norm, scheme, s, n, out=None, out_dtype=torch.float32,
                     stream=None) -> torch.Tensor:
    """gq_dequantize with an explicit output type (float32, bfloat16 or float16)."""
    return gq_dequantize(sums, norm, scheme, s, n, out=out, stream=stream, out_dtype=out_dtype)


def gq_allreduce_mean_to(grads, q, p, scheme, s, seed, step, out=None, out_dtype=torch.float32,
                         norm=None, codes=None, ws=None, stream=None) -> torch.Tensor:
    """gq_allreduce_mean with an explicit output type (float32, bfloat16 or float16)."""
    return gq_allreduce_mean(grads, q, p, scheme, s, seed, step, out=out, norm=norm, codes=codes,
                             ws=ws, stream=stream, out_dtype=out_dtype)


def gq_allreduce_mean_with_norm(grads, norm, scheme, s, seed, step, out=None, codes=None,
                                ws=None, stream=None) -> torch.Tensor:
    """Steps 2-4 with a supplied device norm; a workspace (ws) lets large problems take the
    bulk-copy kernel (gq_allreduce_mean_with_norm_ws)."""
    dt, n, d = _grads(grads)
    if out is None:
        out = torch.empty(d, dtype=torch.float32, device=grads.device)
    if ws is None:
        _check(lib().gq_allreduce_mean_with_norm(_p(grads), dt, n, d, _p(norm), scheme, s, seed,
                                                 step, _p(out), _p(codes), _stream(stream)),
               "gq_allreduce_mean_with_norm")
    else:
        _check(lib().gq_allreduce_mean_with_norm_ws(_p(grads), dt, n, d, _p(norm), scheme, s,
                                                    seed, step, _p(out), _p(codes), _p(ws),
                                                    ws.numel(), _stream(stream)),
               "gq_allreduce_mean_with_norm_ws")
    return out


def gq_allreduce_mean_with_norm_ws(grads, norm, scheme, s, seed, step, ws, out=None, codes=None,
                                   stream=None) -> torch.Tensor:
    """gq_allreduce_mean_with_norm with a workspace (the bulk-copy kernel for large problems)."""
    return gq_allreduce_mean_with_norm(grads, norm, scheme, s, seed, step, out=out, codes=codes,
                                       ws=ws, stream=stream)


def gq_allreduce_mean_segments(grads, q, p, scheme, s, seed, step, outs=None, norms=None,
                               ws=None, stream=None, out_dtype=torch.float32):
    """Per-segment fused pipeline: grads is a list of n x d_l CUDA tensors (same dtype and n);
    returns the list of d_l outputs (all of one type: float32, bfloat16 or float16).  Segment l
    uses step (step << 16) | l."""
    grads = list(grads)
    if not grads:
        raise ValueError("no segments")
    dts = set()
    n = None
    for g in grads:
        dt, gn, _ = _grads(g)
        dts.add(dt)
        if n is not None and gn != n:
            raise ValueError("every segment needs the same number of workers")
        n = gn
    if len(dts) != 1:
        raise ValueError("every segment needs the same dtype")
    dev = grads[0].device
    if outs is None:
        outs = [torch.empty(g.shape[1], dtype=out_dtype, device=dev) for g in grads]
    if len(outs) != len(grads):
        raise ValueError("one output per segment")
    oc = {_out_code(o) for o in outs}
    if len(oc) != 1:
        raise ValueError("every segment output needs the same type")
    if ws is None:
        ws = gq_workspace(dev, stream)
    L = len(grads)
    gp = (ctypes.c_void_p * L)(*[g.data_ptr() for g in grads])
    dv = (ctypes.c_int64 * L)(*[g.shape[1] for g in grads])
    op = (ctypes.c_void_p * L)(*[o.data_ptr() for o in outs])
    _check(lib().gq_allreduce_mean_segments(L, gp, dv, dts.pop(), n, q, p, scheme, s, seed, step,
                                            op, oc.pop(), _p(norms), _p(ws), ws.numel(),
                                            _stream(stream)),
           "gq_allreduce_mean_segments")
    return outs


def gq_norm_partial(grads, q, p, part=None, ws=None, stream=None) -> torch.Tensor:
    """This rank's combinable share of the global norm (fp64: a sum of squares for q = p = 2, a
    maximum for q = p = inf)."""
    dt, m, d = _grads(grads)
    if part is None:
        part = torch.empty(1, dtype=torch.float64, device=grads.device)
    if ws is None:
        ws = gq_workspace(grads.device, stream)
    _check(lib().gq_norm_partial(_p(grads), dt, m, d, q, p, _p(part), _p(ws), ws.numel(),
                                 _stream(stream)), "gq_norm_partial")
    return part


def gq_norm_finish(part, q, p, norm=None, stream=None) -> torch.Tensor:
    """The fp32 norm from the ranks' combined partial."""
    if norm is None:
        norm = torch.empty(1, dtype=torch.float32, device=part.device)
    _check(lib().gq_norm_finish(_p(part), q, p, _p(norm), _stream(stream)), "gq_norm_finish")
    return norm


_SUM_TYPES = {torch.int32: SUM_I32, torch.int8: SUM_I8}


def gq_quantize_sum(grads, norm, scheme, s, seed, step, worker0=0, sums=None, ws=None,
                    stream=None, sum_dtype=torch.int32) -> torch.Tensor:
    """One rank's share of a multi-GPU allreduce: integer code sums of its rows (workers
    worker0 ..), int32 or int8, to be summed over ranks and dequantised with the total worker
    count.  ws (optional workspace) lets large problems take the bulk-copy kernel."""
    dt, m, d = _grads(grads)
    if sums is None:
        sums = torch.empty(d, dtype=sum_dtype, device=grads.device)
    if sums.dtype not in _SUM_TYPES:
        raise TypeError("sums must be int32 or int8")
    _check(lib().gq_quantize_sum(_p(grads), dt, m, d, worker0, _p(norm), scheme, s, seed, step,
                                 _p(sums), _SUM_TYPES[sums.dtype], _p(ws),
                                 0 if ws is None else ws.numel(), _stream(stream)),
           "gq_quantize_sum")
    return sums


def gq_dequantize_sums(sums, norm, scheme, s, n, out=None, stream=None,
                       out_dtype=torch.float32) -> torch.Tensor:
    """Dequantised mean from int32 or int8 sums over n workers."""
    if sums.dtype not in _SUM_TYPES:
        raise TypeError("sums must be int32 or int8")
    d = sums.numel()
    if out is None:
        out = torch.empty(d, dtype=out_dtype, device=sums.device)
    _check(lib().gq_dequantize_sums(_p(sums), _SUM_TYPES[sums.dtype], _p(norm), scheme, s, n, d,
                                    _p(out), _out_code(out), _stream(stream)),
           "gq_dequantize_sums")
    return out


def gq_allreduce_mean_noalloc(grads, q, p, scheme, s, seed, step, out, norm=None, codes=None,
                              stream=None) -> torch.Tensor:
    """gq_allreduce_mean for callers that cannot allocate: the library uses its own fixed device
    scratch instead of a workspace, so `out` (and `norm` / `codes` when wanted) must be passed in."""
    dt, n, d = _grads(grads)
    _check(lib().gq_allreduce_mean_noalloc(_p(grads), dt, n, d, q, p, scheme, s, seed, step,
                                           _p(out), _p(norm), _p(codes), _stream(stream)),
           "gq_allreduce_mean_noalloc")
    return out


def gq_philox4x32_10(ctr_key, out=None, stream=None) -> torch.Tensor:
    """ctr_key: count x 6 int32 tensor (counter words 0..3, key words 0..1, as bit patterns)."""
    count = ctr_key.shape[0]
    if out is None:
        out = torch.empty((count, 4), dtype=torch.int32, device=ctr_key.device)
    _check(lib().gq_philox4x32_10(_p(ctr_key), _p(out), count, _stream(stream)),
           "gq_philox4x32_10")
    return out


def gq_quantize_codes(grads, norm, scheme, s, seed, step, worker0=0, code_bits=8, codes=None,
                      ws=None, stream=None) -> torch.Tensor:
    """One rank's codes (m x pitch, int8 or int4-packed) with its worker offset."""
    dt, m, d = _grads(grads)
    if codes is None:
        codes = torch.empty(m * gq_code_pitch(d) * code_bits // 8, dtype=torch.uint8,
                            device=grads.device)
    _check(lib().gq_quantize_codes(_p(grads), dt, m, d, worker0, _p(norm), scheme, s, seed, step,
                                   _p(codes), code_bits, _p(ws), 0 if ws is None else ws.numel(),
                                   _stream(stream)), "gq_quantize_codes")
    return codes


def gq_exp_dequantize(codes, norm, s, n, d=None, out=None, stream=None,
                      out_dtype=torch.float32) -> torch.Tensor:
    """Mean from extended Global-E codes (int8) reduced over n workers."""
    d = codes.numel() if d is None else d
    if out is None:
        out = torch.empty(d, dtype=out_dtype, device=codes.device)
    _check(lib().gq_exp_dequantize(_p(codes), d, _p(norm), s, n, _p(out), _out_code(out),
                                   _stream(stream)), "gq_exp_dequantize")
    return out


def gq_selftest_wait_timeout(limit_ns: int, ws=None, stream=None):
    """Run the bounded-wait self-test: a wait that nothing completes gives up after limit_ns.
    Returns (status read from the workspace, nanoseconds waited)."""
    ws = gq_workspace(None, stream) if ws is None else ws
    elapsed = torch.zeros(1, dtype=torch.int64, device=ws.device)
    _check(lib().gq_selftest_wait_timeout(_p(ws), ws.numel(), limit_ns, _p(elapsed),
                                          _stream(stream)), "gq_selftest_wait_timeout")
    status = gq_get_status(ws, stream)
    return status, int(elapsed.item())


def gq_get_status(ws, stream=None) -> int:
    return lib().gq_get_status(_p(ws), _stream(stream))


# ---- Global-E allreduce with re-rounding at every hop ------------------------------------------

def gq_exp_tree_stream(level: int, m: int) -> int:
    return int(lib().gq_exp_tree_stream(level, m))


def gq_exp_ring_stream(h: int, c: int) -> int:
    return int(lib().gq_exp_ring_stream(h, c))


def gq_exp_combine(a, b, seed, step, stream_id, out=None, stream=None, j0=0) -> torch.Tensor:
    """One reduction step of the Global-E allreduce on int8 code vectors a, b whose element j is
    coordinate j0 + j of the whole vector (j0 a multiple of 8)."""
    d = a.numel()
    if out is None:
        out = torch.empty(d, dtype=torch.int8, device=a.device)
    _check(lib().gq_exp_combine(_p(a), _p(b), d, j0, seed, step, stream_id, _p(out),
                                _stream(stream)), "gq_exp_combine")
    return out


def gq_exp_allreduce(codes, s, n, d, order, norm, seed, step, out=None, root_codes=None,
                     stream=None) -> torch.Tensor:
    """Tree or ring Global-E allreduce of gq_quantize's code matrix, dequantised to out."""
    if out is None:
        out = torch.empty(d, dtype=torch.float32, device=codes.device)
    _check(lib().gq_exp_allreduce(_p(codes), s, n, d, order, _p(norm), seed, step, _p(out),
                                  _p(root_codes), _stream(stream)), "gq_exp_allreduce")
    return out
