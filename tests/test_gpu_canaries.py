"""Guard bands around every output buffer (the memory checker is closed on this machine; these tests
and the debug build stand in for it).

Each output (means in every output type, codes of both widths, integer sums of both types, norms,
rank partials, segment outputs, re-rounded codes, workspaces) is placed between two 4 KB bands of
a known byte pattern, starting exactly at the buffer's logical end, so that a single byte written
past d, past the code pitch, past a segment or before the start is seen.  Every entry point runs
on ragged and aligned sizes and through each of its kernels (direct loads, bulk copies, the
compacting consumer, zero-row skipping, the single launch, the segmented kernels, the fixed
scratch of the allocation-free call).  After each call the bands must be intact.

When the suite runs against the debug build (GQ_LIBRARY pointing at libgq_debug.so, as
tests/test_gpu_debug_build.py does), every call must also leave the debug word at 0: no store or
bulk copy outside its buffer's logical extent.
"""
import ctypes
import os

import numpy as np
import pytest

from gpu_common import gq_module

pytestmark = pytest.mark.gpu

G = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module")
def gq():
    return gq_module()


class Guarded:
    """count elements of dtype between two guard bands (the tail band starts at the logical
    end, so a write past it is caught even when it stays inside the allocation's padding)."""

    def __init__(self, count, dtype):
        import torch
        elt = torch.empty((), dtype=dtype).element_size()
        self.nbytes = count * elt
        self.buf = torch.full((G + (self.nbytes + 15) // 16 * 16 + G,), PATTERN,
                              dtype=torch.uint8, device="cuda")
        self.t = self.buf[G:G + self.nbytes].view(dtype)

    def check(self, what):
        h = self.buf.cpu().numpy()
        head_bad = np.flatnonzero(h[:G] != PATTERN)
        tail_bad = np.flatnonzero(h[G + self.nbytes:] != PATTERN)
        assert len(head_bad) == 0, "%s: %d bytes written before the buffer" % (what, len(head_bad))
        assert len(tail_bad) == 0, "%s: %d bytes written past the end (first at +%d)" % (
            what, len(tail_bad), int(tail_bad[0]))


def _done(gq, bufs, what):
    import torch
    torch.cuda.synchronize()
    for b in bufs:
        b.check(what)
    st = gq.gq_debug_status()
    if os.environ.get("GQ_EXPECT_DEBUG"):
        assert st == 0, "%s: bounds check failed at line %d" % (what, st)
    else:
        assert st in (-1, 0)


def _x(n, d, dtype, dist="normal", seed=1):
    from allreduce_compatible_gradient_gb300 import workloads
    if dtype == "bf16" and dist == "normal":
        dist = "student_t3"
    return workloads.device_inputs(dist, n, d, seed=seed, dtype=dtype)


def _ws(gq):
    import torch
    w = Guarded(gq.gq_workspace_bytes(), torch.uint8)
    w.t.zero_()
    return w


FUSED = [
    # n, d, dtype, q, p, scheme, s, out dtype, codes
    (3, 1003, "f32", 0, 0, 0, 7, "f32", True),          # direct loads, ragged, int4
    (3, 1003, "bf16", 2, 2, 1, 8, "bf16", True),        # direct, bf16 rows not aligned
    (4, 65_536, "f32", 2, 2, 0, 15, "f16", False),      # single launch
    (4, 65_528, "bf16", 2, 0, 1, 4, "f32", False),      # single launch, ragged slices
    (8, 600_004, "f32", 0, 0, 0, 127, "f32", True),     # bulk copies, ragged last group
    (8, 600_004, "f32", 2, 2, 1, 8, "bf16", False),     # compacting consumer
    (1, 700_003, "f32", 2, 0, 1, 4, "f32", True),       # one worker, unaligned rows
    (6, 1_200_008, "bf16", 0, 2, 0, 7, "f16", False),   # compacting consumer, bf16
    (5, 1_048_576, "f32", 2, 0, 1, 4, "f32", True),     # zero blocks: rows skipped
    (2, 1_048_576, "f32", 2, 2, 0, 7, "f32", False),    # two workers: stages of two rows
    (2, 800_000, "bf16", 0, 0, 1, 4, "bf16", True),     # two workers, codes
]


@pytest.mark.parametrize("n,d,dtype,q,p,scheme,s,od,with_codes", FUSED)
def test_fused_and_unfused(gq, n, d, dtype, q, p, scheme, s, od, with_codes):
    import torch
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
    x = _x(n, d, dtype, "laplace_block_sparse" if n == 5 else "normal")
    ws = _ws(gq)
    out = Guarded(d, tdt[od])
    norm = Guarded(1, torch.float32)
    codes = Guarded(gq.gq_code_bytes(scheme, s, n, d), torch.uint8) if with_codes else None
    gq.gq_allreduce_mean(x, q, p, scheme, s, 3, 4, out=out.t, norm=norm.t,
                         codes=codes.t if codes else None, ws=ws.t)
    _done(gq, [b for b in (out, norm, codes, ws) if b], "gq_allreduce_mean")
    assert gq.gq_get_status(ws.t) == 0
    # the unfused chain into guarded buffers
    norm2 = Guarded(1, torch.float32)
    gq.gq_global_norm(x, q, p, norm=norm2.t, ws=ws.t)
    c2 = Guarded(gq.gq_code_bytes(scheme, s, n, d), torch.uint8)
    gq.gq_quantize(x, norm2.t, scheme, s, 3, 4, codes=c2.t)
    sums = Guarded(d, torch.int32)
    gq.gq_reduce_codes(c2.t, scheme, s, n, d, sums=sums.t)
    out2 = Guarded(d, tdt[od])
    gq.gq_dequantize_to(sums.t, norm2.t, scheme, s, n, out=out2.t)
    out3 = Guarded(d, torch.float32)
    c3 = Guarded(gq.gq_code_bytes(scheme, s, n, d), torch.uint8)
    gq.gq_allreduce_mean_with_norm(x, norm2.t, scheme, s, 3, 4, out=out3.t, codes=c3.t)
    _done(gq, [norm2, c2, sums, out2, out3, c3, ws], "unfused chain")


@pytest.mark.parametrize("big", [False, True])
def test_segments(gq, big):
    import torch
    from allreduce_compatible_gradient_gb300 import workloads
    sizes = [517, 65_536, 3, 300_001, 4096] if not big else [400_000, 1003, 263_168, 310_004]
    segs = workloads.segment_tensors(4, sizes, seed=2)
    ws = _ws(gq)
    for od in (torch.float32, torch.bfloat16):
        outs = [Guarded(sz, od) for sz in sizes]
        norms = Guarded(len(sizes), torch.float32)
        gq.gq_allreduce_mean_segments(segs, 2, 0, 1, 4, 1, 2, outs=[o.t for o in outs],
                                      norms=norms.t, ws=ws.t)
        _done(gq, outs + [norms, ws], "gq_allreduce_mean_segments")


@pytest.mark.parametrize("m,d,with_ws", [(1, 700_000, True), (2, 600_004, True), (3, 1003, False)])
def test_rank_shares(gq, m, d, with_ws):
    import torch
    x = _x(m, d, "f32")
    ws = _ws(gq) if with_ws else None
    part = Guarded(1, torch.float64)
    gq.gq_norm_partial(x, 2, 2, part=part.t, ws=(ws or _ws(gq)).t)
    norm = Guarded(1, torch.float32)
    gq.gq_norm_finish(part.t, 2, 2, norm=norm.t)
    bufs = [part, norm] + ([ws] if ws else [])
    for scheme, s, sdt in ((0, 15, torch.int32), (1, 2, torch.int8)):
        sums = Guarded(d, sdt)
        gq.gq_quantize_sum(x, norm.t, scheme, s, 1, 2, worker0=4, sums=sums.t,
                           ws=ws.t if ws else None)
        out = Guarded(d, torch.float16)
        gq.gq_dequantize_sums(sums.t, norm.t, scheme, s, m + 4, out=out.t)
        bufs += [sums, out]
    for bits, s in ((8, 8), (4, 3)):
        codes = Guarded(m * gq.gq_code_pitch(d) * bits // 8, torch.uint8)
        gq.gq_quantize_codes(x, norm.t, 1, s, 1, 2, worker0=4, code_bits=bits, codes=codes.t,
                             ws=ws.t if ws else None)
        bufs.append(codes)
    _done(gq, bufs, "rank shares")


@pytest.mark.parametrize("n,d", [(3, 1003), (8, 65_541), (5, 16)])
def test_exp_allreduce(gq, n, d):
    import torch
    x = _x(n, d, "f32")
    norm = gq.gq_global_norm(x, 0, 0)
    codes = gq.gq_quantize(x, norm, 1, 8, 1, 2)
    a = gq.gq_quantize_codes(x[:1].clone(), norm, 1, 8, 1, 2, worker0=0, code_bits=8)[:d]
    b = gq.gq_quantize_codes(x[1:2].clone(), norm, 1, 8, 1, 2, worker0=1, code_bits=8)[:d]
    comb = Guarded(d, torch.int8)
    gq.gq_exp_combine(a.view(torch.int8).contiguous(), b.view(torch.int8).contiguous(), 1, 2,
                      gq.gq_exp_tree_stream(1, 0), out=comb.t)
    bufs = [comb]
    for order in (0, 1):
        out = Guarded(d, torch.float32)
        root = Guarded(d, torch.int8)
        gq.gq_exp_allreduce(codes, 8, n, d, order, norm, 1, 2, out=out.t, root_codes=root.t)
        deq = Guarded(d, torch.bfloat16)
        gq.gq_exp_dequantize(root.t, norm, 8, n, out=deq.t)
        bufs += [out, root, deq]
    _done(gq, bufs, "Global-E re-rounding allreduce")


@pytest.mark.parametrize("n,d,with_codes", [(8, 1 << 20, True), (8, 300_007, False),
                                            (4, 65_536, False)])
def test_noalloc(gq, n, d, with_codes):
    import torch
    x = _x(n, d, "f32")
    out = Guarded(d, torch.float32)
    norm = Guarded(1, torch.float32)
    codes = Guarded(gq.gq_code_bytes(0, 127, n, d), torch.uint8) if with_codes else None
    rc = gq.lib().gq_allreduce_mean_noalloc(
        ctypes.c_void_p(x.data_ptr()), 0, n, d, 2, 2, 0, 127, 1, 2,
        ctypes.c_void_p(out.t.data_ptr()), ctypes.c_void_p(norm.t.data_ptr()),
        ctypes.c_void_p(codes.t.data_ptr()) if codes else None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    _done(gq, [b for b in (out, norm, codes) if b], "gq_allreduce_mean_noalloc")
