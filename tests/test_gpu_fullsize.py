"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times.

For each workload the gradients are generated on the GPU (seeded) and the fused gq_allreduce_mean
runs exactly as bench.py calls it (same arguments, no code output).  The oracle then checks that
call's own results:
  * the norm over the whole matrix: the max forms exactly (for p = inf the oracle's norm is the
    maximum of its per-column values, computed over column chunks in parallel threads), the l2
    forms to relative 1e-6 of the oracle's fp64 norm;
  * with the GPU's fp32 norm given to the oracle (the rounding decisions are a function of that
    norm), the dequantised mean: the integer code sums read back from it (out = fp32(scale S),
    exact for |S| < 2^23) equal the oracle's bit for bit, and every element is within 1e-6 N.
    For the three workloads up to 880 M elements this covers every coordinate (the oracle runs
    over column chunks in threads: it is plain C without shared state); for the 5.6 G-element
    BERT-large workload, 256 windows (first, last with the ragged tail, and seeded ones);
  * the same call with a code output: codes equal the oracle's bit for bit on the same columns.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from gpu_common import gq_module, to_host, unpack_codes
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu

WHOLE_LIMIT = 1_000_000_000   # n * d up to which every coordinate is checked
WINDOW = 4096
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def gq():
    return gq_module()


def _scale(N32, scheme, s, n):
    if scheme == 0:
        return float(np.float32(float(N32) / (n * s)))
    return float(np.float32(np.ldexp(float(N32), -(s - 1)) / n))


def _chunks(d, whole, seed):
    """Column ranges to check: all of [0, d) in pieces, or windows."""
    if whole:
        step = max(32, -(-d // (8 * THREADS)) // 32 * 32)
        return [(j, min(d, j + step)) for j in range(0, d, step)]
    rng = np.random.default_rng(seed)
    starts = {0, max(0, d - WINDOW - 3)}
    while len(starts) < 256:
        starts.add(int(rng.integers(0, max(1, d - WINDOW))) // 32 * 32)
    return sorted((s0, min(d, s0 + WINDOW + 3)) for s0 in starts)


def _oracle_norm(oracle, xh, q, p):
    if p != 0:
        return oracle.global_norm(xh, q, p)
    # p = inf: the maximum over coordinates of the per-coordinate q-norms, so chunks of columns
    # combine by a maximum exactly as the whole-matrix call would
    d = xh.shape[1]
    parts = _chunks(d, True, 0)

    def one(r):
        return oracle.global_norm(np.ascontiguousarray(xh[:, r[0]:r[1]]), q, p)
    with ThreadPoolExecutor(THREADS) as ex:
        vals = list(ex.map(one, parts))
    return max(vals)


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_full_size(gq, oracle, name):
    import torch

    cfg = workloads.CONFIGS[name]
    n, d = cfg["n"], cfg["d"]
    sc, s, q, p, seed, step = cfg["scheme"], cfg["s"], cfg["q"], cfg["p"], cfg["seed"], cfg["step"]
    x = workloads.device_inputs(cfg["dist"], n, d, seed=cfg["input_seed"], dtype=cfg["dtype"])
    out = torch.empty(d, dtype=torch.float32, device="cuda")
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = gq.gq_workspace()
    # the bench call
    gq.gq_allreduce_mean(x, q, p, sc, s, seed, step, out=out, norm=norm, ws=ws)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    # the same call with a code output (same norm kernel, so the same norm)
    codes = torch.empty(gq.gq_code_bytes(sc, s, n, d), dtype=torch.uint8, device="cuda")
    norm_c = torch.empty(1, dtype=torch.float32, device="cuda")
    gq.gq_allreduce_mean(x, q, p, sc, s, seed, step, norm=norm_c, codes=codes, ws=ws,
                         out=torch.empty(d, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0

    xh = to_host(x)
    del x
    torch.cuda.empty_cache()
    N32 = np.float32(norm.item())
    want64 = _oracle_norm(oracle, xh, q, p)
    if (q, p) == (0, 0):
        assert N32 == np.float32(want64)
    else:
        assert float(N32) == pytest.approx(want64, rel=1e-6)
    Nc = np.float32(norm_c.item())
    out_h = out.cpu().numpy()
    bits = gq.gq_code_bits(sc, s)
    pitch = gq.gq_code_pitch(d)
    codes_h = codes.cpu().numpy().reshape(n, pitch * bits // 8)
    sc_out = _scale(N32, sc, s, n)
    whole = n * d <= WHOLE_LIMIT

    def check(r):
        j0, j1 = r
        xw = np.ascontiguousarray(xh[:, j0:j1])
        ref_codes, rc = oracle.quantize_cols(xw, j0, N32, sc, s, seed, step)
        assert rc == 0
        ref_sums = oracle.reduce_codes(ref_codes, sc, s)
        ref_out, rc = oracle.dequantize(ref_sums, N32, sc, s, n)
        got = out_h[j0:j1].astype(np.float64)
        sums = np.rint(got / sc_out).astype(np.int64) if sc_out else np.zeros_like(ref_sums)
        bad_sums = int((sums != ref_sums).sum())
        err = float(np.abs(got - ref_out).max())
        if Nc != N32:  # the code call took the two-pass form, the bench call the single launch
            ref_codes, _ = oracle.quantize_cols(xw, j0, Nc, sc, s, seed, step)
        a0, a1 = j0 // 32 * 32, min(pitch, (j1 + 31) // 32 * 32)
        win = unpack_codes(np.ascontiguousarray(codes_h[:, a0 * bits // 8:a1 * bits // 8]).ravel(),
                           sc, s, n, a1 - a0, check_padding=False)
        bad_codes = int((win[:, j0 - a0:j1 - a0] != ref_codes).sum())
        return j0, bad_sums, err, bad_codes

    with ThreadPoolExecutor(THREADS) as ex:
        results = list(ex.map(check, _chunks(d, whole, seed=d)))
    if Nc != N32:  # only the single-launch form splits an l2 sum differently
        assert float(Nc) == pytest.approx(want64, rel=1e-6)
    for j0, bad_sums, err, bad_codes in results:
        assert bad_sums == 0, (j0, bad_sums)
        assert err <= 1e-6 * float(N32), (j0, err)
        assert bad_codes == 0, (j0, bad_codes)
    # padding codes past d are zero
    if pitch > d:
        tail = unpack_codes(np.ascontiguousarray(codes_h[:, (pitch - 32) * bits // 8:]).ravel(),
                            sc, s, n, 32, check_padding=False)
        assert not tail[:, d - (pitch - 32):].any()


@pytest.mark.parametrize("dtype,scheme,s", [("f32", 0, 127), ("bf16", 1, 8)])
def test_columns_past_2_31(gq, oracle, dtype, scheme, s):
    """One worker with d = 2^31 + 2^20 + 4 columns (8.6 GB fp32): column indices and Philox
    counters past 2^31 (word 0 = j / 8 past 2^28), a ragged tail, the bulk-copy kernel's largest
    chunk numbers.  The max norm against the oracle's (over column chunks in threads), sampled
    windows (first, around 2^31, last) against the oracle."""
    import torch
    # a ragged last group (d % 8 != 0) on 16-byte aligned rows: 2^31 + 2^20 + 4 (fp32); bf16
    # rows take the direct-load path here (d % 8 != 0)
    d = 2**31 + 2**20 + 4
    x = workloads.device_inputs("normal", 1, d, seed=31, dtype=dtype)
    ws = gq.gq_workspace()
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    out = gq.gq_allreduce_mean(x, 0, 0, scheme, s, 7, 3, norm=norm, ws=ws)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    norm32 = float(norm.item())
    assert np.float32(norm32) == np.float32(_oracle_norm(oracle, to_host(x), 0, 0))
    for j0 in (0, 2**31 - 512, 2**31 + 2**20 - 1000, d - 1003):
        j1 = min(d, j0 + 1003)
        xw = to_host(x[:, j0:j1].contiguous())
        codes, rc = oracle.quantize_cols(xw, j0, norm32, scheme, s, 7, 3)
        assert rc == 0
        want, rc = oracle.dequantize(oracle.reduce_codes(codes, scheme, s), norm32, scheme, s, 1)
        assert rc == 0
        got = out[j0:j1].cpu().numpy().astype(np.float64)
        assert np.abs(got - want).max() <= 1e-6 * norm32, j0
    del x, out
    torch.cuda.empty_cache()
