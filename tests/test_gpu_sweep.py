"""GPU parity on the sweep grid (n in {2..64} x d in {2^20..2^28}, fp32 N(0,1), Global-L_7 and
Global-E_4 with int4 codes, q = p = 2), in the launch configuration bench.py times (the fused
call).  At these sizes the oracle checks sampled column windows (first, last, seeded interior):
codes bit-exact and out within 1e-6 N, both sides deciding with the GPU's fp32 norm; the norm
itself against the oracle's over the whole matrix to relative 1e-6 (the oracle runs on chunks of
columns copied to the host, in threads, and the chunks' squared norms are added in fp64).  The
grid's corners and the largest point (64 x 2^28, 68.7 GB) run; the rest of the grid is covered
by bench.py --measure sweep.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from gpu_common import EXP, LINEAR, gq_module, unpack_codes
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu

POINTS = [(2, 2**20), (64, 2**20), (2, 2**28), (16, 2**24), (64, 2**28)]
WINDOW = 1003


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
    starts = {0, d - WINDOW}
    while len(starts) < 4:
        starts.add(int(rng.integers(0, d - WINDOW)) // 32 * 32)
    return sorted((s0, s0 + WINDOW) for s0 in starts)


def _oracle_l2_norm(oracle_mod, x):
    """The oracle's (2, 2) norm of the device matrix x over chunks of at most 2^28 elements:
    sqrt of the sum of the chunks' squared norms (fp64)."""
    n, d = x.shape
    w = max(32, (1 << 28) // n // 32 * 32)
    threads = max(1, min(16, os.cpu_count() or 1))
    starts = list(range(0, d, w))
    parts = []
    with ThreadPoolExecutor(threads) as ex:
        for b in range(0, len(starts), threads):  # at most `threads` chunks on the host at once
            chunks = [np.ascontiguousarray(x[:, j:j + w].cpu().numpy())
                      for j in starts[b:b + threads]]
            parts += list(ex.map(lambda c: oracle_mod.global_norm(c, 2, 2), chunks))
            del chunks
    return float(np.sqrt(sum(v * v for v in parts)))


@pytest.mark.parametrize("n,d", POINTS)
def test_sweep_point(gq, oracle_mod, n, d):
    import torch
    x = workloads.device_inputs("normal", n, d, seed=0)
    want_norm = _oracle_l2_norm(oracle_mod, x)
    ws = gq.gq_workspace()
    for scheme, s in workloads.SWEEP_SCHEMES:
        norm = torch.empty(1, dtype=torch.float32, device="cuda")
        out = gq.gq_allreduce_mean(x, 2, 2, scheme, s, 1, 0, norm=norm, ws=ws)
        codes = gq.gq_quantize(x, norm, scheme, s, 1, 0)
        torch.cuda.synchronize()
        assert gq.gq_get_status(ws) == 0
        norm32 = float(norm.item())
        assert norm32 == pytest.approx(want_norm, rel=1e-6)
        bits = gq.gq_code_bits(scheme, s)
        assert bits == 4
        pitch = gq.gq_code_pitch(d)
        cview = codes.view(n, pitch // 2)
        for j0, j1 in _windows(d, seed=n * 7 + d % 97):
            xw = np.ascontiguousarray(x[:, j0:j1].cpu().numpy())  # the window's columns alone
            ref_codes, rc = oracle_mod.quantize_cols(xw, j0, norm32, scheme, s, 1, 0)
            assert rc == 0
            ref_out, rc = oracle_mod.dequantize(oracle_mod.reduce_codes(ref_codes, scheme, s),
                                                norm32, scheme, s, n)
            assert rc == 0
            a0, a1 = j0 // 32 * 32, (j1 + 31) // 32 * 32
            win = unpack_codes(cview[:, a0 // 2:a1 // 2].contiguous().cpu().numpy().ravel(),
                               scheme, s, n, a1 - a0, check_padding=False)
            np.testing.assert_array_equal(win[:, j0 - a0:j1 - a0], ref_codes)
            got = out[j0:j1].cpu().numpy().astype(np.float64)
            assert np.abs(got - ref_out).max() <= 1e-6 * norm32
        del codes, out
    del x
    torch.cuda.empty_cache()
