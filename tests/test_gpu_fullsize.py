"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times.

For each workload: the gradients are generated on the GPU (seeded), the fused gq_allreduce_mean
runs exactly as in bench.py (same call, same arguments), and the oracle checks
  * the norm over the whole matrix (the max norm exactly; l2 forms to relative 1e-6);
  * sampled column windows (first, last with the ragged tail, and seeded interior windows):
    codes bit-exact and the dequantised mean within 1e-6 * N, using the same fp32 norm on both
    sides (the oracle's norm is fed to the GPU if the two fp32 norms differ).
"""
import numpy as np
import pytest

from gpu_common import gq_module, to_host, unpack_codes
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu

WINDOW = 1024


def _windows(d, k=6, seed=0):
    rng = np.random.default_rng(seed)
    starts = {0, max(0, d - WINDOW - 3)}
    while len(starts) < k:
        starts.add(int(rng.integers(0, max(1, d - WINDOW))))
    return sorted((s, min(d, s + WINDOW + 3)) for s in starts)


@pytest.fixture(scope="module")
def gq():
    return gq_module()


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_full_size(gq, name):
    import torch
    from oracle import gq_oracle as oracle

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

    xh = to_host(x)
    want64 = oracle.global_norm(xh, q, p)
    want32 = np.float32(want64)
    got32 = np.float32(norm.item())
    if (q, p) == (0, 0):
        assert got32 == want32
    else:
        assert float(got32) == pytest.approx(want64, rel=1e-6)

    # same fp32 norm on both sides for the element-wise comparison
    if got32 != want32:
        norm_t = torch.tensor([float(want32)], device="cuda")
        out = gq.gq_allreduce_mean_with_norm(x, norm_t, sc, s, seed, step)
    codes = torch.empty(gq.gq_code_bytes(sc, s, n, d), dtype=torch.uint8, device="cuda")
    gq.gq_allreduce_mean_with_norm(x, torch.tensor([float(want32)], device="cuda"), sc, s, seed,
                                   step, codes=codes)
    out_h = out.cpu().numpy().astype(np.float64)
    bits = gq.gq_code_bits(sc, s)
    pitch = gq.gq_code_pitch(d)
    row_bytes = pitch * bits // 8
    codes_h = codes.cpu().numpy().reshape(n, row_bytes)
    for j0, j1 in _windows(d, seed=d):
        ref_codes, rc = oracle.quantize(xh, want32, sc, s, seed, step, j0, j1)
        assert rc == 0
        ref_sums = oracle.reduce_codes(ref_codes, sc, s)
        ref_out, rc = oracle.dequantize(ref_sums, want32, sc, s, n)
        # unpack the GPU codes of this window (windows start on a multiple of 32 columns)
        a0 = j0 // 32 * 32
        a1 = min(pitch, (j1 + 31) // 32 * 32)
        b0, b1 = a0 * bits // 8, a1 * bits // 8
        win = unpack_codes(np.ascontiguousarray(codes_h[:, b0:b1]).ravel(), sc, s, n, a1 - a0,
                           check_padding=False)
        np.testing.assert_array_equal(win[:, j0 - a0:j1 - a0], ref_codes)
        err = np.abs(out_h[j0:j1] - ref_out).max()
        assert err <= 1e-6 * float(want32), (j0, err)
    # padding codes past d are zero
    if pitch > d:
        tail = unpack_codes(np.ascontiguousarray(codes_h[:, (pitch - 32) * bits // 8:]).ravel(),
                            sc, s, n, 32, check_padding=False)
        assert not tail[:, d - (pitch - 32):].any()


@pytest.mark.parametrize("dtype,scheme,s", [("f32", 0, 127), ("bf16", 1, 8)])
def test_columns_past_2_31(gq, dtype, scheme, s):
    """One worker with d = 2^31 + 2^20 + 5 columns (8.6 GB fp32): column indices and Philox
    counters past 2^31 (word 0 = j / 8 past 2^28), a ragged tail, the bulk-copy kernel's largest
    chunk numbers.  The max norm against a library reduction, sampled windows (first, around
    2^31, last) against the oracle."""
    import torch
    from oracle import gq_oracle as oracle
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
    assert norm32 == float(x.abs().max().float().item())
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
