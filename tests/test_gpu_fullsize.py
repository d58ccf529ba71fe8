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
