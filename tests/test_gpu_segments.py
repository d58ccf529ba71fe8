"""GPU parity of the segmented form gq_allreduce_mean_segments (per layer / per bucket).

Each segment l is its own n x d_l problem with its own norm and the random stream of step
(step << 16) | l.  Checked against the oracle segment by segment (codes decided with the GPU's
fp32 norm, which must itself match the oracle's: exactly for the max norm, relative 1e-6 for the
l2 forms; out within 1e-6 * N), and for the max norm bit for bit against one gq_allreduce_mean
call per segment.  Sizes mix single columns, ragged tails and multi-block segments; more than
256 segments exercise the chunked launches; the ResNet-50 layer list runs at full size.
"""
import numpy as np
import pytest

from gpu_common import EXP, INF, LINEAR, gq_module, to_host
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu

ORDERS = [(2, 2), (2, INF), (INF, 2), (INF, INF)]
MIXED = [1, 3, 17, 4099, 1000, 65536 + 24, 8, 2053, 31, 300_001]


@pytest.fixture(scope="module")
def gq():
    return gq_module()


@pytest.fixture(scope="module")
def oracle_mod():
    from oracle import gq_oracle
    gq_oracle.lib()
    return gq_oracle


def _check_segment(oracle_mod, xh, norm32, q, p, scheme, s, seed, step, got, j=None):
    want_norm = oracle_mod.global_norm(xh, q, p)
    if (q, p) == (INF, INF):
        assert norm32 == float(np.float32(want_norm))
    else:
        assert norm32 == pytest.approx(want_norm, rel=1e-6)
    j0, j1 = (0, xh.shape[1]) if j is None else j
    codes, rc = oracle_mod.quantize(xh, norm32, scheme, s, seed, step, j0, j1)
    assert rc == 0
    want, rc = oracle_mod.dequantize(oracle_mod.reduce_codes(codes, scheme, s), norm32, scheme, s,
                                     xh.shape[0])
    assert rc == 0
    err = np.abs(got[j0:j1].astype(np.float64) - want).max() if j1 > j0 else 0.0
    assert err <= 1e-6 * norm32


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("q,p", ORDERS)
@pytest.mark.parametrize("scheme,s", [(LINEAR, 7), (EXP, 8)])
def test_segments_match_oracle(gq, oracle_mod, dtype, q, p, scheme, s):
    import torch
    n, seed, step = 5, 41, 7
    segs = workloads.segment_tensors(n, MIXED, dtype=dtype, seed=3)
    norms = torch.empty(len(segs), dtype=torch.float32, device="cuda")
    outs = gq.gq_allreduce_mean_segments(segs, q, p, scheme, s, seed, step, norms=norms)
    torch.cuda.synchronize()
    nh = norms.cpu().numpy()
    for l, (x, out) in enumerate(zip(segs, outs)):
        _check_segment(oracle_mod, to_host(x), float(nh[l]), q, p, scheme, s, seed,
                       (step << 16) | l, out.cpu().numpy())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scheme,s", [(LINEAR, 15), (EXP, 4)])
def test_segments_equal_single_calls(gq, dtype, scheme, s):
    import torch
    n, seed, step = 8, 9, 123
    segs = workloads.segment_tensors(n, MIXED, dtype=dtype, seed=4)
    outs = gq.gq_allreduce_mean_segments(segs, INF, INF, scheme, s, seed, step)
    ws = gq.gq_workspace()
    for l, (x, out) in enumerate(zip(segs, outs)):
        ref = gq.gq_allreduce_mean(x, INF, INF, scheme, s, seed, step * 65536 + l, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), l


def test_many_segments_chunked(gq, oracle_mod):
    import torch
    rng = np.random.default_rng(5)
    sizes = [int(v) for v in rng.integers(1, 3000, size=600)]
    n, seed, step = 3, 2, 1
    segs = workloads.segment_tensors(n, sizes, seed=6)
    norms = torch.empty(len(segs), dtype=torch.float32, device="cuda")
    outs = gq.gq_allreduce_mean_segments(segs, 2, 2, EXP, 8, seed, step, norms=norms)
    torch.cuda.synchronize()
    nh = norms.cpu().numpy()
    for l in list(range(0, 600, 37)) + [255, 256, 257, 511, 512, 599]:
        _check_segment(oracle_mod, to_host(segs[l]), float(nh[l]), 2, 2, EXP, 8, seed,
                       (step << 16) | l, outs[l].cpu().numpy())


def test_zero_and_nonfinite_segments(gq):
    import torch
    segs = workloads.segment_tensors(4, [100, 200, 300], seed=1)
    segs[1].zero_()
    segs[2][1, 7] = float("nan")
    ws = gq.gq_workspace()
    norms = torch.empty(3, dtype=torch.float32, device="cuda")
    outs = gq.gq_allreduce_mean_segments(segs, INF, INF, LINEAR, 7, 0, 0, norms=norms, ws=ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(outs[0]) > 0
    assert torch.count_nonzero(outs[1]) == 0 and norms[1].item() == 0.0
    assert torch.count_nonzero(outs[2]) == 0 and np.isnan(norms[2].item())
    assert gq.gq_get_status(ws) == 4  # the non-finite norm is recorded


def test_segment_argument_errors(gq):
    import torch
    a = torch.ones(2, 8, device="cuda")
    b = torch.ones(3, 8, device="cuda")
    with pytest.raises(ValueError):
        gq.gq_allreduce_mean_segments([a, b], INF, INF, EXP, 8, 0, 0)
    with pytest.raises(gq.GQError):
        gq.gq_allreduce_mean_segments([a], INF, INF, EXP, 8, 0, 1 << 48)
    with pytest.raises(gq.GQError):
        gq.gq_allreduce_mean_segments([a, torch.ones(64, device="cuda")[1:33].view(2, 16)],
                                      INF, INF, EXP, 8, 0, 0)  # unaligned segment


def test_resnet50_layers_full_size(gq, oracle_mod):
    """The 161 ResNet-50 parameter tensors as segments, 8 workers: every segment's norm, and
    sampled column windows of the largest and of a spread of small ones."""
    import torch
    sizes = workloads.resnet50_layer_sizes()
    n, seed, step = 8, 1, 3
    segs = workloads.segment_tensors(n, sizes, seed=8)
    norms = torch.empty(len(segs), dtype=torch.float32, device="cuda")
    outs = gq.gq_allreduce_mean_segments(segs, INF, INF, LINEAR, 127, seed, step, norms=norms)
    torch.cuda.synchronize()
    nh = norms.cpu().numpy()
    big = int(np.argmax(sizes))
    for l in sorted(set(range(0, 161, 16)) | {big, 160}):
        xh = to_host(segs[l])
        d = sizes[l]
        win = (max(0, d - 4099), d) if d > 8192 else None
        _check_segment(oracle_mod, xh, float(nh[l]), INF, INF, LINEAR, 127, seed,
                       (step << 16) | l, outs[l].cpu().numpy(), j=win)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scheme,s", [(LINEAR, 127), (EXP, 8)])
def test_segments_bulk_copy_path(gq, dtype, scheme, s):
    """Enough 3840-column chunks for the segmented bulk-copy kernel, with a ragged last group,
    an unaligned segment (its groups all by direct loads), tiny segments and 5 workers: every
    segment equals its own gq_allreduce_mean call bit for bit (max norm)."""
    import torch
    sizes = [700_004, 300_001, 1_000_000, 8, 3, 65_544] if dtype == "f32" else \
        [700_008, 300_004, 1_000_000, 8, 3, 65_544]
    n, seed, step = 5, 3, 11
    segs = workloads.segment_tensors(n, sizes, dtype=dtype, seed=12)
    ws = gq.gq_workspace()
    norms = torch.empty(len(segs), dtype=torch.float32, device="cuda")
    outs = gq.gq_allreduce_mean_segments(segs, INF, INF, scheme, s, seed, step, norms=norms, ws=ws)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    for l, (x, out) in enumerate(zip(segs, outs)):
        ref = gq.gq_allreduce_mean(x, INF, INF, scheme, s, seed, step * 65536 + l, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), l
        assert norms[l].item() == float(gq.gq_global_norm(x, INF, INF).item())
