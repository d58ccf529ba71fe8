"""GPU parity of the single-launch form of the fused call (resident_kernel).

A fused call without a code output on 16-byte aligned rows whose matrix fits in the GPU's shared
memory runs as one cooperative launch: each block holds its columns on chip, the blocks combine
the norm at a grid barrier and quantise from shared memory.  Checked here:
  * the launch count query agrees with the size rule at its boundary (from the SM count);
  * against the two-pass path (the same call with a code output): the max-form norms and the
    outputs bit for bit; for the (2, 2) and (inf, 2) norms the norm within 1e-6 and the outputs
    bit for bit against gq_allreduce_mean_with_norm given the single launch's own norm;
  * against the oracle: the norm (exact for the max forms, 1e-6 for the sums) and, with the
    kernel's fp32 norm, every output within 1e-6 N;
  * shapes: one worker, odd worker counts, ragged last groups (fp32, d = 4 mod 8), more workers
    than the (2, inf) fast column sums take, the largest slice that fits; both dtypes, both
    schemes, all four norms, 16-bit outputs;
  * zero and non-finite inputs, and many calls in a row on one workspace (the barrier words
    return to their rest state), with the status word read after each;
  * two problems on two streams at once, each with its own workspace.
"""
import numpy as np
import pytest

from gpu_common import EXP, INF, LINEAR, gq_module, to_device, to_host
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu

ORDERS = [(2, 2), (2, INF), (INF, 2), (INF, INF)]
TILE = 200 * 1024


@pytest.fixture(scope="module")
def gq():
    return gq_module()


@pytest.fixture(scope="module")
def oracle_mod():
    from oracle import gq_oracle
    gq_oracle.lib()
    return gq_oracle


def _sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


def _fits(n, d, elt):
    gpb = -(-(-(-d // 8)) // _sms())
    return n * gpb * 8 * elt <= TILE


def _largest_d(n, elt):
    """The largest d (a multiple of 8) whose n x d matrix takes the single launch."""
    gpb = TILE // (n * 8 * elt)
    return gpb * _sms() * 8


def test_launch_count_rule(gq):
    import torch
    for n, elt, dt in ((8, 4, torch.float32), (3, 2, torch.bfloat16), (1, 4, torch.float32)):
        dmax = _largest_d(n, elt)
        assert gq.gq_fused_launches(dt, n, dmax) == 1
        assert gq.gq_fused_launches(dt, n, dmax + 8) == 2
        assert gq.gq_fused_launches(dt, n, dmax, with_codes=True) == 2
        assert _fits(n, dmax, elt) and not _fits(n, dmax + 8, elt)


def _check(gq, oracle_mod, x, q, p, scheme, s, seed=3, step=5, windows=None):
    import torch
    n, d = x.shape
    dt = x.dtype
    assert gq.gq_fused_launches(dt, n, d) == 1
    ws = gq.gq_workspace()
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    out = gq.gq_allreduce_mean(x, q, p, scheme, s, seed, step, norm=norm, ws=ws)
    # the two-pass path: the same call with a code output
    codes = torch.empty(gq.gq_code_bytes(scheme, s, n, d), dtype=torch.uint8, device="cuda")
    norm2 = torch.empty(1, dtype=torch.float32, device="cuda")
    out2 = gq.gq_allreduce_mean(x, q, p, scheme, s, seed, step, norm=norm2, codes=codes, ws=ws)
    ref = gq.gq_allreduce_mean_with_norm(x, norm, scheme, s, seed, step)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    n32, n2 = float(norm.item()), float(norm2.item())
    if (q, p) in ((INF, INF), (2, INF)):  # maxima: the same norm whatever the split
        assert n32 == n2
        assert torch.equal(out, out2)
    assert n32 == pytest.approx(n2, rel=1e-6)
    assert torch.equal(out, ref)

    xh = to_host(x)
    want = oracle_mod.global_norm(xh, q, p)
    if (q, p) == (INF, INF):
        assert n32 == float(np.float32(want))
    else:
        assert n32 == pytest.approx(want, rel=1e-6)
    out_h = out.cpu().numpy().astype(np.float64)
    spans = windows or [(0, d)]
    for j0, j1 in spans:
        rc_codes, rc = oracle_mod.quantize(xh, n32, scheme, s, seed, step, j0, j1)
        assert rc == 0
        want_out, rc = oracle_mod.dequantize(oracle_mod.reduce_codes(rc_codes, scheme, s), n32,
                                             scheme, s, n)
        assert rc == 0
        assert np.abs(out_h[j0:j1] - want_out).max() <= 1e-6 * n32


SMALL = [(1, 8), (3, 16), (4, 65_536), (5, 1000), (7, 4100), (2, 8196), (16, 3000), (65, 512),
         (300, 1024)]


@pytest.mark.parametrize("n,d", SMALL)
@pytest.mark.parametrize("q,p", ORDERS)
@pytest.mark.parametrize("scheme,s", [(LINEAR, 15), (EXP, 8), (LINEAR, 127), (EXP, 4)])
def test_single_launch_fp32(gq, oracle_mod, n, d, q, p, scheme, s):
    x = to_device(workloads.host_inputs("normal", n, d, seed=n * 31 + d))
    _check(gq, oracle_mod, x, q, p, scheme, s)


@pytest.mark.parametrize("n,d", [(1, 8), (3, 16), (4, 65_536), (5, 1000), (33, 1024), (8, 8200)])
@pytest.mark.parametrize("q,p", ORDERS)
@pytest.mark.parametrize("scheme,s", [(LINEAR, 7), (EXP, 8)])
def test_single_launch_bf16(gq, oracle_mod, n, d, q, p, scheme, s):
    x = to_device(workloads.host_inputs("student_t3", n, d, seed=n + d, dtype="bf16"))
    _check(gq, oracle_mod, x, q, p, scheme, s)


@pytest.mark.parametrize("n,dtype", [(8, "f32"), (3, "bf16"), (1, "f32")])
@pytest.mark.parametrize("q,p", [(INF, INF), (2, INF), (2, 2)])
def test_largest_slice(gq, oracle_mod, n, dtype, q, p):
    """The largest matrix that takes the single launch, checked on sampled windows."""
    elt = 4 if dtype == "f32" else 2
    d = _largest_d(n, elt)
    if dtype == "f32":
        d -= 4  # a ragged last group in the last block
    x = workloads.device_inputs("normal", n, d, seed=d % 1000, dtype=dtype)
    rng = np.random.default_rng(d)
    starts = sorted({0, d - 777} | {int(v) // 8 * 8 for v in rng.integers(0, d - 777, size=3)})
    _check(gq, oracle_mod, x, q, p, LINEAR, 127, windows=[(a, a + 777) for a in starts])


@pytest.mark.parametrize("out16", ["bf16", "f16"])
def test_single_launch_16bit_out(gq, out16):
    import torch
    t16 = {"bf16": torch.bfloat16, "f16": torch.float16}[out16]
    x = workloads.device_inputs("normal", 6, 40_000, seed=4)
    assert gq.gq_fused_launches(x.dtype, 6, 40_000) == 1
    o32 = gq.gq_allreduce_mean(x, 2, 2, EXP, 8, 1, 2)
    o16 = gq.gq_allreduce_mean(x, 2, 2, EXP, 8, 1, 2, out_dtype=t16)
    torch.cuda.synchronize()
    assert torch.equal(o16.cpu(), o32.cpu().to(t16))


def test_zero_and_nonfinite(gq):
    import torch
    ws = gq.gq_workspace()
    n, d = 4, 4096
    out = torch.full((d,), 3.0, device="cuda")
    norm = torch.empty(1, device="cuda")
    for q, p in ORDERS:
        gq.gq_allreduce_mean(torch.zeros((n, d), device="cuda"), q, p, LINEAR, 7, 1, 1, out=out,
                             norm=norm, ws=ws)
        torch.cuda.synchronize()
        assert not out.any() and norm.item() == 0.0
        assert gq.gq_get_status(ws) == 0
        x = torch.randn((n, d), device="cuda")
        x[1, 1234] = float("inf") if q == p else float("nan")
        out.fill_(3.0)
        gq.gq_allreduce_mean(x, q, p, EXP, 4, 1, 1, out=out, norm=norm, ws=ws)
        torch.cuda.synchronize()
        assert not out.any() and not np.isfinite(norm.item())
        assert gq.gq_get_status(ws) == 4


def test_many_calls_one_workspace(gq):
    """The grid barrier's words return to rest after every call: 200 calls in a row on one
    workspace, mixed sizes and norms, each equal to its first result."""
    import torch
    ws = gq.gq_workspace()
    xs = [workloads.device_inputs("normal", n, d, seed=n) for n, d in ((4, 65_536), (1, 8),
                                                                         (8, 300_000))]
    first = {}
    for it in range(200):
        k = it % 3
        q = (2, INF)[it % 2]
        out = gq.gq_allreduce_mean(xs[k], q, q, LINEAR, 15, 1, 7, ws=ws)
        key = (k, q)
        if key in first:
            assert torch.equal(out, first[key])
        else:
            first[key] = out
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0


def test_two_streams_two_workspaces(gq):
    """Single launches of two problems on two streams at once (each with its own workspace)
    give the results of the same calls made one after the other; neither wait runs out."""
    import torch
    xa = workloads.device_inputs("normal", 4, 65_536, seed=11)
    xb = workloads.device_inputs("normal", 8, 300_000, seed=12)
    assert gq.gq_fused_launches(xa.dtype, 4, 65_536) == 1
    assert gq.gq_fused_launches(xb.dtype, 8, 300_000) == 1
    wa, wb = gq.gq_workspace(), gq.gq_workspace()
    ref_a = gq.gq_allreduce_mean(xa, 2, 2, LINEAR, 15, 1, 3, ws=wa)
    ref_b = gq.gq_allreduce_mean(xb, INF, INF, EXP, 8, 2, 4, ws=wb)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    outs_a, outs_b = [], []
    for _ in range(20):
        with torch.cuda.stream(sa):
            outs_a.append(gq.gq_allreduce_mean(xa, 2, 2, LINEAR, 15, 1, 3, ws=wa, stream=sa))
        with torch.cuda.stream(sb):
            outs_b.append(gq.gq_allreduce_mean(xb, INF, INF, EXP, 8, 2, 4, ws=wb, stream=sb))
    torch.cuda.synchronize()
    assert gq.gq_get_status(wa) == 0 and gq.gq_get_status(wb) == 0
    for oa, ob in zip(outs_a, outs_b):
        assert torch.equal(oa, ref_a)
        assert torch.equal(ob, ref_b)
