"""GPU parity of the multi-rank pieces and of the DDP communication hook.

  * gq_quantize_sum: each rank's integer code sums (int32, or int8 when the total fits), with its
    worker offset, equal the oracle's sums over the same rows (bit-exact); summed over the ranks
    and dequantised (gq_dequantize_sums) they give gq_allreduce_mean_with_norm of the stacked
    matrix bit for bit, also at sizes that take the bulk-copy kernel;
  * gq_norm_partial + gq_norm_finish over row blocks combine to the global norm (exactly for the
    max norm, relative 1e-6 for the l2 norm);
  * the hook under DistributedDataParallel (NCCL, world size 1, one GPU): every bucket's result
    equals the oracle's pipeline on that bucket (n = 1, step = iteration * 2^16 + bucket index)
    within 1e-6 * N.
"""
import datetime
import socket

import numpy as np
import pytest

from gpu_common import EXP, INF, LINEAR, gq_module, to_device, to_host
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    return gq_module()


@pytest.fixture(scope="module")
def oracle_mod():
    from oracle import gq_oracle
    gq_oracle.lib()
    return gq_oracle


def _inputs(n, d, dtype, seed):
    dist = "student_t3" if dtype == "bf16" else "normal"
    return workloads.host_inputs(dist, n, d, seed=seed, dtype=dtype)


SPLITS = [(5, 1000, [2, 3]), (8, 4099, [1, 3, 4]), (3, 65536 + 24, [3]), (6, 2053, [1] * 6)]


def _units(scheme, s):
    return s if scheme == LINEAR else 1 << (s - 1)


@pytest.mark.parametrize("wire", ["i32", "i8"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,d,parts", SPLITS)
@pytest.mark.parametrize("scheme,s", [(LINEAR, 7), (LINEAR, 127), (EXP, 4), (EXP, 8)])
def test_quantize_sum_over_ranks(gq, oracle_mod, wire, dtype, n, d, parts, scheme, s):
    import torch
    if wire == "i8" and n * _units(scheme, s) > 127:
        pytest.skip("the sum over the workers does not fit int8")
    sum_dtype = torch.int8 if wire == "i8" else torch.int32
    x = _inputs(n, d, dtype, seed=7 * n + d)
    norm32 = np.float32(oracle_mod.global_norm(x, INF, INF))
    norm = torch.tensor([float(norm32)], device="cuda")
    seed, step = 1234 + s, 99
    xd = to_device(x)
    total = torch.zeros(d, dtype=torch.int32, device="cuda")
    codes, rc = oracle_mod.quantize(x, float(norm32), scheme, s, seed, step)
    assert rc == 0
    r0 = 0
    for m in parts:
        # each rank holds its rows in its own allocation (a row slice of an odd d is unaligned)
        got = gq.gq_quantize_sum(xd[r0:r0 + m].clone(), norm, scheme, s, seed, step, worker0=r0,
                                 sum_dtype=sum_dtype)
        assert got.dtype == sum_dtype
        want = oracle_mod.reduce_codes(codes[r0:r0 + m], scheme, s)
        np.testing.assert_array_equal(got.cpu().numpy().astype(np.int64), want)
        total += got.to(torch.int32)
        r0 += m
    out = gq.gq_dequantize_sums(total.to(sum_dtype), norm, scheme, s, n)
    ref = gq.gq_allreduce_mean_with_norm(xd, norm, scheme, s, seed, step)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


@pytest.mark.parametrize("dtype,d", [("f32", 700_004), ("bf16", 800_000)])
@pytest.mark.parametrize("scheme,s,wire", [(LINEAR, 15, "i8"), (EXP, 8, "i32"), (EXP, 4, "i8")])
def test_quantize_sum_bulk_copy_path(gq, oracle_mod, dtype, d, scheme, s, wire):
    """Ranks of 1, 2 and 1 workers at a size that takes the bulk-copy kernel (a single-worker
    rank uses its one-row form): sums against the oracle on windows, and the dequantised total
    equal to the single-GPU call."""
    import torch
    n, parts = 4, [1, 2, 1]
    sum_dtype = torch.int8 if wire == "i8" else torch.int32
    x = workloads.device_inputs("normal" if dtype == "f32" else "student_t3", n, d, seed=d,
                                dtype=dtype)
    norm = gq.gq_global_norm(x, INF, INF)
    ws = gq.gq_workspace()
    seed, step = 3, 4
    total = torch.zeros(d, dtype=torch.int32, device="cuda")
    sums = []
    r0 = 0
    for m in parts:
        got = gq.gq_quantize_sum(x[r0:r0 + m].clone(), norm, scheme, s, seed, step, worker0=r0,
                                 sum_dtype=sum_dtype, ws=ws)
        sums.append((r0, m, got))
        total += got.to(torch.int32)
        r0 += m
    out = gq.gq_dequantize_sums(total.to(sum_dtype), norm, scheme, s, n)
    ref = gq.gq_allreduce_mean_with_norm(x, norm, scheme, s, seed, step)
    torch.cuda.synchronize()
    assert gq.gq_get_status(ws) == 0
    assert torch.equal(out, ref)
    xh = to_host(x)
    norm32 = float(norm.item())
    for j0, j1 in [(0, 1000), (d // 2, d // 2 + 1000), (d - 1000, d)]:
        codes, rc = oracle_mod.quantize(xh, norm32, scheme, s, seed, step, j0, j1)
        assert rc == 0
        for r0, m, got in sums:
            want = oracle_mod.reduce_codes(codes[r0:r0 + m], scheme, s)
            np.testing.assert_array_equal(got[j0:j1].cpu().numpy().astype(np.int64), want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,d,parts", SPLITS)
@pytest.mark.parametrize("q", [2, INF])
def test_norm_partials_combine(gq, oracle_mod, dtype, n, d, parts, q):
    import torch
    x = _inputs(n, d, dtype, seed=11 * n + d)
    xd = to_device(x)
    ws = gq.gq_workspace()
    acc = None
    r0 = 0
    for m in parts:
        part = gq.gq_norm_partial(xd[r0:r0 + m].clone(), q, q, ws=ws).clone()
        acc = part if acc is None else (acc + part if q == 2 else torch.maximum(acc, part))
        r0 += m
    got = float(gq.gq_norm_finish(acc, q, q).item())
    want = oracle_mod.global_norm(x, q, q)
    if q == INF:
        assert got == float(np.float32(want))
        assert got == float(gq.gq_global_norm(xd, q, q).item())
    else:
        assert got == pytest.approx(want, rel=1e-6)


def test_norm_partial_refuses_mixed_orders(gq):
    import torch
    x = torch.ones(2, 8, device="cuda")
    for q, p in [(2, INF), (INF, 2)]:
        with pytest.raises(gq.GQError):
            gq.gq_norm_partial(x, q, p)
        with pytest.raises(gq.GQError):
            gq.gq_norm_finish(torch.ones(1, dtype=torch.float64, device="cuda"), q, p)


def test_quantize_sum_argument_errors(gq):
    import torch
    x = torch.ones(2, 8, device="cuda")
    norm = torch.ones(1, device="cuda")
    with pytest.raises(gq.GQError):
        gq.gq_quantize_sum(x, norm, EXP, 8, 0, 0, worker0=-1)
    with pytest.raises(gq.GQError):
        gq.gq_quantize_sum(x, norm, EXP, 8, 0, 0, worker0=(1 << 31) - 1)
    with pytest.raises(gq.GQError):  # 2 workers x 2^23 units reach 2^24
        gq.gq_quantize_sum(x, norm, EXP, 24, 0, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture(scope="module")
def nccl_group(gq):
    import torch.distributed as dist
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % _free_port(), rank=0,
                            world_size=1, timeout=datetime.timedelta(seconds=60))
    yield dist
    dist.destroy_process_group()


@pytest.mark.parametrize("dtype,scheme,s,q,reduce", [("f32", EXP, 8, INF, "sum"),
                                                     ("f32", LINEAR, 15, 2, "sum"),
                                                     ("bf16", EXP, 4, INF, "sum"),
                                                     ("f32", EXP, 8, INF, "tree"),
                                                     ("bf16", EXP, 6, 2, "ring")])
def test_ddp_hook_world_one(gq, oracle_mod, nccl_group, dtype, scheme, s, q, reduce):
    import torch
    from allreduce_compatible_gradient_gb300 import comm_hook

    class RecordingOps(comm_hook.LibraryOps):
        def __init__(self):
            super().__init__()
            self.norms = []

        def norm_finish(self, part, q, p):
            n = super().norm_finish(part, q, p)
            self.norms.append(n.clone())
            return n

    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(64, 512), torch.nn.Tanh(),
                                torch.nn.Linear(512, 512), torch.nn.Tanh(),
                                torch.nn.Linear(512, 256), torch.nn.Tanh(),
                                torch.nn.Linear(256, 10)).to(device="cuda", dtype=tdt)
    ddp = torch.nn.parallel.DistributedDataParallel(model, device_ids=[0], bucket_cap_mb=0.25)
    ops = RecordingOps()
    state = comm_hook.GlobalQSGDState(scheme=scheme, s=s, q=q, p=q, seed=5, ops=ops,
                                      reduce=reduce)
    records = []

    def recording_hook(st, bucket):
        x_in = bucket.buffer().clone()
        step = st.bucket_step(bucket.index())
        fut = comm_hook.global_qsgd_hook(st, bucket)
        norm = ops.norms[-1]

        def rec(f):
            out = f.value()
            records.append((step, x_in, out.clone(), norm))
            return out
        return fut.then(rec)

    ddp.register_comm_hook(state, recording_hook)
    gen = torch.Generator(device="cuda").manual_seed(3)
    for _ in range(2):
        xb = torch.randn(16, 64, device="cuda", generator=gen).to(tdt)
        ddp(xb).float().square().mean().backward()
    torch.cuda.synchronize()
    assert state.step == 2 and len(records) >= 4
    for step, x_in, out, norm_t in records:
        if dtype == "bf16":
            xh = x_in.view(torch.int16).cpu().numpy().view(np.uint16).reshape(1, -1)
        else:
            xh = x_in.cpu().numpy().reshape(1, -1)
        norm32 = float(norm_t.item())
        want_norm = oracle_mod.global_norm(xh, q, q)
        if q == INF:
            assert norm32 == float(np.float32(want_norm))
        else:
            assert norm32 == pytest.approx(want_norm, rel=1e-6)
        codes, rc = oracle_mod.quantize(xh, norm32, scheme, s, 5, step)
        assert rc == 0
        want, rc = oracle_mod.dequantize(oracle_mod.reduce_codes(codes, scheme, s), norm32,
                                         scheme, s, 1)
        got = out.float().cpu().numpy().astype(np.float64)
        tol = 1e-6 * norm32
        if dtype == "bf16":  # the bucket stores the fp32 result rounded to bf16
            tol = tol + np.abs(want) * 2.0 ** -8
        assert np.all(np.abs(got - want) <= tol)
