"""The DDP communication hook across processes: CPU ranks (gloo, world size 2) train a small
model through DistributedDataParallel with the Global-QSGD hook registered, and every bucket's
result on every rank must equal the oracle's allreduce_mean of the two ranks' stacked buckets
(worker i = rank i, step = iteration * 2^16 + bucket index, n = 2).  This pins the hook's
choreography: the norm exchange, the worker index keying each rank's random words, the step
folding, the integer sum over ranks and the n of the dequantisation.  A rank that fails inside
the hook must make the other fail by the process group's timeout, not hang.

Test infrastructure only: the four per-bucket steps on each rank are the oracle's (no GPU here),
substituted through the hook's `ops`.
"""
import datetime
import math
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2
ITERS = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The hook's four steps computed by the oracle on host tensors."""

    def __init__(self, oracle):
        self.o = oracle
        self.norms = []
        self.wire = []

    @staticmethod
    def _host(x):
        import torch
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16)
        return x.numpy()

    def norm_partial(self, x, q, p):
        import torch
        v = self.o.global_norm(self._host(x), q, p)
        return torch.tensor([v * v if q == 2 else v], dtype=torch.float64)

    def norm_finish(self, part, q, p):
        import torch
        v = float(part.item())
        n32 = np.float32(math.sqrt(v) if q == 2 else v)
        self.norms.append(float(n32))
        return torch.tensor([n32], dtype=torch.float32)

    def quantize_sum(self, x, norm, scheme, s, seed, step, worker0, sum_dtype):
        import torch
        xh = self._host(x)
        # the oracle numbers workers by row: put this rank's row at index worker0
        stacked = np.zeros((worker0 + 1, xh.shape[1]), dtype=xh.dtype)
        stacked[worker0] = xh[0]
        codes, rc = self.o.quantize(stacked, float(norm.item()), scheme, s, seed, step)
        assert rc == 0
        sums = self.o.reduce_codes(codes[worker0:worker0 + 1], scheme, s)
        self.wire.append(sum_dtype)
        np_type = np.int8 if sum_dtype == torch.int8 else np.int32
        assert np.abs(sums).max(initial=0) <= np.iinfo(np_type).max
        return torch.from_numpy(sums.astype(np_type))

    # the re-rounding allreduce of Global-E
    def quantize_codes(self, x, norm, scheme, s, seed, step, worker0):
        import torch
        xh = self._host(x)
        stacked = np.zeros((worker0 + 1, xh.shape[1]), dtype=xh.dtype)
        stacked[worker0] = xh[0]
        codes, rc = self.o.quantize(stacked, float(norm.item()), scheme, s, seed, step)
        assert rc == 0
        return torch.from_numpy(codes[worker0].copy())

    def exp_combine(self, a, b, seed, step, stream_id, j0):
        import torch
        return torch.from_numpy(self.o.exp_combine(a.numpy(), b.numpy(), seed, step, stream_id,
                                                   j0=j0))

    def exp_dequantize(self, codes, norm, s, n, out):
        got, rc = self.o.dequantize(self.o.exp_units(codes.numpy()), float(norm.item()), 1, s, n)
        assert rc == 0
        import torch
        out.view(-1).copy_(torch.from_numpy(got.astype(np.float32)))
        return out

    def exp_tree_stream(self, level, m):
        return self.o.exp_tree_stream(level, m)

    def exp_ring_stream(self, h, c):
        return self.o.exp_ring_stream(h, c)

    def dequantize(self, sums, norm, scheme, s, n, out):
        import torch
        got, rc = self.o.dequantize(sums.numpy().astype(np.int64), float(norm.item()), scheme, s, n)
        assert rc == 0
        t = torch.from_numpy(got.astype(np.float32))
        if out is None:
            return t
        out.view(-1).copy_(t)
        return out


def _model(dtype):
    import torch
    torch.manual_seed(0)
    # DDP fills its first bucket to 1 MiB, later ones to bucket_cap_mb; gradients arrive in
    # reverse layer order, so this gives two buckets: the last three layers, then the first
    m = torch.nn.Sequential(torch.nn.Linear(64, 512), torch.nn.Tanh(), torch.nn.Linear(512, 512),
                            torch.nn.Tanh(), torch.nn.Linear(512, 256), torch.nn.Tanh(),
                            torch.nn.Linear(256, 10))
    return m.to(dtype)


def _rank_main(rank, port, cfg, q, world):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from oracle import gq_oracle
    from allreduce_compatible_gradient_gb300 import comm_hook

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=8))
    try:
        dtype = torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32
        ddp = torch.nn.parallel.DistributedDataParallel(_model(dtype), bucket_cap_mb=0.25)
        ops = OracleOps(gq_oracle)
        state = comm_hook.GlobalQSGDState(scheme=cfg["scheme"], s=cfg["s"], q=cfg["q"],
                                          p=cfg["q"], seed=cfg["seed"], step=cfg["step0"],
                                          reduce=cfg.get("reduce", "sum"), ops=ops)
        records = []

        def recording_hook(st, bucket):
            if rank == cfg.get("fail_rank") and st.step == cfg["step0"] + 1:
                raise RuntimeError("injected failure")
            x_in = OracleOps._host(bucket.buffer().clone()).copy()
            step = st.bucket_step(bucket.index())
            fut = comm_hook.global_qsgd_hook(st, bucket)
            norm_used = ops.norms[-1]  # this bucket's: later buckets may start before f completes

            def rec(f):
                out = f.value()
                records.append((step, x_in, out.float().numpy().copy(), norm_used))
                return out
            return fut.then(rec)

        ddp.register_comm_hook(state, recording_hook)
        gen = torch.Generator().manual_seed(100 + rank)
        for _ in range(ITERS):
            x = torch.randn(16, 64, generator=gen).to(dtype)
            ddp(x).float().square().mean().backward()
        q.put((rank, "ok", (records, sorted({str(w) for w in ops.wire}))))
    except Exception as e:  # noqa: BLE001 - the failure path is what the test looks at
        q.put((rank, "failed", str(e)[:300]))
    finally:
        try:
            dist.destroy_process_group()
        except Exception:  # noqa: BLE001
            pass


def _run(cfg, world=WORLD):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, cfg, q, world)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, status, payload = q.get(timeout=180)
        res[rank] = (status, payload)
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    return res


CASES = [
    dict(dtype="f32", scheme=1, s=8, q=0, seed=11, step0=0),   # Global-E_8, max norm
    dict(dtype="f32", scheme=0, s=15, q=2, seed=12, step0=5),  # Global-L_15, l2 norm
    dict(dtype="bf16", scheme=1, s=4, q=0, seed=13, step0=1),  # Global-E_4 (int4 codes), bf16
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: "%s-%s%d-q%d" % (
    c["dtype"], "LE"[c["scheme"]], c["s"], c["q"]))
def test_hook_matches_the_oracle(oracle, cfg):
    res = _run(cfg)
    for r in range(WORLD):
        assert res[r][0] == "ok", res[r][1]
    # completions may be recorded in a different order on each rank: match them by step
    recs = [sorted(res[r][1][0], key=lambda rec: rec[0]) for r in range(WORLD)]
    # the wire type: int8 when the sum over the workers fits, else int32
    units = cfg["s"] if cfg["scheme"] == 0 else 1 << (cfg["s"] - 1)
    want_wire = "torch.int8" if WORLD * units <= 127 else "torch.int32"
    assert res[0][1][1] == [want_wire] and res[1][1][1] == [want_wire]
    assert len(recs[0]) == len(recs[1]) and len(recs[0]) >= 2 * ITERS  # several buckets per pass
    steps = [rec[0] for rec in recs[0]]
    assert len(set(steps)) == len(steps)  # every (iteration, bucket) draws its own stream
    assert {st >> 16 for st in steps} == {cfg["step0"] + i for i in range(ITERS)}
    for k in range(len(recs[0])):
        step, x0, out0, norm_used = recs[0][k]
        step1, x1, out1, norm1 = recs[1][k]
        assert step == step1 and norm_used == norm1
        stacked = np.ascontiguousarray(np.stack([x0, x1]))
        want_norm = oracle.global_norm(stacked, cfg["q"], cfg["q"])
        if cfg["q"] == 0:
            assert norm_used == float(np.float32(want_norm))
        else:
            assert norm_used == pytest.approx(want_norm, rel=1e-6)
        codes, rc = oracle.quantize(stacked, norm_used, cfg["scheme"], cfg["s"], cfg["seed"], step)
        assert rc == 0
        sums = oracle.reduce_codes(codes, cfg["scheme"], cfg["s"])
        want, rc = oracle.dequantize(sums, norm_used, cfg["scheme"], cfg["s"], WORLD)
        assert rc == 0
        want32 = want.astype(np.float32)
        if cfg["dtype"] == "bf16":  # the bucket holds bf16: compare after the same rounding
            import torch
            want32 = torch.from_numpy(want32).to(torch.bfloat16).float().numpy()
        np.testing.assert_array_equal(out0, want32)
        np.testing.assert_array_equal(out1, want32)


def test_failed_rank_is_detected_not_hung():
    cfg = dict(CASES[0], fail_rank=1)
    res = _run(cfg)
    assert res[1][0] == "failed" and "injected failure" in res[1][1]
    assert res[0][0] == "failed"  # its next collective times out or loses the peer


def test_state_rejects_bad_configurations():
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from allreduce_compatible_gradient_gb300 import comm_hook
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        with pytest.raises(ValueError):
            comm_hook.GlobalQSGDState(q=2, p=0, ops=object())  # mixed order
        with pytest.raises(ValueError):
            comm_hook.GlobalQSGDState(scheme=1, s=25, ops=object())
        st = comm_hook.GlobalQSGDState(scheme=1, s=8, ops=object(), step=3)
        assert st.bucket_step(5) == (3 << 16) | 5
        with pytest.raises(ValueError):
            st.bucket_step(1 << 16)
        # the ring's random streams number chunks in 12 bits: at most 4096 ranks
        cls = comm_hook.GlobalQSGDState
        orig = cls.world_size
        try:
            cls.world_size = property(lambda self: 4097)
            with pytest.raises(ValueError):
                cls(scheme=1, s=2, reduce="ring", ops=object())
            cls(scheme=1, s=2, reduce="tree", ops=object())
            cls.world_size = property(lambda self: 4096)
            cls(scheme=1, s=2, reduce="ring", ops=object())
        finally:
            cls.world_size = orig
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [3, 4])
@pytest.mark.parametrize("reduce", ["tree", "ring"])
def test_hook_reround_allreduce_matches_the_oracle(oracle, reduce, world):
    """reduce="tree" / "ring": int8 codes over point-to-point sends, re-rounded at every hop;
    every bucket on every rank equals the oracle's tree / ring allreduce of the stacked codes,
    dequantised with n = world size."""
    cfg = dict(dtype="f32", scheme=1, s=8, q=0, seed=21, step0=2, reduce=reduce)
    res = _run(cfg, world)
    for r in range(world):
        assert res[r][0] == "ok", res[r][1]
    recs = [sorted(res[r][1][0], key=lambda rec: rec[0]) for r in range(world)]
    assert all(len(rc) == len(recs[0]) for rc in recs) and len(recs[0]) >= 2 * ITERS
    for k in range(len(recs[0])):
        step, norm_used = recs[0][k][0], recs[0][k][3]
        stacked = np.ascontiguousarray(np.stack([recs[r][k][1] for r in range(world)]))
        assert norm_used == float(np.float32(oracle.global_norm(stacked, 0, 0)))
        codes, rc = oracle.quantize(stacked, norm_used, 1, 8, 21, step)
        assert rc == 0
        d = stacked.shape[1]
        root = (oracle.exp_tree_allreduce(codes, 21, step) if reduce == "tree"
                else oracle.exp_ring_allreduce(codes, d, 21, step))
        want, rc = oracle.dequantize(oracle.exp_units(root), norm_used, 1, 8, world)
        assert rc == 0
        for r in range(world):
            assert recs[r][k][0] == step
            np.testing.assert_array_equal(recs[r][k][2], want.astype(np.float32))
