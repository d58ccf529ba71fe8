"""The Global-E allreduce as the pages run it, across processes: CPU ranks (gloo, world size 4)
exchange code vectors with point-to-point send/recv (the pages build their custom allreduce on
NCCL's point-to-point API) and apply the re-rounding step at every hop.  Checked bit for bit
against the single-process oracle's tree and ring; and a rank that fails before its first send
must make the others fail fast (a short process-group timeout), not hang.

Test infrastructure only: the step on each rank is the oracle's (there is no GPU here).
"""
import datetime
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N, D, S, SEED, STEP = 4, 203, 6, 77, 9


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    sys.path.insert(0, ROOT)
    from allreduce_compatible_gradient_gb300 import workloads
    return workloads.host_inputs("normal", N, D, seed=5)


def _rank_main(rank, port, mode, fail_rank, q):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from oracle import gq_oracle as o
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=N,
                            timeout=datetime.timedelta(seconds=8))
    try:
        x = _inputs()
        # the norm: a scalar max-allreduce of the local maxima (exact for q = p = inf)
        local = torch.tensor([float(np.abs(x[rank]).max())], dtype=torch.float64)
        dist.all_reduce(local, op=dist.ReduceOp.MAX)
        norm32 = np.float32(local.item())
        # this rank's codes: worker index `rank` keys its random words (the oracle quantises all
        # rows at once; each rank keeps its own row)
        codes, _ = o.quantize(x, norm32, o.EXP, S, SEED, STEP)
        mine = codes[rank].copy()
        if rank == fail_rank:
            raise RuntimeError("injected failure")
        if mode == "tree":
            acc = mine
            l = 1
            while (1 << (l - 1)) < N:
                half = 1 << (l - 1)
                if rank % (2 * half) == 0 and rank + half < N:
                    other = torch.empty(D, dtype=torch.int8)
                    dist.recv(other, src=rank + half)
                    acc = o.exp_combine(acc, other.numpy(), SEED, STEP, o.exp_tree_stream(l, rank >> l))
                elif rank % (2 * half) == half:
                    dist.send(torch.from_numpy(acc), dst=rank - half)
                l += 1
            root = torch.from_numpy(acc.copy()) if rank == 0 else torch.empty(D, dtype=torch.int8)
            dist.broadcast(root, src=0)  # the allgather half only copies
            result = root.numpy()
        else:  # ring reduce-scatter, then allgather
            chunk = -(-(-(-D // N)) // 16) * 16  # ceil(D / N) rounded up to a multiple of 16
            bounds = [(min(D, c * chunk), min(D, (c + 1) * chunk)) for c in range(N)]
            acc = {}
            c0 = (rank - 1) % N  # this rank starts chunk c0 (worker c0 + 1)
            acc[c0] = mine[bounds[c0][0]:bounds[c0][1]].copy()
            for h in range(1, N):
                send_c = (rank - h) % N
                recv_c = (rank - h - 1) % N
                lo, hi = bounds[recv_c]
                buf = torch.empty(hi - lo, dtype=torch.int8)
                sreq = dist.isend(torch.from_numpy(acc.pop(send_c)), dst=(rank + 1) % N)
                dist.recv(buf, src=(rank - 1) % N)
                sreq.wait()
                acc[recv_c] = o.exp_combine(buf.numpy(), mine[lo:hi], SEED, STEP,
                                            o.exp_ring_stream(h, recv_c), j0=lo)
            # rank holds the finished chunk (rank - N) % N == rank; gather all chunks
            full = torch.zeros(D, dtype=torch.int8)
            (c_done, part), = acc.items()
            full[bounds[c_done][0]:bounds[c_done][1]] = torch.from_numpy(part)
            parts = [torch.zeros(D, dtype=torch.int8) for _ in range(N)]
            dist.all_gather(parts, full)
            result = sum(p.to(torch.int32) for p in parts).to(torch.int8).numpy()
        q.put((rank, "ok", result.tobytes()))
    except Exception as e:  # noqa: BLE001 - the failure path is what the test looks at
        q.put((rank, "failed", str(e)[:200]))
    finally:
        try:
            dist.destroy_process_group()
        except Exception:  # noqa: BLE001
            pass


def _run(mode, fail_rank=-1):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, mode, fail_rank, q)) for r in range(N)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(N):
        rank, status, payload = q.get(timeout=120)
        res[rank] = (status, payload)
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    return res


def _oracle_root(mode):
    sys.path.insert(0, ROOT)
    from oracle import gq_oracle as o
    x = _inputs()
    norm32 = np.float32(np.abs(x).max())
    codes, _ = o.quantize(x, norm32, o.EXP, S, SEED, STEP)
    if mode == "tree":
        return o.exp_tree_allreduce(codes, SEED, STEP)
    return o.exp_ring_allreduce(codes, D, SEED, STEP)


@pytest.mark.parametrize("mode", ["tree", "ring"])
def test_ranks_match_the_oracle(mode):
    res = _run(mode)
    want = _oracle_root(mode)
    for rank in range(N):
        status, payload = res[rank]
        assert status == "ok", payload
        np.testing.assert_array_equal(np.frombuffer(payload, dtype=np.int8), want)


def test_failed_rank_is_detected_not_hung():
    res = _run("tree", fail_rank=1)
    assert res[1] == ("failed", "injected failure")
    # rank 0 waits on rank 1 at the first level: it must fail by timeout or lost connection
    assert res[0][0] == "failed"
