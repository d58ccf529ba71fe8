"""Host logic of bench.py without a GPU: the replica aggregation across ranks (world size 2 over
gloo, on the CPU), the reference arm's rank and JSON-line behaviour, the --columns option, and
the kernel source hash that keys the committed ncu traffic figures."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, per_rank_ms, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, gbs = bench.aggregate(per_rank_ms[rank], 10**9, world)
    q.put((rank, ms, gbs))
    dist.destroy_process_group()


def test_aggregate_takes_the_slowest_rank():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    per_rank_ms = [2.0, 5.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, per_rank_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, gbs in got:
        assert ms == 5.0                      # max over ranks
        assert gbs == pytest.approx(2 * 1e9 / 5e-3 / 1e9)  # both ranks' bytes over that time


def _run_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config",
                           "gauss_n4_d65536", "--steps", "2", "--warmup", "1", "--gpus",
                           str(world), "--cpu-seconds", "0.2"], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_rank0_prints_one_line_others_exit_quietly():
    r1 = _run_reference(1, 2)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_reference(0, 2)
    assert r0.returncode == 0
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in rec
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["steps"] == 2
    assert rec["value"] > 0 and rec["e2e"]["value"] == rec["value"]
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["config"]["workload"] == "gauss_n4_d65536"


def test_columns_option_names_a_smaller_case():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config",
                        "bert_large_n16_sparse", "--columns", "4096", "--steps", "1", "--warmup",
                        "1", "--cpu-seconds", "0.2"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    rec = json.loads([ln for ln in r.stdout.splitlines() if ln.strip()][-1])
    assert rec["config"]["workload"] == "bert_large_n16_sparse_d4096"
    assert rec["config"]["d"] == 4096 and rec["config"]["n"] == 16


def test_kernel_source_hash_ignores_comments(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "allreduce_compatible_gradient_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "k.cuh").write_text("// a comment\nint f() { return 1; }  // trailing\n/* block\n */\n")
    h0 = bench._kernel_source_hash()
    (csrc / "k.cuh").write_text("// another comment\n\nint f() { return 1; }\n")
    assert bench._kernel_source_hash() == h0
    (csrc / "k.cuh").write_text("int f() { return 2; }\n")
    assert bench._kernel_source_hash() != h0
