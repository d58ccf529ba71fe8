"""Benchmark of the fused Global-QSGD allreduce-mean (gq_allreduce_mean) on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = one call of the whole hot path (global norm -> stochastic quantisation -> integer sum
over the n workers -> dequantisation) over one n x d gradient matrix resident in HBM.  The
metric is GB/s of gradient consumed (n * d * element bytes per step / step time).  Inputs are
synthetic and seeded (allreduce_compatible_gradient_gb300.workloads); the default workload is the
largest single-GPU configuration, BERT-large-sized (n = 16 workers, d = 350,000,000 fp32,
Laplace(0, 1e-3) with half of the 4096-coordinate blocks zero, Global-E_4, q = 2, p = inf);
--config names the others (resnet50_n8, bert_base_n8_bf16, gauss_n4_d65536).

Timing: W warm-up steps, then K steps timed one by one with CUDA events on the launching stream;
L2 is flushed (a 512 MiB write, then a 256 MiB read) between timed steps, outside the timed region.  Under torchrun
every rank runs an independent replica on its own GPU (the path needs no data exchange on one
GPU per problem); elapsed time is the max over ranks.

--impl reference times the CPU oracle (test infrastructure, as it stands) on a bounded column
window of the same workload on the host cores, rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused Global-QSGD GB/s of fp32 grads (n×d) and % of GB300 HBM roofline"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="bert_large_n16_sparse")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sweep-max-gb", type=float, default=120.0,
                    help="--measure sweep: skip points whose n*d*4 bytes exceed this")
    ap.add_argument("--columns", type=int, default=None,
                    help="run the workload with d columns instead of its own (a smaller case of the "
                         "same kernels, e.g. for an ncu capture); named '<workload>_d<columns>'")
    ap.add_argument("--measure", default=None, choices=["exp-reduce", "segments", "sweep"],
                    help="extra measurement instead of the main bench line")
    ap.add_argument("--rounding", default="exact", choices=["exact", "u16"],
                    help="rounding mode: exact (default) or the 16-bit-uniform option")
    return ap.parse_args()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_source_hash() -> str:
    """Hash of the CUDA sources with comments and blank lines removed (a comment edit does not
    make the committed ncu traffic figures stale; a code edit does)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "allreduce_compatible_gradient_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name)) as f:
                text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
            for line in text.splitlines():
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def _ncu_traffic(key: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("kernel_source_hash") != _kernel_source_hash():
        return None
    v = t.get("per_launch_dram_bytes", {}).get(key)
    return None if v is None else float(v)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms; only the samples whose
    timestamps fall inside the timed window are reported."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.5)  # let the first samples arrive before the timed window opens

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # a sample read at host time t describes the GPU up to ~50 ms before t
        for t, ln in self.lines:
            if self.t0 is not None and not (self.t0 <= t <= self.t1 + 0.06):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for name, val in zip(names, parts[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist_init(nranks):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return dist.get_rank(), world, local
    return 0, 1, 0


def _max_over_ranks(value: float, world: int) -> float:
    """The max of `value` over all ranks (a scalar collective on the timing, not on data)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_ms: float, bytes_per_rank: int, world: int) -> tuple:
    """Whole-job throughput: every rank processed `bytes_per_rank`; the job took the slowest
    rank's time.  Returns (ms per step, GB/s)."""
    ms = _max_over_ranks(per_rank_ms, world)
    return ms, world * bytes_per_rank / (ms * 1e-3) / 1e9


def _barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def _oracle_window(cfg: dict, seconds: float):
    """A column window of the workload sized to about `seconds` of single-threaded oracle work,
    generated on the host once: (window width, host inputs)."""
    from allreduce_compatible_gradient_gb300 import workloads
    from oracle import gq_oracle

    d = cfg["d"]
    w = min(d, 1 << 14)
    x = workloads.host_inputs(cfg["dist"], cfg["n"], w, seed=cfg["input_seed"], dtype=cfg["dtype"])
    t0 = time.perf_counter()
    gq_oracle.allreduce_mean(x, cfg["q"], cfg["p"], cfg["scheme"] & 1, cfg["s"], cfg["seed"],
                             cfg["step"])
    dt = time.perf_counter() - t0
    w = int(min(d, max(w, w * seconds / max(dt, 1e-6))))
    w = max(32, w // 32 * 32) if w < d else d
    x = workloads.host_inputs(cfg["dist"], cfg["n"], w, seed=cfg["input_seed"], dtype=cfg["dtype"])
    return w, x


def _time_oracle(cfg: dict, w: int, x) -> dict:
    from oracle import gq_oracle

    elt = 2 if cfg["dtype"] == "bf16" else 4
    t0 = time.perf_counter()
    gq_oracle.allreduce_mean(x, cfg["q"], cfg["p"], cfg["scheme"] & 1, cfg["s"], cfg["seed"],
                             cfg["step"])
    dt = time.perf_counter() - t0
    return {"value": round(cfg["n"] * w * elt / dt / 1e9, 6), "unit": UNIT, "cores": 1,
            "kind": "oracle",
            "sample": "%d x %d columns of %s (same distribution; whole pipeline: norm of the "
                      "window, quantise, sum, dequantise), %.1f s" % (cfg["n"], w, cfg["name"], dt),
            "seconds": round(dt, 3), "window_columns": w}


def cpu_baseline(cfg: dict, seconds: float, host_x=None) -> dict:
    """Time the CPU oracle (as it stands, single-threaded) on a column window of the workload."""
    w, x = _oracle_window(cfg, seconds)
    return _time_oracle(cfg, w, x)


def run_reference(a, cfg):
    """The oracle as the reference arm: rank 0 only; each step times the oracle on one column
    window of the workload (generated once), sized so that the whole run stays near two
    minutes of CPU work."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_step = max(0.2, min(a.cpu_seconds, 120.0 / (a.steps + a.warmup)))
    w, x = _oracle_window(cfg, per_step)
    steps = []
    for i in range(a.warmup + a.steps):
        r = _time_oracle(cfg, w, x)
        if i >= a.warmup:
            steps.append(r)
    val = statistics.median(r["value"] for r in steps)
    elt = 2 if cfg["dtype"] == "bf16" else 4
    # each timed step ran the oracle on a w-column window only: the time of a whole step is
    # extrapolated from the window's throughput (the oracle's work is linear in the columns)
    ms = 1e3 * cfg["n"] * cfg["d"] * elt / (val * 1e9)
    window_ms = statistics.median(1e3 * r["seconds"] for r in steps)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT,
            "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 4),
            "ms_per_step_extrapolated": True, "window_columns": w,
            "window_ms_per_step": round(window_ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg["dtype"], "data": "synthetic",
            "config": _config_block(cfg, a.gpus),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": steps[0]["sample"]},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _config_block(cfg, ngpus):
    return {"workload": cfg["name"], "n": cfg["n"], "d": cfg["d"], "input_dtype": cfg["dtype"],
            "distribution": cfg["dist"],
            "scheme": "Global-L" if cfg["scheme"] & 1 == 0 else "Global-E",
            "rounding": "16-bit uniform" if cfg["scheme"] & 16 else "exact",
            "s": cfg["s"], "q": "inf" if cfg["q"] == 0 else 2, "p": "inf" if cfg["p"] == 0 else 2,
            "philox_seed": cfg["seed"], "parallelism": "replica x%d" % ngpus,
            "l2": "flushed between timed steps (512 MiB write, then 256 MiB read); input %.1f MB > 129 MB L2"
                  % (cfg["n"] * cfg["d"] * (2 if cfg["dtype"] == "bf16" else 4) / 1e6)}


def measure_exp_reduce(a) -> int:
    """Cost of the Global-E custom reduction step against a native sum, on the pages' setting:
    one GPU, a 25 MB buffer (PyTorch DDP's default bucket).  One step of each kind is timed
    with CUDA events; the buffers (75 MB per step) stay in L2 between steps, as on the pages'
    single-buffer micro-measurement."""
    import torch

    import allreduce_compatible_gradient_gb300 as gq

    d = 25_000_000
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    ca = torch.randint(-12, 13, (d,), generator=g, device="cuda", dtype=torch.int8)
    cb = torch.randint(-12, 13, (d,), generator=g, device="cuda", dtype=torch.int8)
    out = torch.empty(d, dtype=torch.int8, device="cuda")
    fa = torch.randn(d // 4, generator=g, device="cuda")  # 25 MB of fp32
    fb = torch.randn(d // 4, generator=g, device="cuda")
    fo = torch.empty_like(fa)
    sid = gq.gq_exp_tree_stream(1, 0)

    def timeit(fn):
        for _ in range(a.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(a.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / a.steps

    t_comb = timeit(lambda: gq.gq_exp_combine(ca, cb, 1, 2, sid, out=out))
    t_i8 = timeit(lambda: torch.add(ca, cb, out=out))
    t_f32 = timeit(lambda: torch.add(fa, fb, out=fo))
    line = {"measure": "exp_reduce_cost", "buffer_bytes": d, "steps": a.steps,
            "combine_ms": round(t_comb, 5), "native_int8_sum_ms": round(t_i8, 5),
            "native_fp32_sum_ms": round(t_f32, 5),
            "combine_gb_per_s_of_buffer": round(d / (t_comb * 1e-3) / 1e9, 1),
            "native_int8_gb_per_s_of_buffer": round(d / (t_i8 * 1e-3) / 1e9, 1),
            "combine_time_over_native_int8": round(t_comb / t_i8, 3),
            "combine_time_over_native_fp32": round(t_comb / t_f32, 3),
            "native_sums": "torch.add on the same buffers (library kernels, reference only)"}
    print(json.dumps(line), flush=True)
    return 0


def measure_segments(a) -> int:
    """The per-layer and per-bucket forms against the whole-vector call, on ResNet-50 with 8
    workers (fp32, Global-L_127, max norm): the 161 parameter tensors as segments, the 5 buckets
    PyTorch DDP forms at its 25 MiB cap, and the whole 25,557,032-vector.  Each step is timed
    with CUDA events on the launching stream after an L2 flush; GB/s counts the fused path's
    algorithmic bytes (x read twice, out written once)."""
    import torch

    import allreduce_compatible_gradient_gb300 as gq
    from allreduce_compatible_gradient_gb300 import workloads

    n, sc, s, q, p, seed = 8, gq.LINEAR, 127, gq.NORM_INF, gq.NORM_INF, 1
    layers = workloads.resnet50_layer_sizes()
    buckets = workloads.ddp_buckets(layers)
    d = sum(layers)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    clean = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    ws = gq.gq_workspace()
    stream = torch.cuda.current_stream()

    def timeit(fn):
        for k in range(a.warmup):
            fn(k)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(a.steps)]
        for k in range(a.steps):
            flush.zero_()
            clean.sum()
            ev[k][0].record(stream)
            fn(a.warmup + k)
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)

    res = {}
    for name, sizes in (("layers_161", layers), ("ddp_buckets_5", buckets), ("whole_1", [d])):
        segs = workloads.segment_tensors(n, sizes, seed=8)
        outs = [torch.empty(sz, dtype=torch.float32, device="cuda") for sz in sizes]
        if len(sizes) == 1:
            ms = timeit(lambda k: gq.gq_allreduce_mean(segs[0], q, p, sc, s, seed, k, out=outs[0],
                                                       ws=ws, stream=stream))
        else:
            ms = timeit(lambda k: gq.gq_allreduce_mean_segments(segs, q, p, sc, s, seed, k,
                                                                outs=outs, ws=ws, stream=stream))
        res[name] = ms
        if name == "whole_1":  # the same call writing a bf16 mean (half the output bytes)
            o16 = torch.empty(d, dtype=torch.bfloat16, device="cuda")
            res["whole_1_bf16_out"] = timeit(
                lambda k: gq.gq_allreduce_mean(segs[0], q, p, sc, s, seed, k, out=o16, ws=ws,
                                               stream=stream))
            del o16
        if name == "layers_161":  # the same layers as 161 separate calls
            def loop(k):
                for l, (x, o) in enumerate(zip(segs, outs)):
                    gq.gq_allreduce_mean(x, q, p, sc, s, seed, (k << 16) | l, out=o, ws=ws,
                                         stream=stream)
            res["layers_161_separate_calls"] = timeit(loop)
        del segs, outs
        torch.cuda.empty_cache()
    if gq.gq_get_status(ws) != 0:
        raise RuntimeError("device status not ok")
    algo = 2 * n * d * 4 + 4 * d
    line = {"measure": "segments", "workload": "resnet50 n=8 fp32 Global-L_127 max norm",
            "d": d, "n": n, "steps": a.steps, "warmup": a.warmup,
            "ddp_bucket_sizes": buckets,
            "ms": {k: round(v, 4) for k, v in res.items()},
            "gb_per_s": {k: round(algo / (v * 1e-3) / 1e9, 1) for k, v in res.items()},
            "l2": "flushed between timed steps"}
    print(json.dumps(line), flush=True)
    return 0


def measure_sweep(a) -> int:
    """The fused call over the sweep grid: n in {2..64} x d in {2^20..2^28}, fp32 N(0,1),
    Global-L_7 and Global-E_4, q = p = 2 (points above --sweep-max-gb skipped).  Each step is
    timed with CUDA events after an L2 flush; GB/s counts n*d*4 bytes of gradient, the fraction
    of the copy peak the call's algorithmic bytes (x read once per launch, out written once)."""
    import torch

    import allreduce_compatible_gradient_gb300 as gq
    from allreduce_compatible_gradient_gb300 import workloads

    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    clean = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    ws = gq.gq_workspace()
    stream = torch.cuda.current_stream()
    points = []
    peak, peak_kind = _peaks()
    for n in workloads.SWEEP_N:
        for d in workloads.SWEEP_D:
            if n * d * 4 > a.sweep_max_gb * 1e9:
                points.append({"n": n, "d": d, "skipped": "n*d*4 above --sweep-max-gb"})
                continue
            try:
                x = workloads.device_inputs("normal", n, d, seed=0)
                out = torch.empty(d, dtype=torch.float32, device="cuda")
            except torch.OutOfMemoryError:
                points.append({"n": n, "d": d, "skipped": "device memory"})
                torch.cuda.empty_cache()
                continue
            for scheme, s in workloads.SWEEP_SCHEMES:
                def step(k):
                    gq.gq_allreduce_mean(x, gq.NORM_L2, gq.NORM_L2, scheme, s, 1, k, out=out,
                                         ws=ws, stream=stream)
                for k in range(a.warmup):
                    step(k)
                torch.cuda.synchronize()
                ts = []
                for k in range(a.steps):
                    flush.zero_()
                    clean.sum()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    step(a.warmup + k)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1))
                ms = statistics.median(ts)
                launches = gq.gq_fused_launches(x.dtype, n, d)
                algo = launches * n * d * 4 + 4 * d  # x read once per launch, out written once
                points.append({"n": n, "d": d, "scheme": "LE"[scheme] + str(s),
                               "ms": round(ms, 4), "launches": launches,
                               "gb_per_s": round(n * d * 4 / (ms * 1e-3) / 1e9, 1),
                               "frac_of_measured_peak": round(algo / (ms * 1e-3) / 1e9 / peak, 4)})
            del x, out
            torch.cuda.empty_cache()
    if gq.gq_get_status(ws) != 0:
        raise RuntimeError("device status not ok")
    print(json.dumps({"measure": "sweep", "peak_gbs": peak, "peak_kind": peak_kind,
                      "steps": a.steps, "warmup": a.warmup, "l2": "flushed between timed steps",
                      "points": points}), flush=True)
    return 0


def _two_pass_roofline(gq, x, q, p, sc, s, seed, a, cfg, stream, flush_l2, norm, out, ws,
                       ms_per_step, in_bytes, d, peak, peak_kind):
    """Roofline of the dominant kernel of the two-pass fused call: the norm pass is timed alone
    through gq_global_norm (the same kernel), the quantise pass as the step minus it."""
    import torch

    ev_k = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
    for k in range(a.steps):
        flush_l2()
        ev_k[k][0].record(stream)
        gq.gq_global_norm(x, q, p, norm=norm, ws=ws, stream=stream)
        ev_k[k][1].record(stream)
        gq.gq_allreduce_mean_with_norm(x, norm, sc, s, seed, a.warmup + k, out=out, ws=ws,
                                       stream=stream)
        ev_k[k][2].record(stream)
    torch.cuda.synchronize()
    t_norm = statistics.mean(e[0].elapsed_time(e[1]) for e in ev_k)
    t_quant_split = statistics.mean(e[1].elapsed_time(e[2]) for e in ev_k)
    # the fused call launches the same norm kernel and then its own quantise pass: that pass
    # takes the step time minus the norm time (both measured above with events on the stream)
    t_quant = max(ms_per_step - t_norm, 1e-6)
    kernels = {
        "norm": {"ms": t_norm, "bytes": in_bytes},
        "quantize_sum_dequantize": {"ms": t_quant, "bytes": in_bytes + 4 * d},
    }
    dom_name = max(kernels, key=lambda k: kernels[k]["ms"])
    dom = kernels[dom_name]
    achieved = dom["bytes"] / (dom["ms"] * 1e-3) / 1e9
    traffic = _ncu_traffic("%s@%s" % (dom_name, cfg["name"]))
    return {"bound": "hbm", "kernel": dom_name, "achieved": round(achieved, 1),
            "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_kind": peak_kind, "traffic": traffic,
            "algorithmic_bytes_per_launch": dom["bytes"],
            "kernels_ms": {k: round(v["ms"], 4) for k, v in kernels.items()},
            "quantize_with_norm_entry_ms": round(t_quant_split, 4),
            "whole_step_frac": round((2 * in_bytes + 4 * d) / (ms_per_step * 1e-3) / 1e9 / peak, 4),
            "whole_step_frac_of_8tbs": round(
                (2 * in_bytes + 4 * d) / (ms_per_step * 1e-3) / 1e12 / 8.0, 4)}


def main():
    a = _args()
    if a.measure == "exp-reduce":
        return measure_exp_reduce(a)
    if a.measure == "segments":
        return measure_segments(a)
    if a.measure == "sweep":
        return measure_sweep(a)
    from allreduce_compatible_gradient_gb300 import workloads

    cfg = dict(workloads.CONFIGS[a.config], name=a.config)
    if a.rounding == "u16":
        cfg["scheme"] |= 16  # GQ_ROUND_U16
        cfg["name"] += "_u16"
    if a.columns is not None:
        if a.columns < 1:
            raise SystemExit("--columns must be positive")
        cfg["d"], cfg["name"] = a.columns, "%s_d%d" % (a.config, a.columns)
    if a.impl == "reference":
        return run_reference(a, cfg)

    import torch

    import allreduce_compatible_gradient_gb300 as gq

    rank, world, local = _dist_init(a.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n, d = cfg["n"], cfg["d"]
    elt = 2 if cfg["dtype"] == "bf16" else 4
    in_bytes = n * d * elt
    x = workloads.device_inputs(cfg["dist"], n, d, seed=cfg["input_seed"] + rank,
                                dtype=cfg["dtype"], device=dev)
    out = torch.empty(d, dtype=torch.float32, device=dev)
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    ws = gq.gq_workspace(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    clean = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def flush_l2():
        # evict the working set: write 512 MiB, then read 256 MiB so that the dirty lines of the
        # write are drained before the timed region starts
        flush.zero_()
        clean.sum()
    stream = torch.cuda.current_stream(dev)
    sc, s, q, p, seed = cfg["scheme"], cfg["s"], cfg["q"], cfg["p"], cfg["seed"]

    def step(k):
        gq.gq_allreduce_mean(x, q, p, sc, s, seed, k, out=out, norm=norm, ws=ws, stream=stream)

    clocks = ClockSampler(local)
    clocks.start()
    for k in range(a.warmup):
        step(k)
    torch.cuda.synchronize()
    if gq.gq_get_status(ws) != 0:
        raise RuntimeError("device status not ok after warm-up")

    # --- timed: the public fused call ---------------------------------------------------------
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(a.steps)]
    _barrier(world)
    torch.cuda.synchronize()
    t_open = time.time()
    for k in range(a.steps):
        flush_l2()
        ev[k][0].record(stream)
        step(a.warmup + k)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    t_close = time.time()
    _barrier(world)
    clocks.window(t_open, t_close)
    clk = clocks.stop()
    times = [e0.elapsed_time(e1) for e0, e1 in ev]
    ms_per_step, value = aggregate(sum(times) / a.steps, in_bytes, world)
    ms_median = _max_over_ranks(statistics.median(times), world)

    # the same steps back to back without the L2 flush (hot): only inputs below the L2 size can
    # gain, since a step streams all of x twice
    hev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(a.steps)]
    _barrier(world)
    torch.cuda.synchronize()
    for k in range(a.steps):
        hev[k][0].record(stream)
        step(a.warmup + a.steps + k)
        hev[k][1].record(stream)
    torch.cuda.synchronize()
    hot_ms = _max_over_ranks(statistics.median(e0.elapsed_time(e1) for e0, e1 in hev), world)
    hot = {"ms_per_step_median": round(hot_ms, 5),
           "value": round(world * in_bytes / (hot_ms * 1e-3) / 1e9, 3), "l2": "not flushed"}

    launches = gq.gq_fused_launches(x.dtype, n, d)
    peak, peak_kind = _peaks()
    if launches == 1:
        # small problem: one launch reads x once and writes out (single-launch form)
        step_bytes = in_bytes + 4 * d
        achieved = step_bytes / (ms_per_step * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": "resident_kernel", "achieved": round(achieved, 1),
                    "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "peak_kind": peak_kind,
                    "traffic": _ncu_traffic("resident@%s" % cfg["name"]),
                    "algorithmic_bytes_per_launch": step_bytes,
                    "kernels_ms": {"resident": round(ms_per_step, 4)},
                    "whole_step_frac": round(achieved / peak, 4)}
    else:
        roofline = _two_pass_roofline(gq, x, q, p, sc, s, seed, a, cfg, stream, flush_l2, norm,
                                      out, ws, ms_per_step, in_bytes, d, peak, peak_kind)

    # --- end to end through the public API with host buffers ---------------------------------
    # Every step copies its n x d input from pinned host memory, runs the call and copies its
    # d outputs back.  For inputs of 64 MiB or more, two device buffers let step k+1's
    # host-to-device copy (one stream) run while step k computes (the launching stream) and its
    # result goes back (a third stream): the host link is full duplex, so the step time is that
    # of the input copy.  Smaller steps run in order on one stream (the extra streams and events
    # would cost more host time than they hide).
    e2e = None
    if not a.no_e2e:
        xh = torch.empty((n, d), dtype=x.dtype, pin_memory=True)
        xh.copy_(x)
        xds = [torch.empty_like(x) for _ in range(2)]
        outs = [torch.empty(d, dtype=torch.float32, device=dev) for _ in range(2)]
        ohs = [torch.empty(d, dtype=torch.float32, pin_memory=True) for _ in range(2)]
        pipelined = in_bytes >= (64 << 20)
        h2d_s, d2h_s = (torch.cuda.Stream(dev), torch.cuda.Stream(dev)) if pipelined else (stream, stream)
        free_x, free_o = [None, None], [None, None]

        def e2e_step(k):
            if not pipelined:
                xds[0].copy_(xh, non_blocking=True)
                gq.gq_allreduce_mean(xds[0], q, p, sc, s, seed, k, out=outs[0], norm=norm, ws=ws,
                                     stream=stream)
                ohs[0].copy_(outs[0], non_blocking=True)
                return
            b = k % 2
            with torch.cuda.stream(h2d_s):
                if free_x[b] is not None:
                    h2d_s.wait_event(free_x[b])  # step k-2 is done with this input buffer
                xds[b].copy_(xh, non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(h2d_s)
            stream.wait_event(landed)
            if free_o[b] is not None:
                stream.wait_event(free_o[b])  # step k-2's result has left this output buffer
            gq.gq_allreduce_mean(xds[b], q, p, sc, s, seed, k, out=outs[b], norm=norm, ws=ws,
                                 stream=stream)
            done = torch.cuda.Event()
            done.record(stream)
            free_x[b] = done
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done)
                ohs[b].copy_(outs[b], non_blocking=True)
                back = torch.cuda.Event()
                back.record(d2h_s)
            free_o[b] = back

        for k in range(2):
            e2e_step(k)
        torch.cuda.synchronize()
        ke = max(3, min(a.steps, 10))
        _barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if pipelined:
            h2d_s.wait_event(e0)
            d2h_s.wait_event(e0)
        for k in range(ke):
            e2e_step(k)
        if pipelined:
            stream.wait_stream(h2d_s)
            stream.wait_stream(d2h_s)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = _max_over_ranks(e0.elapsed_time(e1) / ke, world)
        e2e = {"value": round(world * in_bytes / (e_ms * 1e-3) / 1e9, 3), "unit": UNIT,
               "ms_per_step": round(e_ms, 4), "h2d_bytes_per_step": in_bytes,
               "d2h_bytes_per_step": 4 * d,
               "pipelined": ("two device buffers: step k+1's input copy overlaps step k's call "
                             "and result copy") if pipelined else "no: copies and call in order "
                                                                 "on one stream"}
        del xh, xds, outs, ohs

    if gq.gq_get_status(ws) != 0:
        raise RuntimeError("device status not ok after the timed steps")

    # compression error of one step (outside every timed region): the relative l2 distance of the
    # dequantised mean from the exact mean of the n rows, both in fp64
    step(0)
    torch.cuda.synchronize()
    exact = x.mean(0, dtype=torch.float64)
    mnorm = float(exact.norm())
    rel = float((out.double() - exact).norm()) / mnorm if mnorm > 0 else 0.0
    del exact
    # the variance bound of the quantiser over the whole matrix, E||Q - X||_F^2 <= min(n d N^2 /
    # (4 s^2), N ||X||_1 / s) (Global-L) or ||X||_F^2 / 8 + 2^-(s-1) N ||X||_1 (Global-E), divided
    # by n^2 for the mean of n independently rounded rows
    l1 = sum(float(x[i].abs().sum(dtype=torch.float64)) for i in range(n))
    l2sq = sum(float(x[i].double().square().sum()) for i in range(n))
    N = float(norm.item())
    if sc & 1 == 0:
        bound = min(n * d * N * N / (4.0 * s * s), N * l1 / s)
    else:
        bound = l2sq / 8.0 + 2.0 ** -(s - 1) * N * l1
    rel_bound = (bound ** 0.5) / n / mnorm if mnorm > 0 else 0.0
    compression = {"rel_l2": round(rel, 6), "rel_l2_bound": round(rel_bound, 6),
                   "of": "||out - mean(x)||_2 / ||mean(x)||_2 for one step; bound: the square root "
                         "of the quantiser's variance bound over n^2, over ||mean(x)||_2"}

    cpu = None
    if rank == 0 and not a.no_cpu_baseline:
        cpu = cpu_baseline(cfg, a.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
                "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms_per_step, 5),
                "ms_per_step_median": round(ms_median, 5), "hot": hot,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": cfg["dtype"], "data": "synthetic",
                "config": _config_block(cfg, world), "roofline": roofline,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches * a.steps,
                "clocks": clk, "compression_error": compression, "impl": "ours"}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
