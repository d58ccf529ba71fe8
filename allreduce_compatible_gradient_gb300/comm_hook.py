"""Global-QSGD as a PyTorch DistributedDataParallel communication hook.

Global-QSGD (Xin et al., arXiv 2305.18627), implementation paragraph: the method plugs into DDP
through `register_comm_hook`, and for every gradient bucket the hook quantises, allreduces and
dequantises.  Here each rank is one worker: rank r holds x_r, the flat gradient bucket, and

  1. the global norm N = ||x||_{q,p} over all ranks' buckets: each rank's combinable share
     (gq_norm_partial: a sum of squares for q = p = 2, a maximum for q = p = inf), one scalar
     allreduce (sum or max), then gq_norm_finish -> fp32 N, the same on every rank;
  2. gq_quantize_sum: the rank's stochastically rounded level codes, already in summable integer
     form (Global-L_s: the level index; Global-E_s: 2^(k-1) units of 2^-(s-1)), with worker
     index r keying the random words;
  3. a SUM allreduce of those d integers, exact in any order: int8 on the wire when the total
     over all workers fits (n s <= 127 for Global-L, n 2^(s-1) <= 127 for Global-E; the pages
     sum 8-bit codes natively, which is exact only in that range), a quarter of an fp32
     allreduce's bytes; int32 otherwise;
  4. gq_dequantize_sums with n = world size -> the unbiased estimate of the mean gradient,
     written back into the bucket in its own type (a bf16 bucket gets the fp32 value rounded to
     nearest even).

With reduce="tree" or "ring" (Global-E_s only) the allreduce is the pages' own for exponential
dithering: the ranks exchange int8 level-index codes with point-to-point sends and every hop
re-rounds the sum of two codes back onto the (extended) grid with gq_exp_combine, so the wire
stays one byte per coordinate whatever n and s are, at the price of the extra variance of the
re-rounding; the tree is recursive halving into rank 0 followed by a broadcast, the ring a
reduce-scatter over chunks of ceil(d/n) coordinates rounded up to a multiple of 16, followed by
an allgather (the same definitions as the single-GPU gq_exp_allreduce), and the root's codes are
dequantised with gq_exp_dequantize.

On one GPU with world size 1 this is gq_allreduce_mean of the 1 x d bucket.  The random stream
of bucket b at iteration t uses step t * 2^16 + b (t < 2^48, b < 2^16), so every bucket and
iteration draws fresh words.  The mixed norm orders (2, inf) and (inf, 2) need a d-vector
exchange as large as the uncompressed gradient and are refused.

The arithmetic runs in libgq.so; `ops` may replace the four library calls (the CPU tests of the
multi-process choreography substitute a host implementation there).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch
import torch.distributed as dist

from . import _binding as gq

_STEP_BITS = 16  # bucket index bits folded into the random stream's step


class LibraryOps:
    """The four per-bucket steps, on the current CUDA stream, through libgq.so."""

    def __init__(self):
        self._ws = {}

    def _workspace(self, device):
        key = (device.type, device.index)
        if key not in self._ws:
            self._ws[key] = gq.gq_workspace(device)
        return self._ws[key]

    def norm_partial(self, x, q, p):
        return gq.gq_norm_partial(x, q, p, ws=self._workspace(x.device))

    def norm_finish(self, part, q, p):
        return gq.gq_norm_finish(part, q, p)

    def quantize_sum(self, x, norm, scheme, s, seed, step, worker0, sum_dtype):
        return gq.gq_quantize_sum(x, norm, scheme, s, seed, step, worker0=worker0,
                                  ws=self._workspace(x.device), sum_dtype=sum_dtype)

    def dequantize(self, sums, norm, scheme, s, n, out):
        return gq.gq_dequantize_sums(sums, norm, scheme, s, n, out=out)  # out: the bucket

    # the re-rounding allreduce of Global-E
    def quantize_codes(self, x, norm, scheme, s, seed, step, worker0):
        d = x.shape[1]
        codes = gq.gq_quantize_codes(x, norm, scheme, s, seed, step, worker0=worker0, code_bits=8,
                                     ws=self._workspace(x.device))
        return codes.view(torch.int8)[:d]

    def exp_combine(self, a, b, seed, step, stream_id, j0):
        return gq.gq_exp_combine(a, b, seed, step, stream_id, j0=j0)

    def exp_dequantize(self, codes, norm, s, n, out):
        return gq.gq_exp_dequantize(codes, norm, s, n, out=out)

    def exp_tree_stream(self, level, m):
        return gq.gq_exp_tree_stream(level, m)

    def exp_ring_stream(self, h, c):
        return gq.gq_exp_ring_stream(h, c)


@dataclass
class GlobalQSGDState:
    """Hook state: the quantiser, the norm order, the seed shared by all ranks and the
    iteration counter (advanced after the last bucket of each backward pass)."""

    scheme: int = gq.EXP
    s: int = 8
    q: int = gq.NORM_INF
    p: int = gq.NORM_INF
    seed: int = 0
    reduce: str = "sum"  # "sum" (exact integer sum); Global-E only: "tree" or "ring" (re-rounding)
    process_group: object = None
    ops: object = None
    step: int = 0
    buckets_seen: int = field(default=0, init=False)
    wire_dtype: object = field(default=None, init=False)  # int8 or int32, set from the world size

    def __post_init__(self):
        if (self.q, self.p) not in ((gq.NORM_INF, gq.NORM_INF), (gq.NORM_L2, gq.NORM_L2)):
            raise ValueError("the hook supports the norm orders (2, 2) and (inf, inf); the mixed "
                             "orders need a d-vector exchange")
        if gq.gq_code_bits(self.scheme, self.s) == 0:
            raise ValueError("unsupported quantiser: scheme %d, s %d" % (self.scheme, self.s))
        if not 0 <= self.seed < 2**64:
            raise ValueError("seed must fit 64 bits")
        if self.reduce not in ("sum", "tree", "ring"):
            raise ValueError("reduce must be 'sum', 'tree' or 'ring'")
        if self.reduce != "sum" and self.scheme != gq.EXP:
            raise ValueError("the re-rounding allreduce is Global-E's")
        n = self.world_size
        if self.reduce == "ring" and n > 4096:
            # ring step h of chunk c draws from stream 2^31 + 2^30 + h 2^12 + c: the chunk index
            # has 12 bits, so more ranks would give two steps the same random words
            raise ValueError("reduce='ring' supports at most 4096 ranks (world size %d)" % n)
        per_worker = self.s if self.scheme == gq.LINEAR else 1 << (self.s - 1)
        if n * per_worker >= 1 << 24:
            raise ValueError("world size %d x %d units per worker reaches 2^24: the integer sums "
                             "would not convert exactly" % (n, per_worker))
        # the narrowest integer type that holds the sum over all workers exactly
        self.wire_dtype = torch.int8 if n * per_worker <= 127 else torch.int32
        if self.ops is None:
            self.ops = LibraryOps()

    @property
    def world_size(self) -> int:
        return dist.get_world_size(self.process_group)

    @property
    def rank(self) -> int:
        return dist.get_rank(self.process_group)

    def bucket_step(self, index: int) -> int:
        if not 0 <= index < 1 << _STEP_BITS or self.step >= 1 << (64 - _STEP_BITS):
            raise ValueError("bucket index or iteration out of the random stream's range")
        return (self.step << _STEP_BITS) | index


def _peer(group, r):
    return r if group is None else dist.get_global_rank(group, r)


def _exp_tree(codes, state, step):
    """Recursive halving into rank 0 (row i a multiple of 2^l takes row i + 2^(l-1) at level l,
    re-rounding with stream tree(l, i >> l)), then a broadcast of the root's codes."""
    group, ops, rank, n = state.process_group, state.ops, state.rank, state.world_size
    acc = codes
    level = 1
    while (1 << (level - 1)) < n:
        half = 1 << (level - 1)
        if rank % (2 * half) == 0 and rank + half < n:
            other = torch.empty_like(acc)
            dist.recv(other, src=_peer(group, rank + half), group=group)
            acc = ops.exp_combine(acc, other, state.seed, step,
                                  ops.exp_tree_stream(level, rank >> level), 0)
        elif rank % (2 * half) == half:
            dist.send(acc, dst=_peer(group, rank - half), group=group)
        level += 1
    root = acc if rank == 0 else torch.empty_like(codes)
    dist.broadcast(root, src=_peer(group, 0), group=group)
    return root


def _exp_ring(codes, state, step):
    """Reduce-scatter: chunk c (ceil(d/n) rounded up to 16 coordinates) starts at worker c + 1
    and visits c + 2, ..., c, re-rounding at step h with stream ring(h, c); then an allgather."""
    group, ops, rank, n = state.process_group, state.ops, state.rank, state.world_size
    d = codes.numel()
    chunk = (-(-d // n) + 15) // 16 * 16
    bounds = [(min(d, c * chunk), min(d, (c + 1) * chunk)) for c in range(n)]
    held = (rank - 1) % n  # the chunk this rank starts
    lo, hi = bounds[held]
    acc = codes[lo:hi].clone()
    nxt, prv = _peer(group, (rank + 1) % n), _peer(group, (rank - 1) % n)
    for h in range(1, n):
        recv_c = (rank - h - 1) % n
        rlo, rhi = bounds[recv_c]
        buf = torch.empty(rhi - rlo, dtype=codes.dtype, device=codes.device)
        req = dist.isend(acc, dst=nxt, group=group) if acc.numel() else None
        if rhi > rlo:
            dist.recv(buf, src=prv, group=group)
        if req is not None:
            req.wait()
        acc = (ops.exp_combine(buf, codes[rlo:rhi].contiguous(), state.seed, step,
                               ops.exp_ring_stream(h, recv_c), rlo) if rhi > rlo else buf)
        held = recv_c
    # this rank now holds finished chunk `rank`; gather every chunk, padded to `chunk` codes
    padded = torch.zeros(chunk, dtype=codes.dtype, device=codes.device)
    padded[:acc.numel()] = acc
    parts = [torch.empty_like(padded) for _ in range(n)]
    dist.all_gather(parts, padded, group=group)
    return torch.cat([parts[c][:bounds[c][1] - bounds[c][0]] for c in range(n)])


def global_qsgd_hook(state: GlobalQSGDState, bucket) -> torch.futures.Future:
    """DDP communication hook: quantise, allreduce and dequantise one gradient bucket."""
    buf = bucket.buffer()
    if buf.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("Global-QSGD hook: gradients must be float32 or bfloat16, got %s" % buf.dtype)
    x = buf.view(1, -1)
    group = state.process_group
    ops = state.ops

    part = ops.norm_partial(x, state.q, state.p)
    red = dist.ReduceOp.SUM if state.q == gq.NORM_L2 else dist.ReduceOp.MAX
    dist.all_reduce(part, op=red, group=group)
    norm = ops.norm_finish(part, state.q, state.p)

    step = state.bucket_step(bucket.index())
    state.buckets_seen += 1
    if bucket.is_last():
        state.step += 1
    n = state.world_size
    if state.reduce != "sum":  # Global-E with re-rounding at every hop: int8 codes on the wire
        codes = ops.quantize_codes(x, norm, state.scheme, state.s, state.seed, step, state.rank)
        root = (_exp_tree if state.reduce == "tree" else _exp_ring)(codes, state, step)
        ops.exp_dequantize(root, norm, state.s, n, buf)
        done = torch.futures.Future()
        done.set_result(buf)
        return done

    sums = ops.quantize_sum(x, norm, state.scheme, state.s, state.seed, step, state.rank,
                            state.wire_dtype)
    fut = dist.all_reduce(sums, op=dist.ReduceOp.SUM, group=group, async_op=True).get_future()

    def finish(f):
        total = f.value()[0]
        ops.dequantize(total, norm, state.scheme, state.s, n, buf)  # in the bucket's own type
        return buf

    return fut.then(finish)


def register(model: torch.nn.parallel.DistributedDataParallel, **kwargs) -> GlobalQSGDState:
    """Attach the hook to a DDP model; keyword arguments go to GlobalQSGDState."""
    state = GlobalQSGDState(**kwargs)
    model.register_comm_hook(state, global_qsgd_hook)
    return state
