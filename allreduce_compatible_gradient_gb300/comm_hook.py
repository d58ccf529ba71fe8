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


@dataclass
class GlobalQSGDState:
    """Hook state: the quantiser, the norm order, the seed shared by all ranks and the
    iteration counter (advanced after the last bucket of each backward pass)."""

    scheme: int = gq.EXP
    s: int = 8
    q: int = gq.NORM_INF
    p: int = gq.NORM_INF
    seed: int = 0
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
        n = self.world_size
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
    sums = ops.quantize_sum(x, norm, state.scheme, state.s, state.seed, step, state.rank,
                            state.wire_dtype)
    state.buckets_seen += 1
    if bucket.is_last():
        state.step += 1
    n = state.world_size
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
