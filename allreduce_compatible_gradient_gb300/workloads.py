"""Seeded synthetic gradient generators for the Global-QSGD workloads (inputs only).

This module holds none of the method's arithmetic: it only makes n x d gradient matrices with
the shapes and value distributions of the workloads the method is evaluated on (gradients of
ResNet-50 and BERT-sized models trained data-parallel by n workers).  Both the test suite (which
feeds the same buffers to the CUDA library and to the CPU oracle) and bench.py use it.

Host generators use numpy (small cases); device generators use torch on the GPU (full sizes,
generated in row chunks so temporaries stay small).
"""
from __future__ import annotations

import numpy as np

LINEAR, EXP = 0, 1
NORM_INF, NORM_L2 = 0, 2


def resnet50_layer_sizes() -> list:
    """Parameter tensor sizes of ResNet-50 in module-registration order (161 tensors).

    Stem 7x7 conv 3->64 and its batch-norm weight and bias; four bottleneck stages of
    [3, 4, 6, 3] blocks with widths 64/128/256/512 and expansion 4 (1x1, 3x3, 1x1 convs, each
    followed by a batch-norm weight and bias; the first block of a stage adds a 1x1 downsample
    conv and batch norm); the 2048 x 1000 classifier and its bias.
    """
    sizes = [7 * 7 * 3 * 64, 64, 64]
    c_in = 64
    for width, blocks in zip((64, 128, 256, 512), (3, 4, 6, 3)):
        for b in range(blocks):
            src = c_in if b == 0 else 4 * width
            sizes += [src * width, width, width,
                      9 * width * width, width, width,
                      width * 4 * width, 4 * width, 4 * width]
            if b == 0:
                sizes += [c_in * 4 * width, 4 * width, 4 * width]
        c_in = 4 * width
    sizes += [2048 * 1000, 1000]
    assert len(sizes) == 161 and sum(sizes) == 25_557_032
    return sizes


def ddp_buckets(sizes, elem_bytes: int = 4, cap_bytes: int = 25 << 20,
                first_cap_bytes: int = 1 << 20) -> list:
    """Gradient buckets as PyTorch DDP forms them: parameters taken in reverse registration
    order (the order their gradients become ready), a bucket closed once it holds at least its
    cap (1 MiB for the first, 25 MiB after); returns the buckets' sizes in elements."""
    out, cur, cap = [], 0, first_cap_bytes
    for sz in reversed(list(sizes)):
        cur += sz
        if cur * elem_bytes >= cap:
            out.append(cur)
            cur, cap = 0, cap_bytes
    if cur:
        out.append(cur)
    return out


def segment_tensors(n: int, sizes, dtype: str = "f32", seed: int = 0, device="cuda"):
    """One n x d_l gradient matrix per segment, carved from a single allocation with every
    segment starting on a 16-byte boundary; values N(0, sigma_l^2) with sigma_l log-uniform in
    [1e-4, 1e-1] per segment (per-layer gradient scales differ by orders of magnitude)."""
    import torch

    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    align = 16 // (2 if dtype == "bf16" else 4)
    offs, off = [], 0
    for sz in sizes:
        offs.append(off)
        off += (n * sz + align - 1) // align * align
    buf = torch.empty(max(off, 1), dtype=tdt, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    sig = 10.0 ** np.random.default_rng(seed).uniform(-4, -1, size=len(sizes))
    segs = []
    for o, sz, sg in zip(offs, sizes, sig):
        t = buf[o:o + n * sz].view(n, sz)
        t.normal_(0.0, float(sg), generator=g)
        segs.append(t)
    return segs


# Workloads: the four fixed cases and the sweep.  Philox seed 1, step 0 unless stated.
CONFIGS = {
    "gauss_n4_d65536": dict(n=4, d=65_536, dtype="f32", dist="normal", scheme=LINEAR, s=15,
                            q=NORM_L2, p=NORM_L2, seed=1, step=0, input_seed=0),
    "resnet50_n8": dict(n=8, d=25_557_032, dtype="f32", dist="resnet50", scheme=LINEAR, s=127,
                        q=NORM_INF, p=NORM_INF, seed=1, step=0, input_seed=0),
    "bert_base_n8_bf16": dict(n=8, d=110_000_000, dtype="bf16", dist="student_t3",
                              scheme=EXP, s=8, q=NORM_L2, p=NORM_L2, seed=1, step=0,
                              input_seed=0),
    "bert_large_n16_sparse": dict(n=16, d=350_000_000, dtype="f32", dist="laplace_block_sparse",
                                  scheme=EXP, s=4, q=NORM_L2, p=NORM_INF, seed=1, step=0,
                                  input_seed=0),
}
SWEEP_N = (2, 4, 8, 16, 32, 64)
SWEEP_D = tuple(2**k for k in (20, 22, 24, 26, 28))
SWEEP_SCHEMES = ((LINEAR, 7), (EXP, 4))


def sweep_points(max_bytes: float = 120e9):
    for n in SWEEP_N:
        for d in SWEEP_D:
            if n * d * 4 > max_bytes:
                continue
            for scheme, s in SWEEP_SCHEMES:
                yield dict(n=n, d=d, dtype="f32", dist="normal", scheme=scheme, s=s,
                           q=NORM_L2, p=NORM_L2, seed=1, step=0, input_seed=0)


def sparse_block_mask(d: int, seed: int, block: int = 4096) -> np.ndarray:
    """Boolean mask over the ceil(d/4096) coordinate blocks: exactly floor(nb/2) blocks, chosen
    by a seeded permutation, are zeroed for every worker (sparse layers)."""
    nb = -(-d // block)
    rng = np.random.default_rng(seed + 7919)
    zero = np.zeros(nb, dtype=bool)
    zero[rng.permutation(nb)[: nb // 2]] = True
    return zero


def _round_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def host_inputs(dist: str, n: int, d: int, seed: int = 0, dtype: str = "f32") -> np.ndarray:
    """n x d gradients on the host: float32, or bf16 bit patterns (uint16) for dtype "bf16"."""
    rng = np.random.default_rng(seed)
    if dist == "normal":
        x = rng.standard_normal((n, d), dtype=np.float32)
    elif dist == "resnet50":
        x = np.empty((n, d), dtype=np.float32)
        sizes = _layer_split(d)
        sig = 10.0 ** rng.uniform(-4, -1, size=len(sizes))
        off = 0
        for sz, sg in zip(sizes, sig):
            x[:, off:off + sz] = rng.standard_normal((n, sz), dtype=np.float32) * np.float32(sg)
            off += sz
    elif dist == "student_t3":
        x = (rng.standard_t(3, size=(n, d)) * 1e-3).astype(np.float32)
    elif dist == "laplace_block_sparse":
        x = rng.laplace(0.0, 1e-3, size=(n, d)).astype(np.float32)
        zero = sparse_block_mask(d, seed)
        cols = np.repeat(zero, 4096)[:d]
        x[:, cols] = 0.0
    else:
        raise ValueError(dist)
    if dtype == "bf16":
        return _round_bf16_bits(x)
    return np.ascontiguousarray(x)


def _layer_split(d: int) -> list:
    """ResNet-50 layer sizes when d is the full model; otherwise the same proportions."""
    sizes = resnet50_layer_sizes()
    if d == sum(sizes):
        return sizes
    cuts = np.round(np.cumsum(sizes) / sum(sizes) * d).astype(np.int64)
    out = np.diff(np.concatenate([[0], cuts])).tolist()
    return [int(v) for v in out if v > 0] or [d]


def device_inputs(dist: str, n: int, d: int, seed: int = 0, dtype: str = "f32", device="cuda"):
    """n x d gradients generated on the GPU with a seeded torch generator (full sizes)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = torch.empty((n, d), dtype=tdt, device=device)
    chunk = max(1, min(d, 1 << 26))
    if dist == "resnet50":
        sizes = _layer_split(d)
        sig = torch.tensor(10.0 ** np.random.default_rng(seed).uniform(-4, -1, size=len(sizes)),
                           dtype=torch.float32)
        for i in range(n):
            off = 0
            for sz, sg in zip(sizes, sig.tolist()):
                out[i, off:off + sz].normal_(0.0, sg, generator=g)
                off += sz
        return out
    for i in range(n):
        for j0 in range(0, d, chunk):
            j1 = min(d, j0 + chunk)
            w = j1 - j0
            if dist == "normal":
                v = torch.randn(w, generator=g, device=device)
            elif dist == "student_t3":
                z = torch.randn(w, generator=g, device=device)
                chi = torch.randn((3, w), generator=g, device=device).square_().sum(0)
                v = z / torch.sqrt(chi.clamp_(min=1e-30) / 3.0) * 1e-3
            elif dist == "laplace_block_sparse":
                u = torch.rand(w, generator=g, device=device) - 0.5
                a = (2.0 * u.abs()).clamp_(max=1.0 - 2.0**-24)  # keeps the log finite
                v = -1e-3 * torch.sign(u) * torch.log1p(-a)
            else:
                raise ValueError(dist)
            out[i, j0:j1] = v.to(tdt)
    if dist == "laplace_block_sparse":
        zero = torch.from_numpy(np.repeat(sparse_block_mask(d, seed), 4096)[:d]).to(device)
        out[:, zero] = 0
    return out


def config_bytes(cfg: dict) -> int:
    """Bytes of gradient input n * d * element size."""
    return cfg["n"] * cfg["d"] * (2 if cfg["dtype"] == "bf16" else 4)


def fused_algorithmic_bytes(cfg: dict) -> int:
    """Minimum traffic of the fused path: x read twice (norm pass, quantise pass), out written."""
    return 2 * config_bytes(cfg) + 4 * cfg["d"]

