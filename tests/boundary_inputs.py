"""Gradient matrices whose rounding decisions sit on or next to their boundary (test inputs).

The quantiser rounds element (i, j) up iff r < T, where r is the element's 32-bit Philox word and
T = floor(P(up) 2^32) follows from v = fp32(|x| / N) (the Global-Q operator: unbiased rounding
between the two adjacent levels of the Global-L or Global-E grid).  The CUDA kernels decide most
elements from a 16.16 fixed-point estimate of the grid position and the high 16 bits of r, and
fall back to the exact quotient and the full word when the estimate is within a few units of
2^-16 of the boundary.  These inputs exercise exactly that: for chosen elements |x| is picked so
that T - r takes a prescribed offset: 0 (a tie, which stays down), +-1, +-2^15, and around
+-1, 2, 3 and 4 times 2^16 (the edges of the 16-bit window), each on a random level.

Everything here runs on the CPU and uses only the oracle (its Philox words and its level split):
no value comes from the CUDA path.  The rest of the matrix is seeded noise below the norm.
"""
from __future__ import annotations

import numpy as np

from oracle import gq_oracle as oracle

LINEAR, EXP = 0, 1
INF = 0
W16 = 1 << 16

# offsets T - r that the construction aims at (the ones reachable at the element's precision
# are hit exactly; the others as closely as fp32 / bf16 allow)
DELTAS = (0, 1, -1, 2, -2, 1 << 15, -(1 << 15), W16, -W16, W16 + 1, -W16 - 1, W16 - 1,
          -W16 + 1, 2 * W16, -2 * W16, 2 * W16 + 1, -2 * W16 - 1, 3 * W16, -3 * W16, 4 * W16,
          -4 * W16)


def words(n: int, d: int, seed: int, step: int, worker0: int = 0, col0: int = 0) -> np.ndarray:
    """n x d matrix of the oracle's random words r (uint32), worker worker0 + i, column col0 + j."""
    return np.stack([oracle.philox_words(seed, step, worker0 + i, col0, d) for i in range(n)])


def _target_abs(m: int, T: int, scheme: int, s: int, N: float) -> float:
    """|x| (as a real number) for which the lower level is m and P(up) 2^32 = T exactly."""
    f = T / 2.0**32
    if scheme == LINEAR:
        v = (m + f) / s
    elif m == 0:
        v = f * 2.0 ** -(s - 1)       # between 0 and the lowest level 2^-(s-1)
    else:
        v = 2.0 ** (m - s) * (1.0 + f)  # between 2^-(s-m) and twice that
    return v * float(N)


def _neighbours(x0: float, dtype: str, k: int) -> list:
    """Representable positive values of the element type around x0 (k steps each way)."""
    if dtype == "bf16":
        b0 = int(_bf16_bits(np.float32(x0))[0])
        bits = [b0 + t for t in range(-k, k + 1) if 0 < b0 + t < 0x7F80]
        return [float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0]) for b in bits]
    b0 = int(np.array([x0], dtype=np.float32).view(np.uint32)[0])
    bits = [b0 + t for t in range(-k, k + 1) if 0 < b0 + t < 0x7F800000]
    return [float(v) for v in np.array(bits, dtype=np.uint32).view(np.float32)]


def _bf16_bits(a) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even."""
    b = np.atleast_1d(np.asarray(a, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def place(absx_target: float, m: int, r: int, delta: int, scheme: int, s: int, N: float,
          dtype: str, cap: float | None, k: int):
    """The representable |x| near absx_target whose split (lo, T) has lo == m and T - r closest
    to delta; (|x|, achieved T - r) or None.  cap: largest |x| allowed (the max norm)."""
    best = None
    for c in _neighbours(absx_target, dtype, k):
        if cap is not None and c > cap:
            continue
        lo, T = oracle.level_split(c, float(N), scheme, s)
        if lo != m:
            continue
        got = T - r
        if best is None or abs(got - delta) < abs(best[1] - delta):
            best = (c, got)
    return best


def background(n: int, d: int, rng, scale: float, dtype: str) -> np.ndarray:
    """Seeded N(0, scale^2) noise as float32 (bf16-representable for dtype bf16)."""
    x = (rng.standard_normal((n, d)) * scale).astype(np.float32)
    if dtype == "bf16":
        x = (_bf16_bits(x).astype(np.uint32) << 16).view(np.float32).reshape(n, d)
    return x


def to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 matrix (bf16-representable for bf16) -> the array the oracle and GPU take."""
    if dtype == "bf16":
        return np.ascontiguousarray((x.view(np.uint32) >> 16).astype(np.uint16))
    return np.ascontiguousarray(x)


def levels_for(scheme: int, s: int, rng, small_norm: bool) -> int:
    """A random lower level: any level below the top, or (small_norm: Global-E under the l2 norm
    of all elements, where |x| / N is small) almost always level 0, a few at levels 1 and 2 (few
    enough that the placed elements barely move the norm they are placed for)."""
    if small_norm and scheme == EXP:
        return int(rng.choice([0, 1, 2], p=[0.985, 0.01, 0.005]))
    return int(rng.integers(0, s))


def tie_offsets(R: np.ndarray, scheme: int, s: int) -> np.ndarray:
    """For every word r, the offset delta in {0, -1, +1} for which a threshold T = r + delta is
    exactly reachable, else 2 (none).  Global-E thresholds are the fraction bits of v shifted
    left by 9, so T is any multiple of 512.  Global-L below the first level has T = v s 2^32
    exactly; with v = M 2^-32 (M even, 2^23 <= M < 2^24, so that |x| = 1.5 v is exact too) T is
    any multiple of 4s in [s 2^23, s 2^24)."""
    r = R.astype(np.int64)
    out = np.full(R.shape, 2, dtype=np.int64)
    if scheme == EXP:
        lb = r & 0x1FF
        out[lb == 0] = 0
        out[lb == 1] = -1
        out[lb == 0x1FF] = 1
        return out
    q = 4 * s
    ok = (r >= (s << 23) + 1) & (r < (s << 24) - 1)
    rem = r % q
    out[ok & (rem == 0)] = 0
    out[ok & (rem == 1)] = -1
    out[ok & (rem == q - 1)] = 1
    return out


def make_plan(R: np.ndarray, count: int, scheme: int, s: int, rng, small_norm: bool = False,
              dtype: str = "f32"):
    """Which elements to place and how: positions (flat indices), aimed offsets T - r, lower
    levels and signs.  Up to a quarter of the positions are ones whose word admits an exact tie
    or its neighbours (tie_offsets) and take that offset; the rest take random offsets from
    DELTAS.  bf16 elements have 8 significant bits, so their thresholds are far apart: for them
    the plan is a pool of 24 x count positions aimed at T = r, of which build() keeps those that
    land within the window."""
    n, d = R.shape
    flat = rng.permutation(n * d)
    if dtype == "bf16":
        positions = np.sort(flat[: min(n * d, 24 * count)])
        # Global-L: bf16 steps move v s by up to 2^-7 of itself, so only the low levels have
        # thresholds close together
        levels = [int(rng.integers(0, min(s, 3))) if scheme == LINEAR
                  else levels_for(scheme, s, rng, small_norm) for _ in positions]
        return {"positions": positions, "deltas": np.zeros(len(positions), dtype=np.int64),
                "levels": np.array(levels),
                "signs": np.where(rng.random(len(positions)) < 0.5, -1.0, 1.0),
                "keep_within": 5 * W16, "limit": count}
    tdel = tie_offsets(R, scheme, s).ravel()
    tie = flat[tdel[flat] != 2][: count // 4]
    positions = np.unique(np.concatenate([tie, flat[:count]]))[:count]
    deltas, levels = [], []
    for p in positions:
        t = int(tdel[p])
        deltas.append(t if t != 2 else int(rng.choice(DELTAS)))
        # Global-L ties exist only below the first level (see tie_offsets)
        levels.append(0 if t != 2 and scheme == LINEAR else levels_for(scheme, s, rng, small_norm))
    signs = np.where(rng.random(len(positions)) < 0.5, -1.0, 1.0)
    return {"positions": positions, "deltas": np.array(deltas, dtype=np.int64),
            "levels": np.array(levels), "signs": signs}


def make_plan_l2(R: np.ndarray, count: int, scheme: int, s: int, rng, dtype: str = "f32",
                 budget: float = 0.04):
    """make_plan for the (2, 2) norm, where every |x| / N counts towards N: the placed elements
    keep sum (|x| / N)^2 below `budget`, so that they move the norm little.  Level-0 elements
    (v below the first level, T = v u 2^32 with u = s for Global-L and 2^(s-1) for Global-E) go
    to positions whose word is small enough that v stays below sqrt(budget / 2 / count); for
    Global-E a few elements go to levels 1 and 2 (v of 2^-(s-1) and more) as long as the budget
    allows (a Global-L level of 1 or more is v >= 1/s, too large for it)."""
    n, d = R.shape
    v0 = np.sqrt(budget / 2 / count)
    unit = float(s) if scheme == LINEAR else 2.0 ** (s - 1)
    rmax = min(2.0**32 - 1, v0 * unit * 2.0**32)
    flat = rng.permutation(n * d)
    small = flat[R.ravel()[flat] < rmax]
    tdel = tie_offsets(R, scheme, s).ravel()
    if dtype == "bf16":
        positions = np.sort(small[: 24 * count])
        deltas = np.zeros(len(positions), dtype=np.int64)
    else:
        tie = small[tdel[small] != 2][: count // 4]
        positions = np.unique(np.concatenate([tie, small[:count]]))[:count]
        deltas = np.array([int(tdel[p]) if tdel[p] != 2 else int(rng.choice(DELTAS))
                           for p in positions], dtype=np.int64)
    levels = np.zeros(len(positions), dtype=np.int64)
    left = budget / 2
    for m in ((1, 2) if scheme == EXP else ()):  # level m: v in [2^(m-s), 2^(m-s+1))
        k = int(left / 2 / 4.0 ** (m - s + 1))
        k = min(k, 64, len(positions) // 8)
        idx = rng.choice(len(positions), size=k, replace=False) if k else []
        levels[idx] = m
        left -= k * 4.0 ** (m - s + 1)
    plan = {"positions": positions, "deltas": deltas, "levels": levels,
            "signs": np.where(rng.random(len(positions)) < 0.5, -1.0, 1.0)}
    if dtype == "bf16":
        plan.update(keep_within=5 * W16, limit=count)
    return plan


def build(base: np.ndarray, R: np.ndarray, plan: dict, scheme: int, s: int, N: float,
          dtype: str = "f32", capped: bool = True):
    """Place the plan's elements into a copy of `base` (n x d float32) for the norm N.
    Returns (x float32, info) with the placed positions, the aimed and the achieved T - r."""
    n, d = base.shape
    x = np.array(base, dtype=np.float32, copy=True)
    cap = float(N) if capped else None
    k = 2 if dtype == "bf16" else 24
    pos_out, aimed, got = [], [], []
    keep, limit = plan.get("keep_within"), plan.get("limit")
    for p, delta, m, sg in zip(plan["positions"], plan["deltas"], plan["levels"],
                               plan["signs"]):
        if limit is not None and len(pos_out) >= limit:
            break
        i, j = divmod(int(p), d)
        r = int(R[i, j])
        T = r + int(delta)
        if not 0 <= T < 2**32 or (scheme == EXP and m == 0 and s == 1):
            continue
        hit = place(_target_abs(int(m), T, scheme, s, N), int(m), r, int(delta), scheme, s, N,
                    dtype, cap, k)
        if hit is None or (keep is not None and abs(hit[1]) > keep):
            continue
        x[i, j] = hit[0] * sg
        pos_out.append(int(p))
        aimed.append(int(delta))
        got.append(hit[1])
    info = {"positions": np.array(pos_out, dtype=np.int64), "aimed": np.array(aimed),
            "achieved": np.array(got, dtype=np.int64), "N": float(N)}
    return x, info


def max_norm_matrix(n: int, d: int, scheme: int, s: int, seed: int, step: int, count: int,
                    rng, dtype: str = "f32", worker0: int = 0, col0: int = 0, N: float = 1.5,
                    worst: int = 0):
    """Boundary inputs under the max norm: an anchor element equal to N (v = 1 exactly, the top
    level) fixes ||x||_{inf,inf} = N and every other |x| stays at or below it.  worst: that many
    elements from worst_error_elements as well (Global-L, fp32)."""
    N = float(np.float32(N)) if dtype == "f32" else float(
        (_bf16_bits(np.float32(N)).astype(np.uint32) << 16).view(np.float32)[0])
    base = background(n, d, rng, 0.2 * N, dtype)
    np.clip(base, -N, N, out=base)
    R = words(n, d, seed, step, worker0, col0)
    plan = make_plan(R, count, scheme, s, rng, dtype=dtype)
    x, info = build(base, R, plan, scheme, s, N, dtype, True)
    if worst and scheme == LINEAR and dtype == "f32":
        info["worst"] = worst_error_elements(x, R, N, s, rng, worst, info["positions"])
    taken = set(info["positions"].tolist()) | set(info.get("worst", np.zeros(0)).tolist())
    a = next(int(p) for p in rng.permutation(n * d) if int(p) not in taken)
    x.ravel()[a] = N if rng.random() < 0.5 else -N
    info["anchor"] = a
    return to_dtype(x, dtype), info


def supplied_norm_matrix(n: int, d: int, scheme: int, s: int, seed: int, step: int,
                         count: int, rng, N: float, dtype: str = "f32", worker0: int = 0):
    """Boundary inputs for a norm handed in from outside (N need not be any |x|): besides the
    placed elements, a few |x| equal to N (v = 1) and a few just above it (v clamps to 1).  For
    bf16 gradients N is rounded to bf16 first, so that |x| = N is representable."""
    N = float(np.float32(N))
    if dtype == "bf16":
        N = float((_bf16_bits(np.float32(N)).astype(np.uint32) << 16).view(np.float32)[0])
    base = background(n, d, rng, 0.2 * N, dtype)
    np.clip(base, -N, N, out=base)
    R = words(n, d, seed, step, worker0)
    plan = make_plan(R, count, scheme, s, rng, dtype=dtype)
    x, info = build(base, R, plan, scheme, s, N, dtype, True)
    extra = rng.choice(n * d, size=16, replace=False)
    above = _neighbours(N, dtype, 3)
    for t, a in enumerate(extra):
        v = N if t % 2 == 0 else max(c for c in above if c > N) if any(c > N for c in above) else N
        x.ravel()[a] = v * (1.0 if t % 4 < 2 else -1.0)
    info["saturated"] = extra
    return to_dtype(x, dtype), info


def l2_norm_matrix(n: int, d: int, scheme: int, s: int, seed: int, step: int, count: int,
                   rng, dtype: str = "f32", q: int = 2, p: int = 2, rounds: int = 8):
    """Boundary inputs under a norm computed from the data (the l2 forms): placed for the
    oracle's fp32 norm of the matrix they end up in, found by iterating placement and norm
    until the norm no longer moves (or `rounds` iterations)."""
    base = background(n, d, rng, 1.0, dtype)
    R = words(n, d, seed, step)
    if (q, p) == (2, 2):
        plan = make_plan_l2(R, count, scheme, s, rng, dtype)
    else:
        plan = make_plan(R, count, scheme, s, rng, dtype=dtype)
    N = np.float32(oracle.global_norm(to_dtype(base, dtype), q, p))
    converged = False
    for _ in range(rounds):
        x, info = build(base, R, plan, scheme, s, float(N), dtype, True)
        if "keep_within" in plan:  # bf16: keep the positions that landed, aim them again
            sel = np.isin(plan["positions"], info["positions"])
            plan = {k: plan[k][sel] for k in ("positions", "deltas", "levels", "signs")}
        N2 = np.float32(oracle.global_norm(to_dtype(x, dtype), q, p))
        if N2 == N:
            converged = True
            break
        N = N2
    info["N"] = float(N)
    info["converged"] = converged
    return to_dtype(x, dtype), info


def achieved_offsets(xa: np.ndarray, info: dict, N: float, scheme: int, s: int, seed: int,
                     step: int, worker0: int = 0, col0: int = 0) -> np.ndarray:
    """T - r of the placed elements under the norm N actually used (the oracle's split)."""
    n, d = xa.shape
    out = []
    for p in info["positions"]:
        i, j = divmod(int(p), d)
        v = xa[i, j]
        if xa.dtype == np.uint16:
            v = np.array([int(v) << 16], dtype=np.uint32).view(np.float32)[0]
        lo, T = oracle.level_split(abs(float(v)), float(N), scheme, s)
        out.append(T - oracle.philox_word(seed, step, worker0 + i, col0 + j))
    return np.array(out, dtype=np.int64)


def worst_error_elements(x: np.ndarray, R: np.ndarray, N: float, s: int, rng, count: int,
                         exclude=()) -> np.ndarray:
    """Global-L: place up to `count` elements (in place, into the float32 matrix x) whose fast
    16.16 estimate lies more than one unit of 2^-16 below the exact grid position, at positions
    whose word r puts the estimate one unit below the window's top half (low half of y =
    0xFFFC) while the exact decision rounds up (r < T).  A kernel whose certainty window lacked
    that low value would decide these elements wrong.  Such estimates need a norm whose RN(s / N)
    is off by nearly half a unit and a level near the top (v in [1/2, 1)); N = 0.48058903 is one.
    Returns the flat positions used."""
    from fast_path_model import C0_BITS, estimate_error

    n, d = x.shape
    N32 = np.float32(N)
    ax = (rng.uniform(0.5, 1.0, 400_000) * N32).astype(np.float32)
    ax = ax[ax <= N32]
    pool = ax[estimate_error(ax, N32, s) < -1.0]
    c1 = np.float32(np.float32(s) / N32)
    c0 = np.array([C0_BITS], dtype=np.uint32).view(np.float32)[0]
    pb = (pool.astype(np.float64) * np.float64(c1) + np.float64(c0)).astype(np.float32)
    frac = (pb.view(np.uint32).astype(np.int64) - 0x43000000 - 0xFFFD) & 0xFFFF
    Rf = R.ravel().astype(np.int64)
    order = np.argsort(Rf >> 16, kind="stable")
    hs = (Rf >> 16)[order]
    used = set(int(e) for e in exclude)
    out = []
    for a, f in zip(pool, frac):
        if len(out) >= count:
            break
        need = (int(f) + 1) & 0xFFFF
        lo_i, hi_i = np.searchsorted(hs, need), np.searchsorted(hs, need, side="right")
        _, T = oracle.level_split(float(a), float(N32), LINEAR, s)
        cand = [int(p) for p in order[lo_i:hi_i] if Rf[p] < T and int(p) not in used]
        if not cand:
            continue
        p = cand[int(rng.integers(0, len(cand)))]
        used.add(p)
        x.ravel()[p] = float(a) * (1.0 if rng.random() < 0.5 else -1.0)
        out.append(p)
    return np.array(out, dtype=np.int64)
