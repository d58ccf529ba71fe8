"""Pins for the oracle's Global-E allreduce with re-rounding at every hop (CPU only).

The step being pinned: two extended Global-E codes are decoded to integer units of 2^-(s-1),
added, and the sum is rounded at random between the two powers of two around it.  Pins: exact
split points and thresholds worked by hand; E[step] = a + b exactly over both outcomes (the step
is unbiased); the code follows the split and the random word of its stream; Monte-Carlo means
of one step, of the tree and of the ring equal the exact sums; the tree and ring orders equal
their definitions written out step by step on small n; the ring, which rounds n - 1 times per
coordinate, has more variance than the tree, which rounds about log2 n times.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

TWO32 = 2**32


def test_split_units_by_hand(oracle):
    assert oracle.exp_split_units(0) == (0, 0)
    assert oracle.exp_split_units(1) == (1, 0)          # exactly level 1 (2^0 units)
    assert oracle.exp_split_units(8) == (4, 0)          # exactly level 4 (2^3 units)
    assert oracle.exp_split_units(3) == (2, 2**31)      # between 2 and 4: P(up) = 1/2
    assert oracle.exp_split_units(5) == (3, 2**30)      # between 4 and 8: P(up) = 1/4
    assert oracle.exp_split_units(-7) == (3, 3 * 2**30)  # |t| = 7: P(up) = 3/4
    assert oracle.exp_split_units(2**24 + 1) == (25, 2**8)


@pytest.mark.parametrize("t", [1, 2, 3, 6, 7, 9, 100, 1023, 1025, 65535, 2**20 + 12345, 2**23 - 1])
def test_step_expectation_is_the_sum(oracle, t):
    lo, T = oracle.exp_split_units(t)
    lo_v, hi_v = 2 ** (lo - 1), 2 ** lo
    mean = lo_v + Fraction(T, TWO32) * (hi_v - lo_v)
    assert mean == t                    # exact: the step adds no bias
    assert lo_v <= t < hi_v


def test_combine_follows_split_and_word(oracle):
    rng = np.random.default_rng(1)
    a = rng.integers(-9, 10, 200).astype(np.int8)
    b = rng.integers(-9, 10, 200).astype(np.int8)
    seed, step, sid = 12345, 6, oracle.exp_tree_stream(2, 3)
    out = oracle.exp_combine(a, b, seed, step, sid, j0=40)
    t = oracle.exp_units(a) + oracle.exp_units(b)
    for j in range(200):
        lo, T = oracle.exp_split_units(int(t[j]))
        k = lo + (1 if oracle.philox_word(seed, step, sid, 40 + j) < T else 0)
        assert out[j] == (-k if t[j] < 0 else k)
    assert ((out == 0) == (t == 0)).all()


def test_streams_are_distinct(oracle):
    ids = {oracle.exp_tree_stream(l, m) for l in range(1, 13) for m in range(64)}
    ids |= {oracle.exp_ring_stream(h, c) for h in range(1, 64) for c in range(64)}
    assert len(ids) == 12 * 64 + 63 * 64
    assert min(ids) >= 2**31  # above every worker index


def test_combine_monte_carlo(oracle):
    a = np.array([3, -2, 5, 7, 1, -4, 0, 6], dtype=np.int8)
    b = np.array([2, -3, -4, 7, 1, 4, 0, 1], dtype=np.int8)
    t = (oracle.exp_units(a) + oracle.exp_units(b)).astype(np.float64)
    M = 20000
    acc = np.zeros(8)
    for step in range(M):
        acc += oracle.exp_units(oracle.exp_combine(a, b, 7, step, oracle.exp_tree_stream(1, 0)))
    var = []
    for tv in t:
        lo, T = oracle.exp_split_units(int(tv))
        lo_v = 2 ** (lo - 1) if lo else 0
        var.append((2 * lo_v - abs(tv)) * (abs(tv) - lo_v) if lo else 0.0)
    for j in range(8):
        if var[j] == 0:
            assert acc[j] / M == t[j]
        else:
            assert abs(acc[j] / M - t[j]) < 5.5 * math.sqrt(var[j] / M)


def _tree_by_hand(oracle, rows, seed, step):
    # the definition written out: level by level, row i takes row i + 2^(l-1)
    u = [oracle.exp_units(r).astype(np.int64) for r in rows]
    codes = [np.asarray(r, dtype=np.int8) for r in rows]
    n = len(rows)
    l = 1
    while (1 << (l - 1)) < n:
        half, stride = 1 << (l - 1), 1 << l
        for i in range(0, n - half, stride):
            codes[i] = oracle.exp_combine(codes[i], codes[i + half], seed, step,
                                          oracle.exp_tree_stream(l, i >> l))
        l += 1
    return codes[0]


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 13])
def test_tree_matches_definition(oracle, n):
    rng = np.random.default_rng(n)
    rows = rng.integers(-8, 9, (n, 33)).astype(np.int8)
    got = oracle.exp_tree_allreduce(rows, 99, 5)
    np.testing.assert_array_equal(got, _tree_by_hand(oracle, list(rows), 99, 5))


@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_ring_matches_definition(oracle, n):
    rng = np.random.default_rng(10 + n)
    d = 29
    rows = rng.integers(-8, 9, (n, d)).astype(np.int8)
    got = oracle.exp_ring_allreduce(rows, d, 99, 5)
    chunk = -(-(-(-d // n)) // 16) * 16  # ceil(d / n) rounded up to a multiple of 16
    for j in range(d):
        c = j // chunk
        code = np.array([rows[(c + 1) % n, j]], dtype=np.int8)
        for h in range(1, n):
            nxt = np.array([rows[(c + 1 + h) % n, j]], dtype=np.int8)
            code = oracle.exp_combine(code, nxt, 99, 5, oracle.exp_ring_stream(h, c), j0=j)
        assert got[j] == code[0]


def test_tree_and_ring_are_unbiased_and_ring_noisier(oracle):
    rng = np.random.default_rng(4)
    n, d, M = 8, 16, 4000
    rows = rng.integers(-6, 7, (n, d)).astype(np.int8)
    exact = oracle.exp_units(rows).sum(axis=0).astype(np.float64)
    tree = np.empty((M, d))
    ring = np.empty((M, d))
    for step in range(M):
        tree[step] = oracle.exp_units(oracle.exp_tree_allreduce(rows, 3, step))
        ring[step] = oracle.exp_units(oracle.exp_ring_allreduce(rows, d, 3, step))
    for est in (tree, ring):
        sd = est.std(axis=0) + 1e-12
        z = (est.mean(axis=0) - exact) / (sd / math.sqrt(M))
        assert (np.abs(z) < 5.5).all()
    assert ring.var(axis=0).sum() > tree.var(axis=0).sum()
