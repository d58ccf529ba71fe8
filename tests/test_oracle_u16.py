"""Pins of the oracle's 16-bit-uniform rounding mode (CPU only).

The mode rounds element x up iff H < F, H the high 16 bits of its Philox word and F a 16-bit
fraction of its grid position computed without a division (gqo_level_split_u16).  Pinned here
against what the mathematics fixes, independently of the oracle's own arithmetic:
  * its bias: over all 2^16 values of H (brute force), E[level] is within 2^-16 + 2^-22 of a level
    spacing of the exact position |x| / N (exact rationals), on random and constructed inputs
    of both grids, every s range, subnormal-free magnitudes and the grid's edges;
  * its agreement with the exact mode's split: the same lower level and F within 2 of T >> 16
    (the exact threshold's high half), away from level boundaries;
  * the decision rule: codes are sign (lo + [H < F]) with H from the published Philox word
    mapping; a tie H == F stays down, H == F - 1 rounds up (constructed exactly);
  * Monte-Carlo over steps: the dequantised mean agrees with the true mean within 5 sigma of the
    closed-form spread (the bias is far below that resolution);
  * zero stays zero, |x| = N is the top level, |x| > N saturates, NaN gives 0, norms outside
    [2^-100, 2^100] take the exact mode's decision.
"""
from fractions import Fraction

import numpy as np
import pytest

LINEAR, EXP = 0, 1
BOUND = Fraction(1, 2**16) + Fraction(1, 2**22)


def _pos(ax, N, scheme, s):
    """Exact position of |x| / N: (level value spacing, position in spacing units) for the
    interval of the grid it lies in; position = lower level + fraction."""
    v = Fraction(ax) / Fraction(N)
    if v > 1:
        v = Fraction(1)
    if scheme == LINEAR:
        return v * s
    first = Fraction(1, 2 ** (s - 1))
    if v < first:
        return v / first          # level 0 .. 1, spacing 2^-(s-1)
    e = 0
    while Fraction(2) ** (e + 1) <= v * 2 ** 62:
        e += 1
    e -= 62                        # 2^e <= v < 2^(e+1)
    return (s + e) + (v - Fraction(2) ** e) / Fraction(2) ** e


def _expected_level(lo, F):
    hits = sum(1 for h in range(0, 2**16, 1) if h < F)  # brute force over every H
    return lo + Fraction(hits, 2**16)


def _inputs(scheme, s, rng, k=200):
    out = []
    for N in (1.0, 1.5, 0.7431, 3.0e-5, 2.0e4, 0.48058903):
        N = float(np.float32(N))
        for _ in range(k // 6):
            u = rng.random()
            if scheme == EXP and rng.random() < 0.5:
                u = u * 2.0 ** -(s - 1) * 1.5   # around the first level
            out.append((float(np.float32(u * N)), N))
        out += [(0.0, N), (N, N), (float(np.float32(N / s)), N)]
    return out


@pytest.mark.parametrize("scheme,s", [(LINEAR, 1), (LINEAR, 7), (LINEAR, 127), (EXP, 1),
                                      (EXP, 4), (EXP, 8), (EXP, 24)])
def test_bias_bound_brute_force(oracle, scheme, s):
    rng = np.random.default_rng(100 + s + 7 * scheme)
    worst = Fraction(0)
    for ax, N in _inputs(scheme, s, rng):
        lo, F = oracle.level_split_u16(ax, N, scheme, s)
        got = _expected_level(lo, F)
        want = _pos(ax, N, scheme, s)
        if scheme == EXP and want >= 1 and got >= 1:
            # spacing of the binade: positions are in units of the interval [2^e, 2^(e+1))
            assert int(got) == int(want) or abs(got - want) <= BOUND
        err = abs(got - want)
        worst = max(worst, err)
        assert err <= BOUND, (ax, N, lo, F, float(err))
    assert worst > 0  # the mode is not the exact one: some resolution loss shows


@pytest.mark.parametrize("scheme,s", [(LINEAR, 15), (LINEAR, 127), (EXP, 8), (EXP, 4)])
def test_agrees_with_the_exact_split(oracle, scheme, s):
    rng = np.random.default_rng(7 + s)
    for ax, N in _inputs(scheme, s, rng):
        lo, F = oracle.level_split_u16(ax, N, scheme, s)
        lo_x, T = oracle.level_split(ax, N, scheme, s)
        a = lo * 2**16 + F
        b = lo_x * 2**16 + (T >> 16)
        assert abs(a - b) <= 2, (ax, N, lo, F, lo_x, T)


def test_decision_rule_and_ties(oracle):
    seed, step = 5, 0
    # Global-E under N = 1: w = |x| exactly, F = the top 16 fraction bits of |x|
    for i, j in ((0, 3), (1, 10), (0, 77), (2, 1000)):
        H = oracle.philox_word(seed, step, i, j) >> 16
        for F, want in ((H, 6), (H + 1, 7)):
            if F > 0xFFFF:
                continue
            x = np.zeros((3, 1001), dtype=np.float32)
            x[0, 0] = 1.0
            v = (1.0 + F / 2.0**16) * 0.25      # in [1/4, 1/2): lower level 8 - 2 = 6 under E_8
            x[i, j] = v
            assert oracle.level_split_u16(v, 1.0, EXP, 8) == (6, F)
            codes, rc = oracle.quantize_u16(x, np.float32(1.0), EXP, 8, seed, step)
            assert rc == 0 and codes[i, j] == want, (i, j, F, H)
    # every code of a random matrix follows sign (lo + [H < F])
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 70)).astype(np.float32)
    N = np.float32(np.abs(x).max())
    for scheme, s in ((LINEAR, 7), (EXP, 4)):
        codes, rc = oracle.quantize_u16(x, N, scheme, s, 9, 4)
        assert rc == 0
        for i in range(3):
            for j in range(70):
                lo, F = oracle.level_split_u16(float(x[i, j]), float(N), scheme, s)
                k = lo + ((oracle.philox_word(9, 4, i, j) >> 16) < F)
                assert codes[i, j] == (-k if x[i, j] < 0 else k)


def test_edges(oracle):
    N = 0.75
    assert oracle.level_split_u16(0.0, N, LINEAR, 7) == (0, 0)
    assert oracle.level_split_u16(0.0, N, EXP, 8) == (0, 0)
    assert oracle.level_split_u16(N, N, LINEAR, 7) == (7, 0)
    assert oracle.level_split_u16(N, N, EXP, 8) == (8, 0)
    assert oracle.level_split_u16(2 * N, N, LINEAR, 7) == (7, 0)   # saturates
    assert oracle.level_split_u16(2 * N, N, EXP, 8) == (8, 0)
    assert oracle.level_split_u16(float("nan"), N, LINEAR, 7) == (0, 0)
    assert oracle.level_split_u16(0.3, 2.0**-101, LINEAR, 7) is None   # exact mode applies
    assert oracle.level_split_u16(0.3, 2.0**101, EXP, 4) is None
    x = np.array([[0.3, -0.2, 0.0, 1e-30]], dtype=np.float32)
    for N in (np.float32(2.0**-101), np.float32(2.0**101)):
        a, rc = oracle.quantize_u16(x, N, LINEAR, 7, 1, 1)
        b, rc2 = oracle.quantize(x, N, LINEAR, 7, 1, 1)
        assert rc == rc2 == 0
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("scheme,s", [(LINEAR, 3), (EXP, 3)])
def test_monte_carlo_mean(oracle, scheme, s):
    rng = np.random.default_rng(11)
    n, d, steps = 2, 12, 6000
    x = (rng.random((n, d)) * 2 - 1).astype(np.float32)
    N = np.float32(np.abs(x).max())
    acc = np.zeros(d)
    for step in range(steps):
        codes, rc = oracle.quantize_u16(x, N, scheme, s, 21, step)
        sums = oracle.reduce_codes(codes, scheme, s)
        out, rc = oracle.dequantize(sums, N, scheme, s, n)
        acc += out
    mean = acc / steps
    want = x.astype(np.float64).mean(0)
    # per-element variance of one decision is at most spacing^2 / 4; the mean of n workers
    spacing = float(N) / s if scheme == LINEAR else float(N) * 0.5
    sigma = np.sqrt(n * (spacing ** 2 / 4) / n**2 / steps)
    assert np.all(np.abs(mean - want) <= 5 * sigma + 2 * float(BOUND) * spacing)
