"""Pins for the oracle's stochastic rounding, code sum and dequantisation (CPU only).

What pins what (no reference implementation exists, so every pin is a property the definitions
fix, a hand-derived example or brute force):
  * the hand-worked example in tests/golden/worked_example.txt (level indices, signs, the
    round-up rule, the E decoding and both dequantisation scales);
  * brute force over every up/down outcome on tiny inputs: E[out] equals the mean gradient and
    the variance equals the closed form (unbiasedness of the Global-Q operator);
  * Monte-Carlo over training steps through the real Philox-driven path: z-tests on the mean and
    the variance of the sum (fails if workers or steps share random words);
  * the variance and sparsity bounds re-derived for both grids, on the closed form;
  * fixed points: inputs exactly on a level give the same code for every seed;
  * the n = 1 reduction (codes do not depend on q; equal to QSGD with the local norm).
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

INF = 0
LINEAR, EXP = 0, 1
TWO32 = 2**32
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.txt")


def level_value(scheme, s, k):
    """Value of level index k: k/s (Global-L_s) or 0, 2^-(s-k) (Global-E_s)."""
    if scheme == LINEAR:
        return Fraction(k, s)
    return Fraction(0) if k == 0 else Fraction(1, 2 ** (s - k))


def v32(x, norm):
    v = np.float32(np.abs(np.float32(x)) / np.float32(norm))
    return min(v, np.float32(1.0))


# ----------------------------------------------------------------------------------------------
# hand-worked example
# ----------------------------------------------------------------------------------------------

def _golden():
    recs = {}
    x = None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, *rest = [part.split() for part in line.split("|")]
            if head[0] == "x":
                x = np.array([[float(t) for t in head[1:]], [float(t) for t in rest[0]]],
                             dtype=np.float32)
                continue
            scheme = LINEAR if head[0] == "linear" else EXP
            s = int(head[1])
            recs[(scheme, s)] = dict(
                codes=np.array([[int(t) for t in rest[0]], [int(t) for t in rest[1]]]),
                sums=np.array([int(t) for t in rest[2]]),
                out=np.array([float(t) for t in rest[3]]))
    return x, recs


def test_worked_example(oracle):
    x, recs = _golden()
    assert len(recs) == 2
    for (scheme, s), want in recs.items():
        r = oracle.allreduce_mean(x, INF, INF, scheme, s, seed=0, step=0)
        assert r["rc"] == 0
        assert r["norm32"] == 1.0
        np.testing.assert_array_equal(r["codes"], want["codes"])
        np.testing.assert_array_equal(r["sums"], want["sums"])
        np.testing.assert_array_equal(r["out"], want["out"])


# ----------------------------------------------------------------------------------------------
# level split: the grid and the round-up threshold
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("scheme,s", [(LINEAR, 1), (LINEAR, 7), (LINEAR, 127), (EXP, 1), (EXP, 4),
                                      (EXP, 8), (EXP, 24)])
def test_level_split_brackets_v_and_is_unbiased(oracle, scheme, s):
    rng = np.random.default_rng(s + 1000 * scheme)
    norm = np.float32(3.75)
    xs = np.concatenate([
        rng.uniform(0, 3.75, 400), np.exp(rng.uniform(-60, 1.3, 400)),
        [0.0, 3.75, 1e-45, 3.75 / 2, 3.75 / 4]]).astype(np.float32)
    for a in xs:
        lo, T = oracle.level_split(float(a), float(norm), scheme, s)
        v = Fraction(float(v32(a, norm)))
        assert 0 <= lo <= s
        lo_val = level_value(scheme, s, lo)
        assert lo_val <= v
        if lo == s:
            assert v == 1 and T == 0
            continue
        hi_val = level_value(scheme, s, lo + 1)
        assert v < hi_val
        # E[xi(v)] = lo + P(up) (hi - lo) equals v up to the 2^-32 resolution of T
        mean = lo_val + Fraction(T, TWO32) * (hi_val - lo_val)
        assert 0 <= v - mean < (hi_val - lo_val) / TWO32


def test_level_split_fixed_points(oracle):
    norm = 2.0
    for s in (1, 3, 15, 127):
        for m in range(s + 1):
            a = np.float32(norm * m / s)
            if float(v32(a, norm)) * s != m:
                continue  # m/s not representable: not a fixed point in fp32
            assert oracle.level_split(float(a), norm, LINEAR, s) == (m, 0)
    for s in (1, 4, 8, 24):
        assert oracle.level_split(0.0, norm, EXP, s) == (0, 0)
        for k in range(1, s + 1):
            a = norm * 2.0 ** -(s - k)
            assert oracle.level_split(a, norm, EXP, s) == (k, 0)


def test_level_split_clamps_above_norm(oracle):
    assert oracle.level_split(5.0, 2.0, LINEAR, 9) == (9, 0)
    assert oracle.level_split(5.0, 2.0, EXP, 6) == (6, 0)


def test_exponential_threshold_is_the_mantissa(oracle):
    # v in [2^e, 2^(e+1)): P(up) = v / 2^e - 1 is the 23-bit fraction of v, T = fraction << 9
    rng = np.random.default_rng(4)
    for v in rng.uniform(2.0**-7, 1.0, 500).astype(np.float32):
        lo, T = oracle.level_split(float(v), 1.0, EXP, 8)
        bits = int(np.array(v, dtype=np.float32).view(np.uint32))
        assert T == (bits & 0x7FFFFF) << 9
        assert lo == 8 + ((bits >> 23) - 127)


# ----------------------------------------------------------------------------------------------
# codes come from the level split and the Philox word
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("scheme,s", [(LINEAR, 15), (EXP, 8)])
def test_codes_follow_split_and_word(oracle, scheme, s):
    rng = np.random.default_rng(17)
    x = rng.standard_normal((3, 23)).astype(np.float32)
    norm = np.float32(oracle.global_norm(x, 2, 2))
    seed, step = 0x123456789ABCDEF0, 77
    codes, rc = oracle.quantize(x, norm, scheme, s, seed, step)
    assert rc == 0
    for i in range(3):
        for j in range(23):
            lo, T = oracle.level_split(float(x[i, j]), float(norm), scheme, s)
            k = lo + (1 if oracle.philox_word(seed, step, i, j) < T else 0)
            assert codes[i, j] == (-k if x[i, j] < 0 else k)


def test_window_matches_full(oracle):
    rng = np.random.default_rng(8)
    x = rng.standard_normal((4, 50)).astype(np.float32)
    full, _ = oracle.quantize(x, 3.0, LINEAR, 7, 5, 9)
    win, _ = oracle.quantize(x, 3.0, LINEAR, 7, 5, 9, j0=13, j1=41)
    np.testing.assert_array_equal(full[:, 13:41], win)


# ----------------------------------------------------------------------------------------------
# brute force over every outcome
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("scheme,s,q,p", [(LINEAR, 3, 2, 2), (LINEAR, 1, INF, INF),
                                          (EXP, 3, 2, INF), (EXP, 2, INF, 2)])
@pytest.mark.parametrize("n,d", [(1, 5), (2, 5), (3, 3)])
def test_brute_force_unbiased_and_variance(oracle, scheme, s, q, p, n, d):
    rng = np.random.default_rng(n * 10 + d + 100 * s)
    x = (rng.standard_normal((n, d)) * 2.0).astype(np.float32)
    norm = np.float32(oracle.global_norm(x, q, p))
    outcomes = []  # per element: list of (probability, code)
    var_closed = [Fraction(0)] * d
    for i in range(n):
        for j in range(d):
            lo, T = oracle.level_split(float(x[i, j]), float(norm), scheme, s)
            sg = -1 if x[i, j] < 0 else 1
            if T == 0:
                outcomes.append([(Fraction(1), sg * lo)])
            else:
                pu = Fraction(T, TWO32)
                outcomes.append([(1 - pu, sg * lo), (pu, sg * (lo + 1))])
                v = Fraction(float(v32(x[i, j], norm)))
                hi_v, lo_v = level_value(scheme, s, lo + 1), level_value(scheme, s, lo)
                var_closed[j] += Fraction(float(norm)) ** 2 * (hi_v - v) * (v - lo_v) / n**2
    mean_out = np.zeros(d)
    second = np.zeros(d)
    for combo in itertools.product(*outcomes):
        prob = 1.0
        codes = np.zeros((n, d), dtype=np.int8)
        for e, (pr, c) in enumerate(combo):
            prob *= float(pr)
            codes[e // d, e % d] = c
        sums = oracle.reduce_codes(codes, scheme, s)
        out, rc = oracle.dequantize(sums, float(norm), scheme, s, n)
        assert rc == 0
        mean_out += prob * out
        second += prob * out**2
    xbar = x.astype(np.float64).mean(axis=0)
    tol = float(norm) * (2.0**-32 + 2.0**-23 + 1e-14)
    np.testing.assert_allclose(mean_out, xbar, rtol=0, atol=tol)
    var_enum = second - mean_out**2
    np.testing.assert_allclose(var_enum, [float(v) for v in var_closed], rtol=1e-6,
                               atol=float(norm) ** 2 * 1e-12)


# ----------------------------------------------------------------------------------------------
# Monte-Carlo over steps through the Philox-driven path
# ----------------------------------------------------------------------------------------------

def _closed_form(oracle, x, norm, scheme, s):
    """Per-column variance of out, expected nnz, per-element variance sum."""
    n, d = x.shape
    var = np.zeros(d)
    enz = 0.0
    for i in range(n):
        for j in range(d):
            lo, T = oracle.level_split(float(x[i, j]), float(norm), scheme, s)
            pu = T / TWO32
            if lo == s:
                enz += 1.0
                continue
            v = float(v32(x[i, j], norm))
            hi_v = float(level_value(scheme, s, lo + 1))
            lo_v = float(level_value(scheme, s, lo))
            var[j] += float(norm) ** 2 * (hi_v - v) * (v - lo_v) / n**2
            enz += 1.0 if lo >= 1 else pu
    return var, enz


@pytest.mark.parametrize("scheme,s,q,p", [(LINEAR, 5, 2, 2), (EXP, 4, 2, 2), (LINEAR, 2, INF, INF),
                                          (EXP, 6, 2, INF)])
def test_monte_carlo_unbiased(oracle, scheme, s, q, p):
    n, d, M = 3, 37, 12000
    rng = np.random.default_rng(99 + s)
    x = rng.standard_normal((n, d)).astype(np.float32)
    x[1, 5] = 0.0
    outs = np.empty((M, d))
    nnz = np.empty(M)
    seed = 0xC0FFEE
    for step in range(M):
        r = oracle.allreduce_mean(x, q, p, scheme, s, seed, step)
        assert r["rc"] == 0
        outs[step] = r["out"]
        nnz[step] = np.count_nonzero(r["codes"])
    norm = r["norm32"]
    var, enz = _closed_form(oracle, x, norm, scheme, s)
    xbar = x.astype(np.float64).mean(axis=0)
    mean = outs.mean(axis=0)
    for j in range(d):
        if var[j] == 0:
            assert abs(mean[j] - xbar[j]) <= 1e-6 * float(norm)
        else:
            z = (mean[j] - xbar[j]) / math.sqrt(var[j] / M)
            assert abs(z) < 5.5, (j, z)
    # the variance of the sum matches the closed form that assumes independent workers
    emp = outs.var(axis=0).sum()
    assert emp == pytest.approx(var.sum(), rel=0.06)
    # sparsity: expected number of non-zero codes
    assert abs(nnz.mean() - enz) < 5.5 * math.sqrt(max(nnz.var(), 1e-12) / M) + 1e-9


# ----------------------------------------------------------------------------------------------
# variance and sparsity bounds (re-derived; the page's theorem statement is lost)
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(4))
def test_variance_and_sparsity_bounds(oracle, seed):
    rng = np.random.default_rng(seed)
    n, d = 4, 64
    x = (rng.laplace(size=(n, d)) * rng.uniform(0.01, 1, size=(1, d))).astype(np.float32)
    l1 = float(np.abs(x.astype(np.float64)).sum())
    l2sq = float((x.astype(np.float64) ** 2).sum())
    for q, p in [(2, 2), (INF, INF), (2, INF)]:
        norm = np.float32(oracle.global_norm(x, q, p))
        N = float(norm)
        for s in (1, 2, 5, 31):
            var, enz = _closed_form(oracle, x, norm, LINEAR, s)
            elem_var = var.sum() * n**2  # E||Q(x) - x||^2 over all n*d elements
            assert elem_var <= min(n * d * N**2 / (4 * s * s), N * l1 / s) * (1 + 1e-6)
            if (q, p) == (2, 2):
                assert elem_var <= min(n * d / (4 * s * s), math.sqrt(n * d) / s) * l2sq * (1 + 1e-5)
                assert enz <= s * math.sqrt(n * d) + 1e-9
        for s in (1, 2, 4, 8):
            var, enz = _closed_form(oracle, x, norm, EXP, s)
            elem_var = var.sum() * n**2
            assert elem_var <= (l2sq / 8 + 2.0 ** -(s - 1) * N * l1) * (1 + 1e-5)
            if (q, p) == (2, 2):
                assert elem_var <= (1 / 8 + math.sqrt(n * d) / 2 ** (s - 1)) * l2sq * (1 + 1e-5)
                assert enz <= 2 ** (s - 1) * math.sqrt(n * d) + 1e-9


def test_linear_variance_bound_is_attained(oracle):
    # every v halfway between levels: each element contributes exactly N^2 / (4 s^2)
    s = 4
    x = np.array([[1.0, 0.125, 0.375, -0.625]], dtype=np.float32)  # N = 1 (max norm)
    var, _ = _closed_form(oracle, x, np.float32(1.0), LINEAR, s)
    assert var[1:].tolist() == [1 / (4 * s * s)] * 3


# ----------------------------------------------------------------------------------------------
# n = 1 reduction, code sums, dequantisation, edge cases
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("scheme,s", [(LINEAR, 7), (EXP, 5)])
@pytest.mark.parametrize("p", [2, INF])
def test_single_worker_reduces_to_qsgd(oracle, scheme, s, p):
    rng = np.random.default_rng(31)
    x = rng.standard_normal((1, 41)).astype(np.float32)
    a = oracle.allreduce_mean(x, 2, p, scheme, s, 3, 4)
    b = oracle.allreduce_mean(x, INF, p, scheme, s, 3, 4)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    local = np.float32(np.linalg.norm(x[0].astype(np.float64), 2 if p == 2 else np.inf))
    qsgd, rc = oracle.quantize(x, local, scheme, s, 3, 4)
    np.testing.assert_array_equal(a["codes"], qsgd)


def test_reduce_hand_decoded(oracle):
    codes = np.array([[3, -1, 0], [0, 2, -3]], dtype=np.int8)
    np.testing.assert_array_equal(oracle.reduce_codes(codes, LINEAR, 3), [3, 1, -3])
    # E_3: level k counts 2^(k-1) units: 3 -> 4, -1 -> -1, 2 -> 2, -3 -> -4
    np.testing.assert_array_equal(oracle.reduce_codes(codes, EXP, 3), [4, 1, -4])
    big = np.array([[8], [-8], [8]], dtype=np.int8)
    np.testing.assert_array_equal(oracle.reduce_codes(big, EXP, 8), [128])


def test_dequantize_hand(oracle):
    out, rc = oracle.dequantize(np.array([4, 1, -4]), 2.0, EXP, 3, 2)
    np.testing.assert_array_equal(out, [1.0, 0.25, -1.0])   # 2 * S * 2^-2 / 2
    out, rc = oracle.dequantize(np.array([3, 1]), 2.0, LINEAR, 3, 2)
    np.testing.assert_array_equal(out, [1.0, 1.0 / 3.0])    # 2 * S / (2 * 3)


def test_zero_input(oracle):
    x = np.zeros((3, 9), dtype=np.float32)
    x[1, 4] = -0.0
    for scheme, s in [(LINEAR, 7), (EXP, 4)]:
        r = oracle.allreduce_mean(x, 2, 2, scheme, s, 1, 2)
        assert r["rc"] == 0 and r["norm32"] == 0.0
        assert not r["codes"].any() and not r["out"].any()


def test_nonfinite_input(oracle):
    x = np.ones((2, 5), dtype=np.float32)
    x[0, 3] = np.nan
    r = oracle.allreduce_mean(x, INF, INF, LINEAR, 7, 1, 2)
    assert r["rc"] == 4
    assert not r["codes"].any() and not r["out"].any()


def test_codes_in_range(oracle):
    rng = np.random.default_rng(2)
    x = rng.standard_cauchy((5, 300)).astype(np.float32)
    for scheme, s in [(LINEAR, 1), (LINEAR, 127), (EXP, 1), (EXP, 24)]:
        r = oracle.allreduce_mean(x, INF, 2, scheme, s, 11, 12)
        assert np.abs(r["codes"].astype(int)).max() <= s
        assert ((r["codes"] == 0) | (np.sign(r["codes"]) == np.sign(x))).all()


def test_tie_does_not_round_up(oracle):
    # Round up iff r < T.  Global-E thresholds are the 23-bit fraction of v shifted left by 9,
    # so a word r with nine low zero bits is a reachable threshold: build v with T == r exactly
    # (must stay at the lower level) and v with T == r + 512 (must round up).
    seed, step = 5, 0
    j = next(j for j in range(1, 50000)
             if oracle.philox_word(seed, step, 0, j) & 0x1FF == 0
             and oracle.philox_word(seed, step, 0, j) != 0)
    r = oracle.philox_word(seed, step, 0, j)
    for frac, want in [(r >> 9, 6), ((r >> 9) + 1, 7)]:
        x = np.zeros((1, j + 1), dtype=np.float32)
        x[0, 0] = 1.0  # max norm N = 1
        v = (1.0 + frac / 2.0**23) * 0.25  # in [1/4, 1/2): level index 8 - 2 = 6 under E_8
        x[0, j] = v
        assert oracle.level_split(v, 1.0, EXP, 8) == (6, frac << 9)
        codes, rc = oracle.quantize(x, np.float32(1.0), EXP, 8, seed, step)
        assert codes[0, j] == want


def test_nan_element_under_supplied_norm(oracle):
    x = np.array([[np.nan, 1.0, np.inf, -2.0]], dtype=np.float32)
    codes, rc = oracle.quantize(x, np.float32(2.0), LINEAR, 5, 1, 1)
    assert rc == 0
    assert codes[0, 0] == 0 and codes[0, 2] == 5 and codes[0, 3] == -5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scheme,s", [(0, 7), (0, 127), (1, 4), (1, 24)])
def test_column_window_given_alone(oracle, dtype, scheme, s):
    """quantize_cols on a window's columns alone equals quantize on that window of the whole
    matrix: the random words stay keyed by the global column index."""
    from allreduce_compatible_gradient_gb300 import workloads
    n, d = 5, 4099
    x = workloads.host_inputs("normal", n, d, seed=17, dtype=dtype)
    norm32 = float(np.float32(oracle.global_norm(x, 2, 2)))
    for j0, j1 in [(0, 8), (3, 1003), (1001, 4099), (4096, 4099)]:
        want, rc = oracle.quantize(x, norm32, scheme, s, 9, 2, j0, j1)
        assert rc == 0
        got, rc = oracle.quantize_cols(np.ascontiguousarray(x[:, j0:j1]), j0, norm32, scheme, s,
                                       9, 2)
        assert rc == 0
        np.testing.assert_array_equal(got, want)
    # keyed by the global index: the same columns under another offset decide differently
    other, _ = oracle.quantize_cols(np.ascontiguousarray(x[:, 1001:4099]), 0, norm32, scheme, s,
                                    9, 2)
    assert not np.array_equal(other, oracle.quantize(x, norm32, scheme, s, 9, 2, 1001, 4099)[0])
