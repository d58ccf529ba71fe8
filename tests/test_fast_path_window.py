"""CPU model of the kernels' fast rounding decision, checked against the oracle on the boundary
inputs, with its certainty window and with narrower (wrong) windows.

The quantise kernels decide an element without dividing: P (the position of v = fp32(|x| / N) on
the level grid) is estimated in 16.16 fixed point as the bits of fp32(|x| c1 + c0) with one fused
multiply-add (c1 = RN(s / N) for Global-L, RN(1 / N) 2^(s-1) for Global-E; c0 = 128 + 0xFFFD
2^-16 puts the estimate in the binade [128, 256), whose unit is 2^-16), or, for Global-E levels
of 1 and more, as the biased exponent and 16 fraction bits of fp32(|x| RN(1 / N)).  With H the
high 16 bits of the element's random word, y = bits - H holds the level index (plus 0x4300) in
its high half, and the decision counts as certain when the low half is at most 0xFFFB: the
estimate is within 2 units of 2^-16 of P and the unknown low half of the word adds less than
one.  Otherwise the kernel recomputes the element exactly (correctly rounded quotient, full
word), as the oracle defines it.

This model restates that arithmetic on the CPU (exact fused multiply-add through rationals) and
asserts, on the inputs the GPU boundary tests use, that every decision it calls certain equals
the oracle's.  It also shows the inputs are sharp enough: with the window one unit narrower on
either side, some certain decisions are wrong, so the GPU tests would fail on such a kernel.
"""
import numpy as np
import pytest

import boundary_inputs as bi
from fast_path_model import fast_decision

# the norm 0.48058903 has RN(127 / N) off by nearly half a unit: with it, the Global-L_127 case
# also gets elements whose fast estimate is more than one unit low (worst_error_elements)
WORST_N = 0.48058903


def _cases():
    out = []
    for scheme, s in [(0, 127), (0, 15), (0, 7), (1, 8), (1, 4)]:
        for N in (1.5, 0.8191):
            out.append((scheme, s, N))
    out.append((0, 127, WORST_N))
    return out


def _boundary(oracle, scheme, s, N, seed=3, step=5):
    rng = np.random.default_rng(100 + s + int(N * 1000))
    worst = 256 if N == WORST_N else 0
    x, info = bi.max_norm_matrix(4, 1 << 14, scheme, s, seed, step, 1536, rng, N=N,
                                 worst=worst)
    N32 = np.float32(oracle.global_norm(x, 0, 0))
    codes, rc = oracle.quantize(x, N32, scheme, s, seed, step)
    assert rc == 0
    d = x.shape[1]
    rows = []
    for p in np.concatenate([info["positions"], info.get("worst", np.zeros(0, np.int64))]):
        i, j = divmod(int(p), d)
        r = oracle.philox_word(seed, step, i, j)
        rows.append((abs(float(x[i, j])), r, abs(int(codes[i, j]))))
    return float(N32), rows


@pytest.mark.parametrize("scheme,s,N", _cases())
def test_certain_decisions_equal_the_oracle(oracle, scheme, s, N):
    N32, rows = _boundary(oracle, scheme, s, N)
    uncertain = 0
    for ax, r, k in rows:
        certain, kf = fast_decision(ax, N32, scheme, s, r)
        if certain:
            assert kf == k, (ax, r, kf, k)
        else:
            uncertain += 1
    # the inputs sit on the boundary: many decisions need the exact path
    assert uncertain >= len(rows) // 20


@pytest.mark.parametrize("window", [0xFFFC, 0xFFFD])
def test_a_narrower_window_decides_some_boundary_inputs_wrong(oracle, window):
    """Planted on this CPU model only: a window narrower than the kernels' (low half above
    0xFFFB) calls some boundary decisions certain that are wrong."""
    wrong = 0
    for scheme, s, N in _cases():
        N32, rows = _boundary(oracle, scheme, s, N)
        for ax, r, k in rows:
            certain, kf = fast_decision(ax, N32, scheme, s, r, window)
            wrong += certain and kf != k
    assert wrong > 0


def test_top_of_the_window_matters(oracle):
    """The other edge: calling a low half of 0xFFFF certain (a window one value narrower at its
    top) is wrong for some boundary inputs too."""
    wrong = 0
    for scheme, s, N in _cases():
        N32, rows = _boundary(oracle, scheme, s, N)
        for ax, r, k in rows:
            certain, kf = fast_decision(ax, N32, scheme, s, r)
            low_ffff = not certain and fast_decision(ax, N32, scheme, s, r, 0xFFFF)[0]
            y_top = low_ffff and not fast_decision(ax, N32, scheme, s, r, 0xFFFE)[0]
            wrong += y_top and fast_decision(ax, N32, scheme, s, r, 0xFFFF)[1] != k
    assert wrong > 0


def test_worst_estimates_are_more_than_one_unit_low(oracle):
    from fast_path_model import estimate_error
    rng = np.random.default_rng(5)
    x, info = bi.max_norm_matrix(4, 1 << 14, 0, 127, 3, 5, 64, rng, N=WORST_N, worst=128)
    assert len(info["worst"]) >= 64
    a = np.abs(x.ravel()[info["worst"]])
    assert (estimate_error(a, np.float32(WORST_N), 127) < -1.0).all()
