"""CPU model of the quantise kernels' fast rounding decision (test infrastructure).

The kernels decide an element without dividing: P (the position of v = fp32(|x| / N) on the level
grid) is estimated in 16.16 fixed point as the bits of fp32(|x| c1 + c0) from one fused
multiply-add (c1 = RN(s / N) for Global-L, RN(1 / N) 2^(s-1) for Global-E; c0 = 128 + 0xFFFD
2^-16 puts the estimate in the binade [128, 256), whose unit is 2^-16), or, for Global-E levels
of 1 and more, as the biased exponent and 16 fraction bits of fp32(|x| RN(1 / N)).  With H the
high 16 bits of the element's random word, y = bits - H holds the level index plus 0x4300 in its
high half, and the decision counts as certain when the low half is at most 0xFFFB.  Otherwise
the kernel recomputes the element exactly, as the oracle defines it.

fast_decision restates that arithmetic exactly (the fused multiply-add through rationals);
estimate_error is a vectorised form used to search for inputs whose estimate is furthest from
the exact position.
"""
from fractions import Fraction

import numpy as np

LINEAR, EXP = 0, 1
C0_BITS = 0x4300FFFD
OFF = 0x4300


def f32(x) -> float:
    return float(np.float32(x))


def bits32(v: float) -> int:
    return int(np.array([v], dtype=np.float32).view(np.uint32)[0])


def round_f32(q: Fraction) -> float:
    """q rounded to the nearest fp32 (ties to even); normal range only."""
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    scaled = a / Fraction(2) ** (e - 23)  # in [2^23, 2^24)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return sign * float(Fraction(m) * Fraction(2) ** (e - 23))


def fma32(a: float, b: float, c: float) -> float:
    return round_f32(Fraction(a) * Fraction(b) + Fraction(c))


def fast_decision(ax: float, N: float, scheme: int, s: int, r: int, window: int = 0xFFFB):
    """(certain, k) of the kernels' fast path for |x| = ax under the fp32 norm N and word r."""
    rcp = f32(np.float32(1.0) / np.float32(N))
    c0 = float(np.array([C0_BITS], dtype=np.uint32).view(np.float32)[0])
    if scheme == LINEAR:
        c1 = f32(np.float32(s) / np.float32(N))
    else:
        c1 = rcp * 2.0 ** (s - 1)  # exact: a power-of-two scaling
    pb = bits32(fma32(ax, c1, c0))
    if scheme == EXP:
        vb = min(bits32(f32(np.float32(ax) * np.float32(rcp))), 0x3F800000)
        if vb >= (128 - s) << 23:  # v >= 2^-(s-1): exponent and fraction bits of v
            pb = (vb >> 7) + (((s - 127) << 16) + C0_BITS)
            pb &= 0xFFFFFFFF
    y = (pb - (r >> 16)) & 0xFFFFFFFF
    k = (y >> 16) - OFF
    certain = (y & 0xFFFF) <= window and not (scheme == LINEAR and k > s)
    return certain, k



def estimate_error(ax: np.ndarray, N: float, s: int) -> np.ndarray:
    """Global-L: estimate minus exact position, in units of 2^-16, for fp32 magnitudes ax with
    |x| c1 >= 2^-30 (there the float64 sum |x| c1 + c0 is exact, so its conversion to fp32 is the
    kernels' single rounding)."""
    ax = np.asarray(ax, dtype=np.float32)
    N32 = np.float32(N)
    c1 = np.float32(np.float32(s) / N32)
    c0 = np.array([C0_BITS], dtype=np.uint32).view(np.float32)[0]
    pb = (ax.astype(np.float64) * np.float64(c1) + np.float64(c0)).astype(np.float32)
    P_est = pb.view(np.uint32).astype(np.int64) - 0x43000000 - 0xFFFD
    v = (ax / N32).astype(np.float32)
    return P_est - v.astype(np.float64) * s * 65536.0
