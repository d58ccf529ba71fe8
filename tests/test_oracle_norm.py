"""Pins for the oracle's global norm ||x||_{q,p} (CPU only).

Closed forms on constructed inputs, numpy.linalg.norm applied per axis (the q-norm over the
workers of each coordinate, then the p-norm over coordinates), an exactly rounded sum, the n = 1
reduction and permutation invariances.  A transposed reading (q over coordinates, p over workers)
fails the numpy and closed-form checks on non-square inputs.
"""
import math

import numpy as np
import pytest

INF = 0
ORDERS = [(2, 2), (2, INF), (INF, 2), (INF, INF)]


def _np_order(o):
    return np.inf if o == INF else 2


def numpy_norm(x, q, p):
    x64 = x.astype(np.float64)
    per_coord = np.linalg.norm(x64, ord=_np_order(q), axis=0)  # over workers
    return float(np.linalg.norm(per_coord, ord=_np_order(p)))


def to_bf16_bits(a):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (uint16)."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("n,d", [(1, 1), (3, 5), (4, 7), (7, 3)])
def test_all_ones_closed_forms(oracle, n, d):
    x = np.ones((n, d), dtype=np.float32)
    # (2, 2) takes sqrt per coordinate and squares it back: a few fp64 roundings
    assert oracle.global_norm(x, 2, 2) == pytest.approx(math.sqrt(n * d), rel=1e-15)
    assert oracle.global_norm(x, 2, INF) == math.sqrt(n)
    assert oracle.global_norm(x, INF, 2) == math.sqrt(d)
    assert oracle.global_norm(x, INF, INF) == 1.0


def test_one_hot(oracle):
    x = np.zeros((5, 9), dtype=np.float32)
    x[3, 6] = -2.5
    for q, p in ORDERS:
        assert oracle.global_norm(x, q, p) == 2.5


@pytest.mark.parametrize("q,p", ORDERS)
@pytest.mark.parametrize("n,d", [(2, 3), (3, 17), (8, 5), (5, 64)])
def test_matches_numpy_per_axis(oracle, q, p, n, d):
    rng = np.random.default_rng(n * 100 + d)
    x = rng.standard_normal((n, d)).astype(np.float32) * rng.uniform(0.1, 10, size=(n, 1)).astype(np.float32)
    got = oracle.global_norm(x, q, p)
    want = numpy_norm(x, q, p)
    assert got == pytest.approx(want, rel=1e-13, abs=0)


def test_orders_are_not_interchangeable(oracle):
    # a worker-heavy input: the (2, inf) and (inf, 2) norms differ, so a swapped reading fails
    x = np.array([[3.0, 0.0, 0.0], [4.0, 0.0, 1.0]], dtype=np.float32)
    assert oracle.global_norm(x, 2, INF) == 5.0          # column 0: sqrt(9 + 16)
    assert oracle.global_norm(x, INF, 2) == math.sqrt(17.0)  # max per column: 4, 0, 1
    assert oracle.global_norm(x, 2, 2) == pytest.approx(math.sqrt(26.0), rel=1e-15)
    assert oracle.global_norm(x, INF, INF) == 4.0


def test_l2_l2_exactly_rounded_sum(oracle):
    # ||x||_{2,2} = ||vec x||_2; squares of fp32 values are exact in fp64 and fsum rounds the
    # exact sum once, so sqrt(fsum) is within a few fp64 ulps of the oracle.
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((6, 5000)) * np.exp(rng.uniform(-8, 8, size=(6, 5000)))).astype(np.float32)
    exact = math.sqrt(math.fsum(float(v) * float(v) for v in x.ravel()))
    assert oracle.global_norm(x, 2, 2) == pytest.approx(exact, rel=4e-16 * 5000 ** 0.5 + 1e-15)


@pytest.mark.parametrize("p", [2, INF])
def test_single_worker_norm_is_independent_of_q(oracle, p):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, 33)).astype(np.float32)
    a, b = oracle.global_norm(x, 2, p), oracle.global_norm(x, INF, p)
    assert a == b
    assert a == pytest.approx(float(np.linalg.norm(x[0].astype(np.float64), _np_order(p))), rel=1e-15)


@pytest.mark.parametrize("q,p", ORDERS)
def test_permutation_invariance(oracle, q, p):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((5, 21)).astype(np.float32)
    base = oracle.global_norm(x, q, p)
    xr = np.ascontiguousarray(x[rng.permutation(5)])
    xc = np.ascontiguousarray(x[:, rng.permutation(21)])
    assert oracle.global_norm(xr, q, p) == pytest.approx(base, rel=1e-15)
    assert oracle.global_norm(xc, q, p) == pytest.approx(base, rel=1e-15)


def test_bf16_widening(oracle):
    bits = np.array([[0x3F80, 0xC000, 0x3F00, 0x0000, 0x8000, 0x4049]], dtype=np.uint16)
    # 1.0, -2.0, 0.5, +0, -0, 3.140625
    assert oracle.global_norm(bits, INF, INF) == 3.140625
    assert oracle.global_norm(bits, 2, 2) == pytest.approx(math.sqrt(1 + 4 + 0.25 + 3.140625**2), rel=1e-15)
    rng = np.random.default_rng(9)
    x = rng.standard_t(3, size=(4, 50)).astype(np.float32)
    b = to_bf16_bits(x)
    for q, p in ORDERS:
        assert oracle.global_norm(b, q, p) == oracle.global_norm(bf16_bits_to_f32(b), q, p)


def test_nonfinite_inputs(oracle):
    x = np.ones((3, 4), dtype=np.float32)
    x[1, 2] = np.inf
    for q, p in ORDERS:
        assert math.isinf(oracle.global_norm(x, q, p))
    x[0, 0] = np.nan
    for q, p in ORDERS:
        assert math.isnan(oracle.global_norm(x, q, p))


def test_invalid_arguments(oracle):
    x = np.ones((2, 2), dtype=np.float32)
    assert oracle.global_norm(x, 1, 2) == -1.0
    assert oracle.global_norm(x, 2, 3) == -1.0


def test_norm_bounds_every_element(oracle):
    # |x_ij| <= ||x||_{q,p} for q, p >= 1, and the fp32 rounding keeps it (monotone rounding)
    rng = np.random.default_rng(21)
    x = rng.standard_cauchy((7, 40)).astype(np.float32)
    for q, p in ORDERS:
        assert np.float32(oracle.global_norm(x, q, p)) >= np.abs(x).max()
