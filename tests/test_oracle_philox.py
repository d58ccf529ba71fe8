"""Pins for the oracle's Philox4x32-10 (CPU only).

The block function is pinned to the published known-answer vectors (tests/golden/); the word
mapping (counter = (j/4, i, step lo, step hi), key = (seed lo, seed hi), word j mod 4) is pinned
by its definition on top of the pinned block function and by independence checks that fail if a
counter field is dropped.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            w = [int(t, 16) for t in line.split()]
            assert len(w) == 10
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


@pytest.mark.parametrize("row", _kat_rows())
def test_known_answer_vectors(oracle, row):
    ctr, key, want = row
    got = oracle.philox4x32_10(ctr, key)
    assert [int(v) for v in got] == want


def test_word_mapping(oracle):
    rng = np.random.default_rng(7)
    for _ in range(200):
        seed = int(rng.integers(0, 2**64, dtype=np.uint64))
        step = int(rng.integers(0, 2**64, dtype=np.uint64))
        i = int(rng.integers(0, 1000))
        j = int(rng.integers(0, 2**34))
        ctr = [(j >> 2) & 0xFFFFFFFF, i, step & 0xFFFFFFFF, step >> 32]
        key = [seed & 0xFFFFFFFF, seed >> 32]
        assert oracle.philox_word(seed, step, i, j) == int(oracle.philox4x32_10(ctr, key)[j & 3])


def test_first_call_is_the_zero_vector(oracle):
    # seed 0, step 0, worker 0, coordinates 0..3 -> counter 0, key 0 -> first KAT vector
    want = _kat_rows()[0][2]
    assert [oracle.philox_word(0, 0, 0, j) for j in range(4)] == want


def test_words_uniform_and_independent(oracle):
    # 4 workers x 4096 coordinates x 2 steps: top-nibble histogram is flat and the words of
    # neighbouring workers, coordinates (same call / next call) and steps are uncorrelated.
    n, d = 4, 4096
    w = np.array([[[oracle.philox_word(3, st, i, j) for j in range(d)] for i in range(n)]
                  for st in range(2)], dtype=np.float64) / 2**32
    counts = np.bincount((w.ravel() * 16).astype(int), minlength=16)
    expected = w.size / 16
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 60.0  # 15 dof; p ~ 1e-7
    u = w - 0.5
    sd = 1 / np.sqrt(12)
    def corr(a, b):
        return float((a * b).mean() / sd**2)
    lim = 5 / np.sqrt(u[0, 0].size)
    assert abs(corr(u[0, 0], u[0, 1])) < lim          # workers
    assert abs(corr(u[0, 0, :-1], u[0, 0, 1:])) < lim  # adjacent coordinates
    assert abs(corr(u[0, 0, :-4], u[0, 0, 4:])) < lim  # next Philox call
    assert abs(corr(u[0, 0], u[1, 0])) < lim          # steps
