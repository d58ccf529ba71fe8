"""Pins for the oracle's Philox4x32-10 (CPU only).

The block function is pinned to the published known-answer vectors (tests/golden/); the word
mapping (high 16 bits from half j mod 8 of Philox(j/8, i, step lo, step hi), low 16 bits from half
j mod 8 of Philox(2^31 + j/8, i, step lo, step hi), key = (seed lo, seed hi)) is pinned by its
definition on top of the pinned block function and by independence checks that fail if a counter
field is dropped.
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


def _half(words, h):
    w = int(words[h >> 1])
    return (w >> 16) if (h & 1) else (w & 0xFFFF)


def test_word_mapping(oracle):
    rng = np.random.default_rng(7)
    for _ in range(200):
        seed = int(rng.integers(0, 2**64, dtype=np.uint64))
        step = int(rng.integers(0, 2**64, dtype=np.uint64))
        i = int(rng.integers(0, 1000))
        j = int(rng.integers(0, 2**34))
        key = [seed & 0xFFFFFFFF, seed >> 32]
        a = oracle.philox4x32_10([j >> 3, i, step & 0xFFFFFFFF, step >> 32], key)
        b = oracle.philox4x32_10([(j >> 3) | 0x80000000, i, step & 0xFFFFFFFF, step >> 32], key)
        want = (_half(a, j & 7) << 16) | _half(b, j & 7)
        assert oracle.philox_word(seed, step, i, j) == want


def test_first_call_is_the_zero_vector(oracle):
    # seed 0, step 0, worker 0, coordinates 0..7: the high halves come from counter 0, key 0,
    # i.e. the halves of the first known-answer vector, low half of each word first
    kat = _kat_rows()[0][2]
    want = [kat[h >> 1] >> 16 if h & 1 else kat[h >> 1] & 0xFFFF for h in range(8)]
    assert [oracle.philox_word(0, 0, 0, j) >> 16 for j in range(8)] == want
    assert want == [0xE8D5, 0x6627, 0xC58D, 0xE169, 0xAC4C, 0xBC57, 0xDBD8, 0x9B00]


def test_words_uniform_and_independent(oracle):
    # 4 workers x 4096 coordinates x 2 steps: top-nibble histogram is flat, the low halves are
    # flat too, and the words of
    # neighbouring workers, coordinates (same call / next call) and steps are uncorrelated.
    n, d = 4, 4096
    w = np.array([[[oracle.philox_word(3, st, i, j) for j in range(d)] for i in range(n)]
                  for st in range(2)], dtype=np.float64) / 2**32
    for vals in (w.ravel(), (w.ravel() * 65536) % 1.0):  # high bits, then the low half
        counts = np.bincount((vals * 16).astype(int), minlength=16)
        expected = w.size / 16
        chi2 = float(((counts - expected) ** 2 / expected).sum())
        assert chi2 < 60.0  # 15 dof; p ~ 1e-7
    hi = (w * 65536).astype(np.int64)
    lo = ((w * 2**32).astype(np.int64)) & 0xFFFF
    assert abs(np.corrcoef(hi.ravel(), lo.ravel())[0, 1]) < 5 / np.sqrt(hi.size)
    u = w - 0.5
    sd = 1 / np.sqrt(12)
    def corr(a, b):
        return float((a * b).mean() / sd**2)
    lim = 5 / np.sqrt(u[0, 0].size)
    assert abs(corr(u[0, 0], u[0, 1])) < lim          # workers
    assert abs(corr(u[0, 0, :-1], u[0, 0, 1:])) < lim  # adjacent coordinates
    assert abs(corr(u[0, 0, :-8], u[0, 0, 8:])) < lim  # next Philox call
    assert abs(corr(u[0, 0], u[1, 0])) < lim          # steps
