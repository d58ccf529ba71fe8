"""The boundary inputs of the GPU parity tests (tests/boundary_inputs.py) really put decisions on
their boundary: checked on the CPU with the oracle alone (its level split and Philox words).

For Global-E the threshold T is a multiple of 512 and for Global-L below the first level a
multiple of 4s, so exact ties T == r and their neighbours T == r +- 1 exist only for words with
the matching low bits; the construction finds them and must hit them exactly.  The other
elements must land near multiples of 2^16 from r, where the kernels' 16-bit estimate is least
certain.
"""
import numpy as np
import pytest

import boundary_inputs as bi

W16 = 1 << 16


def test_philox_words_equal_single_words(oracle):
    w = oracle.philox_words(7, 2**40 + 3, 5, 1000, 37)
    assert [int(v) for v in w] == [oracle.philox_word(7, 2**40 + 3, 5, 1000 + j) for j in range(37)]


@pytest.mark.parametrize("scheme,s", [(0, 127), (0, 7), (1, 8), (1, 4)])
def test_max_norm_f32_hits_ties_and_window(oracle, scheme, s):
    rng = np.random.default_rng(11)
    x, info = bi.max_norm_matrix(4, 1 << 15, scheme, s, 3, 5, 1024, rng)
    N = np.float32(oracle.global_norm(x, 0, 0))
    assert N == np.float32(1.5)
    got = bi.achieved_offsets(x, info, N, scheme, s, 3, 5)
    np.testing.assert_array_equal(got, info["achieved"])
    assert (got == 0).sum() >= 20 and (got == 1).sum() >= 10 and (got == -1).sum() >= 10
    # the aimed offset is reached exactly where the word admits it (tie_offsets) and the
    # division by N = 1.5 reaches the needed v (most of the time), else within 512
    R = bi.words(4, 1 << 15, 3, 5)
    tie = bi.tie_offsets(R, scheme, s).ravel()[info["positions"]] != 2
    assert tie.sum() >= 40
    hit = got[tie] == info["aimed"][tie]
    assert hit.mean() >= 0.7 and (np.abs(got[tie] - info["aimed"][tie]) <= 513).all()
    near = np.abs(got) < 5 * W16
    assert near.mean() > 0.9
    # every window edge is populated
    for k in (1, 2, 3, 4):
        assert (np.abs(np.abs(got) - k * W16) < W16 // 4).sum() >= 10


@pytest.mark.parametrize("scheme,s", [(0, 127), (1, 8)])
def test_max_norm_bf16_lands_in_window(oracle, scheme, s):
    rng = np.random.default_rng(12)
    x, info = bi.max_norm_matrix(4, 1 << 15, scheme, s, 3, 5, 512, rng, dtype="bf16")
    assert x.dtype == np.uint16
    N = np.float32(oracle.global_norm(x, 0, 0))
    got = bi.achieved_offsets(x, info, N, scheme, s, 3, 5)
    np.testing.assert_array_equal(got, info["achieved"])
    assert len(got) >= 256 and (np.abs(got) <= 5 * W16).all()


def test_l2_norm_converges_and_hits(oracle):
    rng = np.random.default_rng(13)
    x, info = bi.l2_norm_matrix(4, 1 << 15, 1, 8, 3, 5, 1024, rng)
    assert info["converged"]
    N = np.float32(oracle.global_norm(x, 2, 2))
    assert float(N) == info["N"]
    got = bi.achieved_offsets(x, info, N, 1, 8, 3, 5)
    assert (got == 0).sum() >= 20 and (np.abs(got) < 5 * W16).mean() > 0.9


def test_supplied_norm_has_saturated_elements(oracle):
    rng = np.random.default_rng(14)
    N = 0.7431
    x, info = bi.supplied_norm_matrix(2, 4096, 0, 15, 3, 5, 256, rng, N)
    a = np.abs(x.ravel()[info["saturated"]])
    assert (a == np.float32(N)).any() and (a > np.float32(N)).any()
    codes, rc = oracle.quantize(x, np.float32(N), 0, 15, 3, 5)
    assert rc == 0
    assert (np.abs(codes.ravel()[info["saturated"]]) == 15).all()  # v clamps to 1: the top level
