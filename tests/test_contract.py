"""The code-flip clause of the accuracy contract, checked on made-up data so that
the GPU tests' helper is known to accept exactly what the contract allows."""
import numpy as np
import pytest

from contract import assert_code_flips_at_ties


def _case():
    rng = np.random.default_rng(3)
    M, K = 4, 4096
    xn = rng.standard_normal((M, K)).astype(np.float32)
    s = np.full(M, 40.0, np.float32)
    xn[1, 7] = np.float32(2.5 / 40.0)  # xn * s = 2.5 (a tie up to float rounding)
    xn[2, 9] = np.float32(2.2 / 40.0)  # xn * s = 2.2 (no tie)
    q = np.rint(xn.astype(np.float64) * 40.0).astype(np.int8)
    return q, xn, s


def test_identical_codes_pass():
    q, xn, s = _case()
    assert_code_flips_at_ties(q.copy(), q, xn, s)


def test_flip_at_a_tie_passes():
    q, xn, s = _case()
    c = q.copy()
    c[1, 7] += 1
    assert_code_flips_at_ties(c, q, xn, s)


def test_flip_away_from_a_tie_fails():
    q, xn, s = _case()
    c = q.copy()
    c[2, 9] += 1
    with pytest.raises(AssertionError, match="away from a tie"):
        assert_code_flips_at_ties(c, q, xn, s)


def test_flip_by_two_fails():
    q, xn, s = _case()
    c = q.copy()
    c[1, 7] += 2
    with pytest.raises(AssertionError, match="more than one"):
        assert_code_flips_at_ties(c, q, xn, s)


def test_too_many_flips_fail():
    q, xn, s = _case()
    c = q.copy()
    c[1, 7] += 1
    c[1, 8] += 1  # two flips in 16384 codes: above 1e-4
    with pytest.raises(AssertionError, match="codes differ"):
        assert_code_flips_at_ties(c, q, xn, s)
