"""The end-to-end accuracy contract on int8 codes, shared by the GPU parity
tests and checked itself on the CPU (tests/test_contract.py)."""
import numpy as np


def assert_code_flips_at_ties(codes, q_ora, xn_ora, s_ora, what=""):
    """End-to-end int8 codes against the oracle's: at most 1e-4 of them differ,
    each by one, and only where the oracle's xn * a_scale lies within 1e-3 of a
    half-integer (a rounding tie that the order of the sum of squares can tip)."""
    d = np.abs(codes.astype(np.int32) - q_ora.astype(np.int32))
    assert d.max(initial=0) <= 1, f"{what}: a code differs by more than one"
    assert np.mean(d != 0) <= 1e-4, f"{what}: {int(np.sum(d != 0))} codes differ"
    if np.any(d):
        v = np.abs(xn_ora[d != 0].astype(np.float64) * np.repeat(s_ora.astype(np.float64)[:, None],
                                                                 codes.shape[1], axis=1)[d != 0])
        assert np.all(np.abs(v - np.floor(v) - 0.5) <= 1e-3), f"{what}: a code differs away from a tie"
