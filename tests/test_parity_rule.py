"""The GPU-vs-oracle acceptance rule itself (oracle/compare.py), on the CPU.

A sampled index may differ from the float64 inverse CDF only where float
rounding can explain it: the threshold must lie within 1e-5 (relative) of every
CDF boundary between the two answers.  These tests feed the checker fabricated
"GPU" answers: legitimate rounding mismatches must be excused and counted, and
an answer several keys off must fail even when the threshold happens to sit next
to the oracle's own boundary.
"""

import math

import numpy as np
import pytest

from oracle import compare, prop_head


def _cdf(p):
    return np.cumsum(np.asarray(p, dtype=np.float64))


def test_one_boundary_within_rounding_is_excused():
    F = _cdf([0.1, 0.2, 0.3, 0.4])  # boundaries 0.1, 0.3, 0.6, 1.0
    t = 0.3 * (1 + 3e-6)            # just above F(1): the float64 answer is key 2
    assert compare.excused(F, t, 1, 2)
    assert compare.excused(F, t, 2, 1)
    assert compare.excused(F, t, 2, 2)


def test_several_keys_off_is_not_excused_even_next_to_a_boundary():
    # 10 keys of mass 0.1: boundaries 0.1, 0.2, ..., 1.0
    F = _cdf(np.full(10, 0.1))
    t = F[6] * (1 + 1e-7)  # next to the oracle's boundary F(6): the oracle picks key 7
    # a kernel that returned key 4 crossed F(4), F(5), F(6): only F(6) is near t
    assert not compare.excused(F, t, 4, 7)
    # and a kernel three keys above the oracle's answer crossed F(7), F(8), F(9)
    t2 = F[6] * (1 - 1e-7)  # just below F(6): the oracle picks key 6
    assert not compare.excused(F, t2, 9, 6)
    # one key off in either case is rounding
    assert compare.excused(F, t, 6, 7)
    assert compare.excused(F, t2, 7, 6)


def test_zero_mass_keys_between_the_answers_share_one_boundary():
    # keys 2..4 have no mass: F(1) = F(2) = F(3) = F(4) = 0.5
    F = _cdf([0.25, 0.25, 0.0, 0.0, 0.0, 0.5])
    t = 0.5 * (1 - 2e-6)
    assert compare.excused(F, t, 1, 5)  # every boundary crossed is the same value 0.5
    assert not compare.excused(F, 0.4, 1, 5)


def _problem(seed=3, n=300, d=64):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    return q, K, V


def test_check_prop_head_counts_rounding_and_rejects_a_planted_slip():
    q, K, V = _problem()
    S, tile = 64, 64
    # choose U so that one threshold sits a hair above the CDF boundary F(j)
    ref0 = prop_head(q, K, V, S, 0.0, tile, want_F=True)
    F = ref0.F
    j = int(np.searchsorted(F, 0.3))  # a boundary near 0.3
    t = F[j] * (1 + 2e-7)
    m = int(t * S)
    U = t - m / S
    assert 0.0 <= U < 1.0 / S and F[j + 1] > t and F[j] - F[j - 3] > 1e-3
    ref = prop_head(q, K, V, S, U, tile, want_F=True)
    assert ref.J[m] == j + 1

    # a rounding mismatch at sample m (one key down): excused, counted, and `out`
    # compared with the gather over the GPU's own indices
    idx = ref.J.copy()
    idx[m] = j
    out = compare.gather_mean(idx, V)
    rep = compare.check_prop_head(q, K, V, S, U, tile, out, idx)
    assert rep.excused == 1 and rep.samples == S

    # a slip of several keys at the same sample: rejected
    idx_bad = ref.J.copy()
    idx_bad[m] = j - 3
    with pytest.raises(AssertionError, match=f"sample {m} "):
        compare.check_prop_head(q, K, V, S, U, tile, compare.gather_mean(idx_bad, V), idx_bad)

    # a wrong output with the right indices: rejected by the 2e-3 bound
    with pytest.raises(AssertionError, match="out err"):
        compare.check_prop_head(q, K, V, S, U, tile, ref.out + 3e-3, ref.J)


def test_report_bound_helper():
    rep = compare.Report(heads=4, samples=1000, excused=10)
    assert compare.excused_within_bound(rep)
    rep.excused = 11
    assert not compare.excused_within_bound(rep)
    # small totals still allow a couple of boundary cases
    assert compare.excused_within_bound(compare.Report(heads=1, samples=16, excused=2))
    assert math.isclose(compare.EXCUSED_FRACTION, 0.01)
