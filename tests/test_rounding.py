"""CPU checks of the rounding-aware attention allowance used by the bf16
parity tests."""

import numpy as np

import rounding
from oracle import fusion as orc


def test_neighbours_bracket_the_value():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(5000) * 10.0 ** rng.uniform(-3, 3, 5000)
    r, o = rounding._neighbours(x)
    lo, hi = np.minimum(r, o), np.maximum(r, o)
    assert np.all(lo <= x) and np.all(x <= hi)
    assert np.array_equal(orc.round_bf16(lo), lo) and np.array_equal(orc.round_bf16(hi), hi)
    assert np.all(np.abs(x - r) <= np.abs(x - o))        # the stored one is the nearer


def test_ambiguous_marks_midpoints_only():
    mid = 1.0 + 2.0 ** -8                                  # halfway between 1 and 1 + 2^-7
    assert rounding.ambiguous(np.array([mid]), np.array([0.0]))[0]
    assert not rounding.ambiguous(np.array([1.0]), np.array([1e-6]))[0]
    assert rounding.ambiguous(np.array([mid + 1e-7]), np.array([2e-7]))[0]
    assert not rounding.ambiguous(np.array([mid + 1e-5]), np.array([2e-7]))[0]


def test_allowance_is_stated_tolerance_without_ambiguity():
    # values far from every midpoint: the allowance is the stated tolerance
    rng = np.random.default_rng(4)
    d, D = 8, 16
    H = orc.round_bf16(rng.standard_normal((6, D)))
    W = [orc.round_bf16(rng.standard_normal((n * d, D)) / 4) for n in (2, 1, 1)]
    S = np.arange(6)
    Kf, Vf, O, _ = orc.recompute_selected(H, *W, S, 6, np.zeros((6, 1, d)), np.zeros((6, 1, d)),
                                          2, 1, d, 1e4, store=orc.round_bf16)
    allow, base, _ = rounding.allowance(H, *W, S, Kf, Vf, O, S, 2, 1, d, 1e4, tol=2e-2)
    assert base == 2e-2 * np.max(np.abs(O))
    assert np.all(allow >= base) and np.all(allow <= 1.5 * base)
