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


def test_stitched_bounds_and_their_flips():
    # stitched values: a chunk at offset 0 stored in the layer's type is
    # copied bit for bit (no error); a rotated or dequantised one is not
    rng = np.random.default_rng(5)
    d = 8
    K = [orc.round_bf16(rng.standard_normal((3, 1, d))) for _ in range(2)]
    V = [orc.round_bf16(rng.standard_normal((3, 1, d))) for _ in range(2)]
    K64, eK, V64, eV = rounding.stitched_bounds(K, V, 1e4, quantized=False)
    assert np.array_equal(K64[:3], K[0][:]) and not np.any(eK[:3]) and not np.any(eV)
    assert np.all(eK[3:] > 0)
    assert np.allclose(K64[3:], orc.rope_rotate(K[1], 3, 1e4))
    _, eKq, _, eVq = rounding.stitched_bounds(K, V, 1e4, quantized=True)
    assert np.all(eKq[:3] > 0) and np.all(eVq > 0)


def test_allowance_grows_only_for_rows_that_see_a_stitched_flip():
    # one reused key element planted on a bf16 midpoint: rows whose causal
    # prefix holds it get a wider allowance, rows before it do not
    rng = np.random.default_rng(6)
    d, D, n, T = 8, 16, 6, 8
    H = orc.round_bf16(rng.standard_normal((T, D)))
    W = [orc.round_bf16(rng.standard_normal((m * d, D)) / 4) for m in (2, 1, 1)]
    K64 = rng.standard_normal((n, 1, d)) * 4
    V64 = orc.round_bf16(rng.standard_normal((n, 1, d)))
    K64[4, 0, 3] = 2.0 + 2.0 ** -7                   # halfway between 2 and 2 + 2^-6
    eK = np.zeros_like(K64)
    eV = np.zeros_like(V64)
    Kf0 = np.zeros((T, 1, d))
    Vf0 = np.zeros((T, 1, d))
    Kf0[:n], Vf0[:n] = orc.round_bf16(K64), V64
    idx = np.array([1])
    Kf, Vf, O, S = orc.recompute_selected(H, *W, idx, n, Kf0, Vf0, 2, 1, d, 1e4,
                                          store=orc.round_bf16)
    rows = np.arange(len(S))                          # positions 1, 6, 7
    plain, base, _ = rounding.allowance(H, *W, S, Kf, Vf, O, rows, 2, 1, d, 1e4)
    wide, _, _ = rounding.allowance(H, *W, S, Kf, Vf, O, rows, 2, 1, d, 1e4,
                                    stitched=(K64, eK, V64, eV))
    assert np.array_equal(wide[0], plain[0])          # position 1 does not reach row 4
    assert np.all(wide[1:] > plain[1:])               # positions 6 and 7 do
