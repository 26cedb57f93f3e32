"""Pins for the CPU oracle: each check comes from something other than the
oracle's own formula (closed forms, hand-worked values, a textbook library
routine, brute force, structural facts the pages state)."""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import fusion as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------- bf16 storage ----

def test_round_bf16_matches_torch_on_fp32_values():
    rng = _rng(40)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(orc.round_bf16(x.astype(np.float64)), want)


def test_round_bf16_nearest_by_brute_force():
    # the result is the nearest of the two bf16 neighbours, ties to the even one
    rng = _rng(41)
    for x in np.concatenate([rng.standard_normal(300) * 37.0, [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -3.0]]):
        e = math.floor(math.log2(abs(x)))
        ulp = 2.0 ** (e - 7)
        lo = math.floor(x / ulp) * ulp
        hi = lo + ulp
        dl, dh = x - lo, hi - x
        want = lo if dl < dh else hi if dh < dl else (lo if (lo / ulp) % 2 == 0 else hi)
        assert orc.round_bf16(np.array([x]))[0] == want, x
    assert orc.round_bf16(np.array([0.0]))[0] == 0.0


# ---------------------------------------------------------------- RoPE ----

def test_rope_inv_freq_closed_form():
    th = orc.rope_inv_freq(4, 10000.0)
    assert th.tolist() == [1.0, 0.01]
    th = orc.rope_inv_freq(128, 1e6)
    assert th[0] == 1.0
    for j in (1, 17, 63):
        assert abs(th[j] - 1e6 ** (-(2.0 * j) / 128.0)) <= 1e-15 * th[j]


def test_rope_hand_example_d4():
    # d = 4, base 1e4: theta = (1, 0.01); pairs are (x0, x2) and (x1, x3).
    x = np.array([1.0, 2.0, 3.0, 4.0])
    y = orc.rope_rotate(x, 1, 10000.0)
    c1, s1 = math.cos(1.0), math.sin(1.0)
    c2, s2 = math.cos(0.01), math.sin(0.01)
    want = [1 * c1 - 3 * s1, 2 * c2 - 4 * s2, 3 * c1 + 1 * s1, 4 * c2 + 2 * s2]
    assert np.allclose(y, want, rtol=0, atol=1e-15)


def test_rope_matches_complex_multiplication():
    # (x_j, x_{j+d/2}) as the complex number z_j; R^p multiplies by e^{i p theta_j}.
    rng = _rng(1)
    d, base = 64, 5e5
    x = rng.standard_normal((5, 3, d))
    pos = rng.integers(0, 40000, size=(5, 3))
    y = orc.rope_rotate(x, pos, base)
    h = d // 2
    for a in range(5):
        for b in range(3):
            for j in range(h):
                theta = base ** (-(2.0 * j) / d)
                z = complex(x[a, b, j], x[a, b, j + h]) * complex(math.cos(pos[a, b] * theta),
                                                                     math.sin(pos[a, b] * theta))
                assert abs(y[a, b, j] - z.real) < 1e-11
                assert abs(y[a, b, j + h] - z.imag) < 1e-11


def test_rope_matches_explicit_rotation_matrix():
    rng = _rng(2)
    d, base, p = 8, 1e4, 37
    x = rng.standard_normal(d)
    M = np.zeros((d, d))
    for j in range(d // 2):
        a = p * base ** (-(2.0 * j) / d)
        M[j, j], M[j, j + d // 2] = math.cos(a), -math.sin(a)
        M[j + d // 2, j], M[j + d // 2, j + d // 2] = math.sin(a), math.cos(a)
    assert np.allclose(orc.rope_rotate(x, p, base), M @ x, rtol=0, atol=1e-14)


def test_rope_zero_offset_is_identity():
    x = _rng(3).standard_normal((7, 2, 64))
    assert np.array_equal(orc.rope_rotate(x, 0, 1e6), x)


def test_rope_composition_and_inverse():
    rng = _rng(4)
    x = rng.standard_normal((9, 128))
    a, b = 1234, 31790
    ab = orc.rope_rotate(orc.rope_rotate(x, a, 1e6), b, 1e6)
    assert np.max(np.abs(ab - orc.rope_rotate(x, a + b, 1e6))) < 1e-11
    back = orc.rope_rotate(orc.rope_rotate(x, a, 1e6), -a, 1e6)
    assert np.max(np.abs(back - x)) < 1e-12
    assert np.allclose(np.linalg.norm(ab, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_dot_product_depends_on_offset_only():
    rng = _rng(5)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    s, t = 17, 411
    ref = orc.rope_rotate(q, s, 1e4) @ orc.rope_rotate(k, t, 1e4)
    for c in (1, 1000, 25000):
        v = orc.rope_rotate(q, s + c, 1e4) @ orc.rope_rotate(k, t + c, 1e4)
        assert abs(v - ref) < 1e-9


def test_rope_correction_50_to_1050():
    g = json.load(open(os.path.join(GOLDEN, "rope_correction_50_to_1050.json")))
    k = _rng(6).standard_normal((4, 128))
    cached = orc.rope_rotate(k, g["cached_pos"], 1e4)
    fixed = orc.rope_rotate(cached, g["correction"], 1e4)
    assert np.max(np.abs(fixed - orc.rope_rotate(k, g["reused_pos"], 1e4))) < 1e-11
    assert g["cached_pos"] + g["correction"] == g["reused_pos"]


# ------------------------------------------------------- PIC and stitch ----

def _tiny_model(seed, D=32, Hq=4, Hkv=2, d=8):
    rng = _rng(seed)
    Wq = rng.standard_normal((Hq * d, D)) / math.sqrt(D)
    Wk = rng.standard_normal((Hkv * d, D)) / math.sqrt(D)
    Wv = rng.standard_normal((Hkv * d, D)) / math.sqrt(D)
    return Wq, Wk, Wv


def test_stitch_offsets_hand_worked():
    # lengths (3, 1, 4): chunk offsets 0, 3, 4.
    rng = _rng(7)
    lens = (3, 1, 4)
    Ks = [rng.standard_normal((n, 2, 8)) for n in lens]
    Vs = [rng.standard_normal((n, 2, 8)) for n in lens]
    Kf, Vf = orc.stitch_rerotate(Ks, Vs, 1e4)
    assert Kf.shape == (8, 2, 8)
    assert np.array_equal(Kf[0:3], Ks[0])               # offset 0: unchanged
    for row, (ci, r, o) in enumerate([(0, 0, 0), (0, 1, 0), (0, 2, 0), (1, 0, 3),
                                      (2, 0, 4), (2, 1, 4), (2, 2, 4), (2, 3, 4)]):
        d = 8
        for j in range(d // 2):
            a = o * 1e4 ** (-(2.0 * j) / d)
            x, y = Ks[ci][r, :, j], Ks[ci][r, :, j + 4]
            assert np.allclose(Kf[row, :, j], x * math.cos(a) - y * math.sin(a), atol=1e-14)
            assert np.allclose(Kf[row, :, j + 4], y * math.cos(a) + x * math.sin(a), atol=1e-14)
    assert np.array_equal(Vf, np.concatenate(Vs))


def test_stitched_pic_equals_projection_at_fused_positions():
    # R^{o_i} R^r k = R^{o_i + r} k: with an unperturbed state the stitched
    # cache equals keys projected directly at request positions (Eq. 4 / Eq. 3).
    Wq, Wk, Wv = _tiny_model(8)
    rng = _rng(9)
    lens = [5, 9, 3, 7]
    H = rng.standard_normal((sum(lens), 32))
    Ks, Vs, o = [], [], 0
    for n in lens:
        K, V = orc.pic_precompute(H[o:o + n], Wk, Wv, 2, 8, 1e4)
        Ks.append(K)
        Vs.append(V)
        o += n
    Kf, Vf = orc.stitch_rerotate(Ks, Vs, 1e4)
    direct_k = (H @ Wk.T).reshape(-1, 2, 8)
    # direct rotation through the complex form, independent of rope_rotate
    h = 4
    for t in range(H.shape[0]):
        for j in range(h):
            th = 1e4 ** (-(2.0 * j) / 8)
            z = (direct_k[t, :, j] + 1j * direct_k[t, :, j + h]) * np.exp(1j * t * th)
            assert np.allclose(Kf[t, :, j], z.real, atol=1e-12)
            assert np.allclose(Kf[t, :, j + h], z.imag, atol=1e-12)
    assert np.allclose(Vf, (H @ Wv.T).reshape(-1, 2, 8), atol=1e-12)


# ---------------------------------------------------------------- KIVI ----

def test_kivi_roundtrip_within_half_step():
    rng = _rng(10)
    K = rng.standard_normal((50, 3, 16)) * np.exp(rng.standard_normal((1, 3, 16)))
    q, s, z = orc.kivi_quantize_key(K)
    assert q.dtype == np.uint8 and s.shape == (3, 16) and z.shape == (3, 16)
    err = np.abs(orc.kivi_dequantize(q, s[None], z[None]) - K)
    assert np.all(err <= s[None] / 2 * (1 + 1e-12) + 1e-15)
    assert q.min() == 0 and q.max() == 255
    V = rng.standard_normal((50, 3, 16))
    q, s, z = orc.kivi_quantize_value(V)
    assert s.shape == (50, 3)
    err = np.abs(orc.kivi_dequantize(q, s[..., None], z[..., None]) - V)
    assert np.all(err <= s[..., None] / 2 * (1 + 1e-12) + 1e-15)


def test_kivi_exact_on_grid():
    rng = _rng(11)
    zero = rng.integers(-8, 8, size=(2, 4)) / 4.0
    scale = rng.integers(1, 9, size=(2, 4)) / 64.0
    codes = rng.integers(0, 256, size=(20, 2, 4)).astype(np.float64)
    codes[0], codes[1] = 0, 255            # each channel spans the full range
    K = zero + codes * scale
    q, s, z = orc.kivi_quantize_key(K)
    assert np.array_equal(q.astype(np.float64), codes)
    assert np.array_equal(orc.kivi_dequantize(q, s[None], z[None]), K)


def test_kivi_constant_channel_and_int4():
    K = np.ones((10, 1, 4)) * 3.25
    q, s, z = orc.kivi_quantize_key(K)
    assert np.all(q == 0) and np.all(s == 0) and np.all(z == 3.25)
    assert np.array_equal(orc.kivi_dequantize(q, s[None], z[None]), K)
    q, s, z = orc.kivi_quantize_value(_rng(12).standard_normal((6, 2, 8)), bits=4)
    assert q.max() == 15 and q.min() == 0


def test_kivi_key_stats_are_per_channel_over_tokens():
    rng = _rng(13)
    K = rng.standard_normal((30, 2, 8))
    _, s0, _ = orc.kivi_quantize_key(K)
    K2 = K.copy()
    K2[4, 1, 5] = 100.0                    # only channel (head 1, j 5) changes
    _, s1, _ = orc.kivi_quantize_key(K2)
    changed = s0 != s1
    assert changed[1, 5] and changed.sum() == 1


# ----------------------------------------------------------- deviation ----

def test_deviation_zero_for_unperturbed_tokens():
    Wq, Wk, Wv = _tiny_model(14)
    H = _rng(15).standard_normal((40, 32))
    _, V = orc.pic_precompute(H, Wk, Wv, 2, 8, 1e4)
    sc = orc.deviation_scores(H, Wv, V, 2, 8)
    assert np.max(np.abs(sc)) < 1e-12


def test_deviation_hand_worked_2d():
    W = np.eye(2)
    H = np.array([[1.0, 0.0], [1.0, 0.0], [0.0, 2.0], [3.0, 0.0]])
    Vc = np.array([[1.0, 1.0], [-5.0, 0.0], [7.0, 0.0], [0.0, 0.0]]).reshape(4, 1, 2)
    sc = orc.deviation_scores(H, W, Vc, 1, 2)
    assert abs(sc[0] - (1 - 1 / math.sqrt(2))) < 1e-15      # 45 degrees
    assert abs(sc[1] - 2.0) < 1e-15                          # opposite
    assert abs(sc[2] - 1.0) < 1e-15                          # orthogonal
    assert abs(sc[3] - 1.0) < 1e-15                          # zero cached vector


def test_deviation_averages_over_kv_heads():
    W = np.eye(4)
    H = np.array([[1.0, 2.0, 3.0, -1.0], [1.0, 2.0, 3.0, -1.0]])
    Vc = np.array([[[2.0, 4.0], [-3.0, 1.0]],        # head 0 parallel, head 1 opposite
                   [[2.0, 4.0], [1.0, 3.0]]])        # head 0 parallel, head 1 orthogonal
    sc = orc.deviation_scores(H, W, Vc, 2, 2)
    assert abs(sc[0] - 1.0) < 1e-15 and abs(sc[1] - 0.5) < 1e-15


def test_deviation_invariant_to_positive_rescale():
    Wq, Wk, Wv = _tiny_model(16)
    rng = _rng(17)
    H = rng.standard_normal((12, 32))
    _, V = orc.pic_precompute(rng.standard_normal((12, 32)), Wk, Wv, 2, 8, 1e4)
    a = orc.deviation_scores(H, Wv, V, 2, 8)
    b = orc.deviation_scores(H * rng.uniform(0.1, 10, size=(12, 1)), Wv, V, 2, 8)
    assert np.max(np.abs(a - b)) < 1e-13


# ---------------------------------------------------------------- top-k ----

def _brute_topk(s, k):
    # among the k-subsets with the largest sum, the lexicographically smallest
    best, best_set = None, None
    for comb in itertools.combinations(range(len(s)), k):
        tot = sum(float(s[i]) for i in comb)
        if best is None or tot > best + 0.0 or (tot == best and comb < best_set):
            best, best_set = tot, comb
    return list(best_set)


def test_topk_matches_subset_brute_force_with_ties():
    rng = _rng(18)
    for trial in range(40):
        n = int(rng.integers(1, 10))
        s = rng.integers(-2, 3, size=n).astype(np.float32) * np.float32(0.25)
        for k in range(n + 1):
            assert orc.select_topk(s, k).tolist() == _brute_topk(s, k)


def test_topk_edge_cases():
    s = np.full(20, 0.5, np.float32)
    assert orc.select_topk(s, 7).tolist() == list(range(7))
    assert orc.select_topk(s, 0).tolist() == []
    assert orc.select_topk(np.arange(5, dtype=np.float32), 5).tolist() == [0, 1, 2, 3, 4]
    z = np.array([0.0, -0.0, 1.0, -0.0], np.float32)
    z[0] = -0.0
    assert orc.select_topk(z, 2).tolist() == [0, 2]          # -0 == +0, lower index wins
    with pytest.raises(ValueError):
        orc.select_topk(np.array([1.0, np.nan], np.float32), 1)


def test_k_from_ratio():
    assert orc.k_from_ratio(0.30, 256) == 76
    assert orc.k_from_ratio(0.15, 4096) == 614
    assert orc.k_from_ratio(0.30, 10240) == 3072
    assert orc.k_from_ratio(0.10, 32768) == 3276
    assert orc.k_from_ratio(0.29, 100) == 29        # 0.29 * 100 = 28.999999999999996
    assert orc.k_from_ratio(1.0, 33) == 33 and orc.k_from_ratio(0.0, 33) == 0
    assert orc.k_from_ratio(1.5, 10) == 10 and orc.k_from_ratio(-0.1, 10) == 0


# ------------------------------------------------------------ attention ----

def _complex_rope(x, pos, base):
    d = x.shape[-1]
    h = d // 2
    th = np.array([base ** (-(2.0 * j) / d) for j in range(h)])
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * np.asarray(pos, np.float64)[..., None] * th)
    return np.concatenate([z.real, z.imag], axis=-1)


def _sdpa_full_prefill(H, Wq, Wk, Wv, Hq, Hkv, d, base):
    T = H.shape[0]
    pos = np.arange(T)[:, None]
    q = _complex_rope((H @ Wq.T).reshape(T, Hq, d), pos, base)
    k = _complex_rope((H @ Wk.T).reshape(T, Hkv, d), pos, base)
    v = (H @ Wv.T).reshape(T, Hkv, d)
    g = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(g, dim=0)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(g, dim=0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    return o[0].permute(1, 0, 2).numpy(), k, v


def _pic_chunks(H, lens, Wk, Wv, Hkv, d, base):
    Ks, Vs, o = [], [], 0
    for n in lens:
        K, V = orc.pic_precompute(H[o:o + n], Wk, Wv, Hkv, d, base)
        Ks.append(K)
        Vs.append(V)
        o += n
    return Ks, Vs


def test_ratio_one_reproduces_full_prefill():
    Hq, Hkv, d, D, base = 4, 2, 8, 32, 1e4
    Wq, Wk, Wv = _tiny_model(19, D, Hq, Hkv, d)
    rng = _rng(20)
    lens, nq = [6, 11, 5], 4
    N = sum(lens)
    Hc = rng.standard_normal((N + nq, D))
    H = Hc + 0.3 * rng.standard_normal(Hc.shape)        # perturbed current state
    Ks, Vs = _pic_chunks(Hc, lens, Wk, Wv, Hkv, d, base)
    res = orc.layer_step(H, Wq, Wk, Wv, Ks, Vs, 1.0, Hq, Hkv, d, base)
    O_ref, k_ref, v_ref = _sdpa_full_prefill(H, Wq, Wk, Wv, Hq, Hkv, d, base)
    assert res["S"].tolist() == list(range(N + nq))
    assert np.max(np.abs(res["O"] - O_ref)) < 1e-12
    assert np.max(np.abs(res["K_fused"] - k_ref)) < 1e-12
    assert np.max(np.abs(res["V_fused"] - v_ref)) < 1e-12


def _brute_attention_row(q, K, V, p):
    # explicit per-element softmax with Python loops
    d = q.shape[0]
    logits = [sum(q[c] * K[j][c] for c in range(d)) / math.sqrt(d) for j in range(p + 1)]
    m = max(logits)
    w = [math.exp(l - m) for l in logits]
    z = sum(w)
    return [sum(w[j] * V[j][c] for j in range(p + 1)) / z for c in range(d)]


def test_selected_rows_brute_force_tiny():
    Hq, Hkv, d, D, base = 4, 2, 4, 16, 1e4
    Wq, Wk, Wv = _tiny_model(21, D, Hq, Hkv, d)
    rng = _rng(22)
    lens, nq = [4, 5, 3], 3
    N, T = 12, 15
    Hc = rng.standard_normal((T, D))
    H = Hc + 0.5 * rng.standard_normal((T, D))
    Ks, Vs = _pic_chunks(Hc, lens, Wk, Wv, Hkv, d, base)
    Kc, Vc = orc.stitch_rerotate(Ks, Vs, base)
    Kf0 = np.zeros((T, Hkv, d))
    Vf0 = np.zeros((T, Hkv, d))
    Kf0[:N], Vf0[:N] = Kc, Vc
    idx = np.array([0, 4, 7, 11])
    Kf, Vf, O, S = orc.recompute_selected(H, Wq, Wk, Wv, idx, N, Kf0, Vf0, Hq, Hkv, d, base)
    assert S.tolist() == [0, 4, 7, 11, 12, 13, 14]
    # fused cache by hand: fresh rows at S, stitched PIC elsewhere
    Kexp, Vexp = Kf0.copy(), Vf0.copy()
    for s in S:
        Kexp[s] = _complex_rope((H[s] @ Wk.T).reshape(Hkv, d), s, base)
        Vexp[s] = (H[s] @ Wv.T).reshape(Hkv, d)
    assert np.max(np.abs(Kf - Kexp)) < 1e-12 and np.max(np.abs(Vf - Vexp)) < 1e-12
    g = Hq // Hkv
    for r, s in enumerate(S):
        q = _complex_rope((H[s] @ Wq.T).reshape(Hq, d), s, base)
        for h in range(Hq):
            want = _brute_attention_row(q[h], Kexp[:, h // g], Vexp[:, h // g], int(s))
            assert np.max(np.abs(O[r, h] - np.array(want))) < 1e-12


def test_ratio_zero_is_direct_reuse():
    Hq, Hkv, d, D, base = 4, 2, 8, 32, 1e4
    Wq, Wk, Wv = _tiny_model(23, D, Hq, Hkv, d)
    rng = _rng(24)
    lens, nq = [7, 9], 5
    Hc = rng.standard_normal((21, D))
    H = Hc + 0.2 * rng.standard_normal(Hc.shape)
    Ks, Vs = _pic_chunks(Hc, lens, Wk, Wv, Hkv, d, base)
    res = orc.layer_step(H, Wq, Wk, Wv, Ks, Vs, 0.0, Hq, Hkv, d, base)
    assert res["idx"].tolist() == [] and res["S"].tolist() == list(range(16, 21))
    assert np.array_equal(res["K_fused"][:16], res["K_stitched"])
    assert np.array_equal(res["V_fused"][:16], res["V_stitched"])


def test_figure3_structure():
    g = json.load(open(os.path.join(GOLDEN, "fig3_structure.json")))
    Hq, Hkv, d, D, base = 2, 1, 4, 8, 1e4
    Wq, Wk, Wv = _tiny_model(25, D, Hq, Hkv, d)
    rng = _rng(26)
    n = g["n_tokens"]
    Hc = rng.standard_normal((n, D))
    H = Hc + 0.5 * rng.standard_normal((n, D))
    Ks, Vs = _pic_chunks(Hc, [2, 2, 2], Wk, Wv, Hkv, d, base)
    Kc, Vc = orc.stitch_rerotate(Ks, Vs, base)
    idx = np.array(g["selected_zero_based"])
    Kf, Vf, O, S = orc.recompute_selected(H, Wq, Wk, Wv, idx, n, Kc, Vc, Hq, Hkv, d, base)
    for t, src in enumerate(g["fused_entry_source"]):
        fresh_v = (H[t] @ Wv.T).reshape(Hkv, d)
        if src == "PIC":
            assert np.array_equal(Kf[t], Kc[t]) and np.array_equal(Vf[t], Vc[t])
        else:
            assert np.allclose(Vf[t], fresh_v, atol=1e-13)
    # the row of t4 reads t1 (PIC), t2 (New), t3 (PIC), t4 (New)
    srcs = g["prefix_read_by_t4"]
    Kmix = np.stack([Kc[0], Kf[1], Kc[2], Kf[3]])
    Vmix = np.stack([Vc[0], Vf[1], Vc[2], Vf[3]])
    assert list(srcs.values()) == ["PIC", "New", "PIC", "New"]
    q = _complex_rope((H[3] @ Wq.T).reshape(Hq, d), 3, base)
    r = S.tolist().index(3)
    for h in range(Hq):
        want = _brute_attention_row(q[h], Kmix[:, 0], Vmix[:, 0], 3)
        assert np.max(np.abs(O[r, h] - np.array(want))) < 1e-12


def test_gqa_query_head_reads_kv_head_h_div_g():
    Hq, Hkv, d, D, base = 4, 2, 4, 16, 1e4
    Wq, Wk, Wv = _tiny_model(27, D, Hq, Hkv, d)
    Wv = Wv.copy()
    Wv[d:] = 0.0                            # KV head 1 has zero values
    rng = _rng(28)
    H = rng.standard_normal((6, D))
    Kf0 = np.zeros((6, Hkv, d))
    Vf0 = np.zeros((6, Hkv, d))
    _, _, O, _ = orc.recompute_selected(H, Wq, Wk, Wv, np.arange(6), 6, Kf0, Vf0, Hq, Hkv, d, base)
    assert np.all(O[:, 2:] == 0.0)         # heads 2, 3 -> KV head 1
    assert np.all(np.abs(O[1:, :2]).sum(axis=-1) > 0)


def test_pic_differs_from_full_only_when_perturbed():
    # Eq. 5: independently cached chunks miss the current context; in the
    # synthetic recipe the perturbation e_t stands for that missing context.
    Hq, Hkv, d, D, base = 4, 2, 8, 32, 1e4
    Wq, Wk, Wv = _tiny_model(29, D, Hq, Hkv, d)
    rng = _rng(30)
    Hc = rng.standard_normal((24, D))
    Ks, Vs = _pic_chunks(Hc, [8, 8, 8], Wk, Wv, Hkv, d, base)
    Kc, Vc = orc.stitch_rerotate(Ks, Vs, base)
    _, k_full, v_full = _sdpa_full_prefill(Hc, Wq, Wk, Wv, Hq, Hkv, d, base)
    assert np.max(np.abs(Kc - k_full)) < 1e-12 and np.max(np.abs(Vc - v_full)) < 1e-12
    Hp = Hc + 0.1 * rng.standard_normal(Hc.shape)
    _, k_full, v_full = _sdpa_full_prefill(Hp, Wq, Wk, Wv, Hq, Hkv, d, base)
    assert np.max(np.abs(Kc - k_full)) > 1e-3 and np.max(np.abs(Vc - v_full)) > 1e-3


def test_layer_step_scores_and_selection_consistent():
    Hq, Hkv, d, D, base = 4, 2, 8, 32, 1e4
    Wq, Wk, Wv = _tiny_model(31, D, Hq, Hkv, d)
    rng = _rng(32)
    lens, nq = [10, 10, 10], 6
    Hc = rng.standard_normal((36, D))
    e = np.exp(-3 + 1.5 * rng.standard_normal(36))
    H = Hc + e[:, None] * rng.standard_normal(Hc.shape)
    Ks, Vs = _pic_chunks(Hc, lens, Wk, Wv, Hkv, d, base)
    res = orc.layer_step(H, Wq, Wk, Wv, Ks, Vs, 0.3, Hq, Hkv, d, base)
    sc, idx = res["score"], res["idx"]
    assert len(idx) == 9
    unsel = np.setdiff1d(np.arange(30), idx)
    assert sc[idx].min() >= sc[unsel].max()
    # the most perturbed tokens deviate most
    assert np.corrcoef(np.argsort(np.argsort(e[:30])), np.argsort(np.argsort(sc)))[0, 1] > 0.5


# Static selectors (QCFuse related work, EPIC boundary tokens; KVBoost 4.6.1,
# SelectiveRecompute seam windows)
def test_static_select_hand_worked():
    # chunks of 5, 3 and 4 tokens at positions 0, 5 and 8
    s, l = [0, 5, 8], [5, 3, 4]
    assert orc.static_select(s, l, 12, "chunk_head", 2).tolist() == [0, 1, 5, 6, 8, 9]
    assert orc.static_select(s, l, 12, "chunk_head", 4).tolist() == [0, 1, 2, 3, 5, 6, 7, 8, 9, 10, 11]
    assert orc.static_select(s, l, 12, "seam_tail", 2).tolist() == [3, 4, 6, 7]
    # windows overlap and reach back across a short chunk; the start clamps at 0
    assert orc.static_select(s, l, 12, "seam_tail", 4).tolist() == [1, 2, 3, 4, 5, 6, 7]
    assert orc.static_select(s, l, 12, "seam_tail", 9).tolist() == list(range(8))
    assert orc.static_select(s, l, 12, "seam_tail", 0).tolist() == []
    assert orc.static_select([0], [12], 12, "seam_tail", 16).tolist() == []   # one chunk: no seam


def test_static_select_counts_from_the_pages():
    # KVBoost 4.6.1: R = 16 and two seams in a 512-token prompt: 32 tokens
    assert len(orc.static_select([0, 170, 340], [170, 170, 172], 512, "seam_tail", 16)) == 32
    # chunk heads: every chunk contributes min(n, len) positions
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 40, size=20)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    for n in (0, 1, 7, 64):
        got = orc.static_select(starts, lens, int(lens.sum()), "chunk_head", n)
        assert len(got) == int(np.minimum(lens, n).sum())
        assert np.all(np.diff(got) > 0)


# Query-aware attention mass (QCFuse section 3.2.1, Eqs. 9-10; Eq. 20)
def _mass_hand_setup(n_q_heads, n_kv_heads, q_head, key_head, hot):
    """d = 2 (one RoPE pair, theta_0 = 1 radian per position), N = 2 context
    keys, one query token at position 2.  W_Q maps x = (1, 0) to q = (1, 0)
    for query head `q_head` only; after R^2 that q is (cos 2, sin 2).  Key
    `hot` of KV head `key_head` is sqrt(2) ln 3 (cos 2, sin 2), every other
    key is 0: that head's logits are ln 3 at `hot` and 0 elsewhere, so its
    weights are 3/4 and 1/4; every other query head (q = 0) spreads 1/2, 1/2."""
    Wq = np.zeros((n_q_heads * 2, 2))
    Wq[2 * q_head:2 * q_head + 2] = np.eye(2)
    K = np.zeros((2, n_kv_heads, 2))
    K[hot, key_head] = math.sqrt(2.0) * math.log(3.0) * np.array([math.cos(2.0), math.sin(2.0)])
    return np.array([[1.0, 0.0]]), Wq, K


def test_attention_mass_hand_worked_d2():
    H, Wq, K = _mass_hand_setup(2, 1, 0, 0, 1)
    got = orc.attention_mass_scores(H, Wq, K, 2, 1, 2, 1e4)
    assert np.allclose(got, [0.25 + 0.5, 0.75 + 0.5], atol=1e-12)


def test_attention_mass_gqa_query_head_reads_kv_head_h_div_g():
    # Hq = 4, Hkv = 2: query head 2 reads KV head 1 (not 2 % 2 = 0)
    H, Wq, K = _mass_hand_setup(4, 2, 2, 1, 0)
    K[1, 0] = K[0, 1]              # KV head 0 would favour the other key
    got = orc.attention_mass_scores(H, Wq, K, 4, 2, 2, 1e4)
    assert np.allclose(got, [0.75 + 1.5, 0.25 + 1.5], atol=1e-12)


def test_attention_mass_matches_complex_form_and_library_softmax():
    # d = 4: pairs (0, 2) and (1, 3) as complex numbers turned by e^{i p theta_j};
    # q . k = Re(sum_j z_q,j conj(z_k,j)); the softmax is scipy's.
    from scipy.special import softmax
    rng = _rng(31)
    n, n_query, hq, hkv, d, base = 7, 3, 4, 2, 4, 100.0
    H = rng.standard_normal((n_query, 5))
    Wq = rng.standard_normal((hq * d, 5))
    K = rng.standard_normal((n, hkv, d))
    want = np.zeros(n)
    for u in range(n_query):
        qraw = (Wq @ H[u]).reshape(hq, d)
        for h in range(hq):
            logits = []
            for t in range(n):
                acc = 0.0
                for j in range(2):
                    theta = base ** (-2.0 * j / d)
                    zq = complex(qraw[h, j], qraw[h, j + 2]) * complex(
                        math.cos((n + u) * theta), math.sin((n + u) * theta))
                    zk = complex(K[t, h // 2, j], K[t, h // 2, j + 2])
                    acc += (zq * zk.conjugate()).real
                logits.append(acc / 2.0)                       # 1 / sqrt(4)
            want += softmax(np.array(logits))
    got = orc.attention_mass_scores(H, Wq, K, hq, hkv, d, base)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_attention_mass_invariants():
    rng = _rng(32)
    n, n_query, hq, hkv, d, D = 40, 6, 8, 2, 16, 24
    H = rng.standard_normal((n_query, D))
    Wq = rng.standard_normal((hq * d, D)) * 0.5
    K = rng.standard_normal((n, hkv, d))
    I = orc.attention_mass_scores(H, Wq, K, hq, hkv, d, 1e4)
    # every (query token, head) spreads a total weight of 1 over the context
    assert abs(I.sum() - n_query * hq) < 1e-9
    assert np.all(I > 0)
    # the same vector added to every key of a head moves each logit row by a
    # constant: the softmax, hence the mass, does not change
    shift = rng.standard_normal((1, hkv, d)) * 3.0
    assert np.allclose(orc.attention_mass_scores(H, Wq, K + shift, hq, hkv, d, 1e4), I,
                       rtol=1e-10, atol=1e-12)
    # zero keys: uniform weights
    assert np.allclose(orc.attention_mass_scores(H, Wq, 0 * K, hq, hkv, d, 1e4),
                       n_query * hq / n, atol=1e-12)
    # no query token: nothing spread; no context: nothing to score
    assert np.array_equal(orc.attention_mass_scores(H[:0], Wq, K, hq, hkv, d, 1e4), np.zeros(n))
    assert orc.attention_mass_scores(H, Wq, K[:0], hq, hkv, d, 1e4).shape == (0,)


# Key deviation over layers (KVBoost section 4.6.2, Alg. 2 step 2 as printed)
def _rot2(angle, scale=1.0):
    return scale * np.array([math.cos(angle), math.sin(angle)])


def test_key_deviation_hand_worked_d2():
    # d = 2 (theta_0 = 1 radian per position), W_K = I, x_t = (1, 0): the fresh
    # key of token t is (cos t, sin t).  Stale keys turned further by phi_t
    # (and scaled, which a cosine ignores) give delta_t = 1 - cos(phi_t).
    phi, scale = [0.0, math.pi / 3, math.pi], [1.0, 2.0, 0.5]
    H = np.array([[1.0, 0.0]] * 3)
    K = np.stack([_rot2(t + p, s) for t, (p, s) in enumerate(zip(phi, scale))])[:, None, :]
    got = orc.key_deviation_scores([H], [np.eye(2)], [K], 1, 2, 1e4)
    assert np.allclose(got, [0.0, 0.5, 2.0], atol=1e-12)
    # a second layer whose stale keys are all a quarter turn off (delta 1):
    # the two layers' deviations are averaged
    K2 = np.stack([_rot2(t + math.pi / 2) for t in range(3)])[:, None, :]
    got2 = orc.key_deviation_scores([H, H], [np.eye(2), np.eye(2)], [K, K2], 1, 2, 1e4)
    assert np.allclose(got2, [0.5, 0.75, 1.5], atol=1e-12)
    # a zero stale key has cosine 0
    got3 = orc.key_deviation_scores([H], [np.eye(2)], [0 * K], 1, 2, 1e4)
    assert np.allclose(got3, [1.0, 1.0, 1.0], atol=1e-12)


def test_key_deviation_averages_over_key_heads():
    # Hkv = 2 heads of d = 2 reading the same x: head 0 matches, head 1 is a
    # quarter turn off -> 1 - (1 + 0) / 2
    H = np.array([[1.0, 0.0]] * 2)
    Wk = np.vstack([np.eye(2), np.eye(2)])
    K = np.stack([np.stack([_rot2(t), _rot2(t + math.pi / 2)]) for t in range(2)])
    got = orc.key_deviation_scores([H], [Wk], [K], 2, 2, 1e4)
    assert np.allclose(got, [0.5, 0.5], atol=1e-12)


def test_key_deviation_zero_on_unperturbed_stitched_cache():
    # QCFuse Eqs. 3-4 with KVBoost Eq. 3: a stitched PIC key of an unperturbed
    # token equals its fresh key at the request position, in every layer;
    # perturbing the probe's input of some tokens raises exactly those
    rng = _rng(41)
    lens = [5, 9, 4]
    n = sum(lens)
    layers = []
    for l in range(3):
        Wq, Wk, Wv = _tiny_model(50 + l)
        H = rng.standard_normal((n, 32))
        starts = np.cumsum([0] + lens[:-1])
        Kc, Vc = zip(*[orc.pic_precompute(H[s:s + ln], Wk, Wv, 2, 8, 1e4)
                       for s, ln in zip(starts, lens)])
        K, _ = orc.stitch_rerotate(list(Kc), list(Vc), 1e4)
        layers.append((H, Wk, K))
    Hs, Ws, Ks = zip(*layers)
    assert np.max(np.abs(orc.key_deviation_scores(Hs, Ws, Ks, 2, 8, 1e4))) < 1e-12
    bumped = [h.copy() for h in Hs]
    bumped[1][[3, 11]] += 0.5 * rng.standard_normal((2, 32))
    d = orc.key_deviation_scores(bumped, Ws, Ks, 2, 8, 1e4)
    assert np.all(d[[3, 11]] > 1e-6) and np.max(np.abs(np.delete(d, [3, 11]))) < 1e-12
