"""Rounding-aware comparison of attention rows of a bf16 layer.

A bf16 layer stores q, k, v in bf16.  The GPU rounds values it accumulated
in fp32, the oracle rounds fp64 values; where an fp64 value lies closer to a
bf16 rounding midpoint than the fp32 accumulation error, the two sides may
round it to adjacent bf16 numbers, and both are correct.  For most rows this
changes nothing; for a row whose softmax splits between keys with very
different values (heavy-tailed perturbation recipes make such keys) a single
such element can move the output far beyond 2e-2.

This module marks those ambiguous elements from the oracle's own values,
evaluates with the attention definition how far flipping each one to its
other bf16 neighbour moves each checked output row, and returns a
per-(row, head) allowance: the stated tolerance plus twice the summed
movement.  Rows without ambiguous elements that matter keep the stated
tolerance.
"""

from __future__ import annotations

import math

import numpy as np

from oracle import fusion as orc

U32 = 2.0 ** -24          # fp32 unit roundoff


def _neighbours(x64: np.ndarray):
    """(stored bf16 value, its other bf16 neighbour around x64)."""
    r = orc.round_bf16(x64)
    _, e = np.frexp(x64)
    ulp = np.ldexp(1.0, e - 8)
    other = np.where(x64 >= r, r + ulp, r - ulp)
    return r, other


def ambiguous(x64: np.ndarray, err: np.ndarray) -> np.ndarray:
    """True where the distance to the bf16 rounding midpoint is within the
    error bound, so either neighbour is a correct rounding."""
    r, other = _neighbours(x64)
    return np.abs(x64 - 0.5 * (r + other)) <= err


def projection_error(X: np.ndarray, W: np.ndarray, x64: np.ndarray) -> np.ndarray:
    """Bound on |fp32-accumulated x - exact x| for x = X W^T: the rounding
    errors of a length-K sum behave like a random walk over the partial sums,
    std about u sqrt(K) ||a o b||_2 / sqrt(2); four standard deviations, plus
    one rounding of the result."""
    K = X.shape[1]
    l2 = np.sqrt((X * X) @ (W * W).T)
    return 4.0 * U32 * math.sqrt(K / 2.0) * l2.reshape(x64.shape) + U32 * np.abs(x64)


def rotated_error(err: np.ndarray, x: np.ndarray, pos, base: float) -> np.ndarray:
    """Carry an error bound through R^pos, adding the fp32 rounding of the
    rotation and an angle error of 4e-7 rad (fp32 angle reduction)."""
    d = x.shape[-1]
    h = d // 2
    ang = np.asarray(pos, np.float64)[..., None] * orc.rope_inv_freq(d, base)
    c, s = np.abs(np.cos(ang)), np.abs(np.sin(ang))
    ea, eb = err[..., :h], err[..., h:]
    mag = np.abs(x[..., :h]) + np.abs(x[..., h:])
    extra = (2.0 * U32 + 4e-7) * mag
    return np.concatenate([ea * c + eb * s + extra, eb * c + ea * s + extra], axis=-1)


def allowance(H, Wq, Wk, Wv, S, Kf, Vf, O_ref, rows, n_q_heads, n_kv_heads, head_dim, base,
              tol=2e-2):
    """Per-(checked row, head) allowance for max |O_gpu - O_oracle|.

    ``Kf``/``Vf``: the oracle's fused cache after the scatter (stored
    values); ``O_ref``: its attention rows for ``rows`` (indices into S).
    Returns (allowance [len(rows), Hq], stated tolerance, count of
    (row, head) pairs whose allowance exceeds the stated tolerance)."""
    d = head_dim
    g = n_q_heads // n_kv_heads
    X = np.asarray(H, np.float64)[S]
    Wq, Wk, Wv = (np.asarray(w, np.float64) for w in (Wq, Wk, Wv))
    R = X.shape[0]
    q0 = (X @ Wq.T).reshape(R, n_q_heads, d)
    k0 = (X @ Wk.T).reshape(R, n_kv_heads, d)
    v64 = (X @ Wv.T).reshape(R, n_kv_heads, d)
    q64 = orc.rope_rotate(q0, S[:, None], base)
    k64 = orc.rope_rotate(k0, S[:, None], base)
    eq = rotated_error(projection_error(X, Wq, q0), q0, S[:, None], base)
    ek = rotated_error(projection_error(X, Wk, k0), k0, S[:, None], base)
    ev = projection_error(X, Wv, v64)
    q_st, q_ot = _neighbours(q64)
    _, k_ot = _neighbours(k64)
    _, v_ot = _neighbours(v64)
    amb_q = ambiguous(q64, eq)
    amb_k = ambiguous(k64, ek)
    amb_v = ambiguous(v64, ev)
    scale = 1.0 / math.sqrt(d)
    base_tol = tol * float(np.max(np.abs(O_ref)))
    out = np.full((len(rows), n_q_heads), base_tol)
    for o, r in enumerate(rows):
        p = int(S[r])
        ref = np.nonzero(S <= p)[0]          # refreshed rows in this row's prefix
        jpos = S[ref]
        for h in range(n_q_heads):
            kv = h // g
            Kj = Kf[:p + 1, kv]
            Vj = Vf[:p + 1, kv]
            q = q_st[r, h]
            l = (Kj @ q) * scale
            m = l.max()
            w = np.exp(l - m)
            Z = w.sum()
            Ov = (w @ Vj) / Z
            move = 0.0
            # flips of this row's q
            for c in np.nonzero(amb_q[r, h])[0]:
                w2 = np.exp(l + (q_ot[r, h, c] - q[c]) * Kj[:, c] * scale - m)
                move += float(np.max(np.abs((w2 @ Vj) / w2.sum() - Ov)))
            # flips of refreshed keys: one logit changes per flipped element
            ai, ac = np.nonzero(amb_k[ref, kv])
            if ai.size:
                j = jpos[ai]
                lj = l[j] + q[ac] * (k_ot[ref[ai], kv, ac] - Kf[j, kv, ac]) * scale
                wj = np.exp(np.minimum(lj - m, 700.0))
                Z2 = Z - w[j] + wj
                dev = np.max(np.abs(Vj[j] - Ov), axis=-1)
                move += float(np.sum(np.abs(wj - w[j]) * dev / Z2))
            # flips of refreshed values
            ai, ac = np.nonzero(amb_v[ref, kv])
            if ai.size:
                j = jpos[ai]
                move += float(np.sum(w[j] / Z * np.abs(v_ot[ref[ai], kv, ac] - Vf[j, kv, ac])))
            out[o, h] = base_tol + 2.0 * move
    return out, base_tol, int(np.sum(out > base_tol * (1 + 1e-12)))
