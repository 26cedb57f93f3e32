"""Oracle: a plain, slow, fp64 CPU statement of one layer-step of RAG
KV-cache fusion with RoPE re-rotation and selective recomputation.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this module: only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library; numpy (fp64) is the only dependency, and ``numpy.matmul`` is the
only library primitive used as a step.

Sources (page title, then section / equation):

* QCFuse: Query-Aware Cache Fusion via Compressed View for Efficient RAG
  Serving -- section 2.1 (Eqs. 1-7): context ``C = [c_1; ...; c_m]`` with the
  user query after it; per-chunk position-independent caches built at
  chunk-local positions (Eq. 3); position remapping and stitching (Eq. 4);
  selective recomputation with ratio ``rho = |P| / N`` over a partially fused
  prefix (Eq. 6); the fused cache (Eq. 7); top-k selection (Eq. 11).
* KVBoost: Chunk-Level KV Cache Reuse with Deviation-Guided Recomputation --
  section 3.1 (Eqs. 1-2, projections and causal attention), section 3.2
  (Eq. 3, RoPE and its relative-offset property), section 4.5 (Eq. 7, KIVI
  asymmetric quantisation), section 4.6.1 (Alg. 1, SelectiveRecompute seam
  windows), section 4.6.2 (Alg. 2, deviation -> top-k -> patch).
* QCFuse section 3.2.1 (Eqs. 9-10) and section 3.4.2 (Eq. 20): the
  query-aware importance of a context token, the attention mass the user
  query's tokens and heads put on it, summed over the critical layers.

Readings taken where the pages leave a step open:

* RoPE uses the rotate-half pairing ``(j, j + d/2)`` with
  ``theta_j = base^(-2j/d)``; KVBoost targets HuggingFace RoPE models.
* The deviation is computed on V at one layer (1 - cosine between the
  freshly projected V and the cached V, averaged over KV heads); KVBoost's
  Alg. 2 writes it on K averaged over all layers and heads.  ``key_deviation_scores`` states that printed form: the fresh key is
  ``R^t W_K x_t`` at the token's request position, the stale key the
  stitched cache's, and H is the number of key (KV) heads.
* Query rows are always recomputed, never scored, and are not counted in
  ``N`` or ``k``.  ``k = floor(rho * N + 1e-9)``; the epsilon keeps binary
  fractions such as ``0.29 * 100`` from dropping a token.
* Refreshed K/V of all selected rows are written before any attention row
  is evaluated, so a selected row sees the refreshed entries of earlier
  selected rows (QCFuse Eq. 6 text: "already refreshed prefix positions").
* The attention mass of Eq. 10 is taken with the softmax over the context
  keys only (the arguments the equation names: the query states and the
  context keys), not over the context plus the query's own keys; the
  query's inputs at the layer are the query rows of ``H``.
* Top-k breaks ties toward the lower token index; ``-0`` counts as ``+0``;
  a NaN score is an error.
* KIVI codes are unsigned ``0 .. 2^b - 1`` with ``zero = min``; a channel
  (or token) whose max equals its min gets scale 0 and code 0.
* A bf16 layer stores its fused cache and its Q in bf16: with ``store=``
  ``round_bf16`` the stitched keys and values and the fresh q, k, v are
  rounded to bf16 where they are materialised, and attention reads the
  stored values.  Every other step stays in fp64.

Every function is pinned by tests that do not re-run its own formula:
closed forms, special cases, a textbook library routine, brute force.
"""

from __future__ import annotations

import math
from typing import List, Optional, Sequence

import numpy as np

F64 = np.float64

__all__ = [
    "round_bf16", "rope_inv_freq", "rope_rotate", "pic_precompute", "kivi_quantize_key",
    "kivi_quantize_value", "kivi_dequantize", "stitch_rerotate",
    "deviation_scores", "key_deviation_scores", "k_from_ratio", "select_topk", "static_select",
    "attention_mass_scores", "selected_rows",
    "project_rows", "recompute_selected", "layer_step",
]


# --------------------------------------------------------------------------
# Storage rounding of a bf16 layer
# --------------------------------------------------------------------------

def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value (8 significant bits, ties to even),
    returned as fp64.  A bf16 layer stores its fused cache and its Q in this
    format; the oracle applies it where the layer materialises those tensors.
    Normal range only (|x| >= 2^-126), which covers every value here."""
    x = np.asarray(x, dtype=F64)
    m, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


# --------------------------------------------------------------------------
# RoPE (KVBoost section 3.2, Eq. 3)
# --------------------------------------------------------------------------

def rope_inv_freq(head_dim: int, base: float) -> np.ndarray:
    """Frequencies ``theta_j = base^(-2j/d)`` for ``j = 0 .. d/2 - 1``."""
    j = np.arange(head_dim // 2, dtype=F64)
    return np.power(F64(base), -2.0 * j / head_dim)


def rope_rotate(x: np.ndarray, pos, base: float) -> np.ndarray:
    """Apply the rotation ``R^pos`` to the last axis of ``x``.

    Pair ``(x_j, x_{j+d/2})`` is rotated by the angle ``pos * theta_j``:
    ``x'_j = x_j cos a - x_{j+d/2} sin a`` and
    ``x'_{j+d/2} = x_{j+d/2} cos a + x_j sin a``.  ``pos`` broadcasts
    against ``x.shape[:-1]``; it may be any integer (negative undoes a
    rotation).
    """
    x = np.asarray(x, dtype=F64)
    d = x.shape[-1]
    h = d // 2
    ang = np.asarray(pos, dtype=F64)[..., None] * rope_inv_freq(d, base)
    c = np.cos(ang)
    s = np.sin(ang)
    a = x[..., :h]
    b = x[..., h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


# --------------------------------------------------------------------------
# Position-independent chunk caches (QCFuse section 2.1.2, Eq. 3)
# --------------------------------------------------------------------------

def pic_precompute(H_chunk: np.ndarray, Wk: np.ndarray, Wv: np.ndarray,
                   n_kv_heads: int, head_dim: int, base: float):
    """Cache of one chunk computed alone, at chunk-local positions 0..len-1.

    With a single projection layer standing in for the model, the key of
    local token ``r`` is ``R^r (W_K x_r)`` and its value is ``W_V x_r``
    (KVBoost section 3.1, Eq. 1; section 3.2, Eq. 3).  Returns K, V of
    shape ``[len, Hkv, d]``.
    """
    H_chunk = np.asarray(H_chunk, dtype=F64)
    n = H_chunk.shape[0]
    K = (H_chunk @ np.asarray(Wk, F64).T).reshape(n, n_kv_heads, head_dim)
    V = (H_chunk @ np.asarray(Wv, F64).T).reshape(n, n_kv_heads, head_dim)
    K = rope_rotate(K, np.arange(n)[:, None], base)
    return K, V


# --------------------------------------------------------------------------
# KIVI asymmetric quantisation (KVBoost section 4.5, Eq. 7)
# --------------------------------------------------------------------------

def _kivi_quantize(x: np.ndarray, axis, bits: int):
    x = np.asarray(x, dtype=F64)
    levels = float(2 ** bits - 1)
    mn = x.min(axis=axis, keepdims=True)
    mx = x.max(axis=axis, keepdims=True)
    span = mx - mn
    safe = np.where(span > 0, span, 1.0)
    q = np.where(span > 0, np.rint((x - mn) / safe * levels), 0.0)
    return q.astype(np.uint8 if bits <= 8 else np.uint16), span / levels, mn


def kivi_quantize_key(K: np.ndarray, bits: int = 8):
    """Per-channel key quantisation of one chunk's ``[len, Hkv, d]`` keys.

    Statistics run over the chunk's tokens for each (head, channel).
    Returns ``(q [len, Hkv, d], scale [Hkv, d], zero [Hkv, d])``.
    """
    q, scale, zero = _kivi_quantize(K, 0, bits)
    return q, scale[0], zero[0]


def kivi_quantize_value(V: np.ndarray, bits: int = 8):
    """Per-token value quantisation: statistics over the head dimension of
    each (token, head).  Returns ``(q [len, Hkv, d], scale [len, Hkv],
    zero [len, Hkv])``."""
    q, scale, zero = _kivi_quantize(V, -1, bits)
    return q, scale[..., 0], zero[..., 0]


def kivi_dequantize(q: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """``x = zero + q * scale`` (scale and zero broadcast against q)."""
    return np.asarray(zero, F64) + np.asarray(q, F64) * np.asarray(scale, F64)


# --------------------------------------------------------------------------
# Position remapping and stitching (QCFuse section 2.1.2, Eq. 4)
# --------------------------------------------------------------------------

def stitch_rerotate(K_chunks: Sequence[np.ndarray], V_chunks: Sequence[np.ndarray],
                    base: float, store=None):
    """``KV^PIC(C) = [Pi_1(KV_1); ...; Pi_m(KV_m)]``.

    Chunk ``i`` starts at request position ``o_i = sum_{j<i} len_j``.  Its
    keys, cached at local positions ``r``, are rotated by ``R^{o_i}`` so that
    they carry ``R^{o_i + r}`` (KVBoost section 3.2: a key cached at 50 and
    reused at 1050 needs ``R^{1000}``); its values are copied unchanged.
    Returns the context rows ``[N, Hkv, d]`` of the fused K and V, passed
    through ``store`` (the storage rounding of the fused cache) if given.
    """
    Ks, Vs = [], []
    o = 0
    for K, V in zip(K_chunks, V_chunks):
        Ks.append(rope_rotate(K, o, base))
        Vs.append(np.asarray(V, F64))
        o += K.shape[0]
    K, V = np.concatenate(Ks, axis=0), np.concatenate(Vs, axis=0)
    if store is not None:
        K, V = store(K), store(V)
    return K, V


# --------------------------------------------------------------------------
# Deviation score (KVBoost section 4.6.2, Alg. 2 step 2, taken on V)
# --------------------------------------------------------------------------

def deviation_scores(H_ctx: np.ndarray, Wv: np.ndarray, V_cached: np.ndarray,
                     n_kv_heads: int, head_dim: int) -> np.ndarray:
    """``score_t = 1 - (1/Hkv) sum_h cos(W_V x_t [h], V_cached[t, h])``.

    ``H_ctx`` holds the current hidden states of the N context tokens,
    ``V_cached`` their stitched cached values ``[N, Hkv, d]``.  The cosine
    denominator is clamped at 1e-30 (a zero vector gives cosine 0).
    """
    H_ctx = np.asarray(H_ctx, F64)
    n = H_ctx.shape[0]
    Vn = (H_ctx @ np.asarray(Wv, F64).T).reshape(n, n_kv_heads, head_dim)
    Vc = np.asarray(V_cached, F64).reshape(n, n_kv_heads, head_dim)
    dot = np.sum(Vn * Vc, axis=-1)
    den = np.sqrt(np.sum(Vn * Vn, axis=-1)) * np.sqrt(np.sum(Vc * Vc, axis=-1))
    cos = dot / np.maximum(den, 1e-30)
    return 1.0 - cos.mean(axis=1)


def key_deviation_scores(H_ctx_layers: Sequence[np.ndarray], Wk_layers: Sequence[np.ndarray],
                         K_stale_layers: Sequence[np.ndarray], n_kv_heads: int, head_dim: int,
                         base: float) -> np.ndarray:
    """KVBoost Alg. 2 step 2 as the page writes it, on the keys of L layers:
    ``delta_t = 1 - (1/(L Hkv)) sum_{l,h} cos(K~_t^(l,h), K_t^(l,h))``.

    Per layer l: ``H_ctx_layers[l]`` ``[N, D]`` holds the layer's inputs at
    the N context tokens (the probe pass), ``Wk_layers[l]`` its key
    projection, ``K_stale_layers[l]`` ``[N, Hkv, d]`` the assembled keys (the
    stitched cache).  The fresh key of token t is ``K~_t = R^t W_K x_t``, at
    the token's request position t, as the probe pass places it.  H in the
    formula is the number of key heads, Hkv.  The cosine denominator is
    clamped at 1e-30 (a zero vector gives cosine 0).
    """
    n_layers = len(H_ctx_layers)
    if n_layers == 0 or len(Wk_layers) != n_layers or len(K_stale_layers) != n_layers:
        raise ValueError("one H, W_K and stale K per layer")
    n = np.asarray(H_ctx_layers[0]).shape[0]
    acc = np.zeros(n, dtype=F64)
    for X, Wk, Ks in zip(H_ctx_layers, Wk_layers, K_stale_layers):
        X = np.asarray(X, F64)
        Kn = (X @ np.asarray(Wk, F64).T).reshape(n, n_kv_heads, head_dim)
        Kn = rope_rotate(Kn, np.arange(n)[:, None], base)
        Ko = np.asarray(Ks, F64).reshape(n, n_kv_heads, head_dim)
        dot = np.sum(Kn * Ko, axis=-1)
        den = np.sqrt(np.sum(Kn * Kn, axis=-1)) * np.sqrt(np.sum(Ko * Ko, axis=-1))
        acc += np.sum(dot / np.maximum(den, 1e-30), axis=1)
    return 1.0 - acc / (n_layers * n_kv_heads)


# --------------------------------------------------------------------------
# Selection (QCFuse Eq. 6 and Eq. 11; KVBoost Alg. 2 step 3)
# --------------------------------------------------------------------------

def k_from_ratio(ratio: float, n_ctx: int) -> int:
    """Number of recomputed context tokens: ``floor(rho * N + 1e-9)`` in
    ``[0, N]``."""
    k = int(math.floor(float(ratio) * int(n_ctx) + 1e-9))
    return max(0, min(int(n_ctx), k))


def select_topk(score: np.ndarray, k: int) -> np.ndarray:
    """Indices of the ``k`` largest scores, ties to the lower index, returned
    in ascending index order.  Comparisons are made on the given values
    (an fp32 array is compared as fp32: widening is exact)."""
    s = np.asarray(score)
    if np.isnan(s).any():
        raise ValueError("NaN deviation score")
    s = s.astype(F64) + 0.0          # -0 -> +0
    n = s.shape[0]
    if not 0 <= k <= n:
        raise ValueError("k out of range")
    order = np.lexsort((np.arange(n), -s))   # primary: larger score; then lower index
    return np.sort(order[:k]).astype(np.int64)


def static_select(chunk_starts: Sequence[int], chunk_lens: Sequence[int], n_ctx: int,
                  kind: str, n: int) -> np.ndarray:
    """Positions of one request chosen from its chunk layout alone, ascending.

    kind "chunk_head" (QCFuse, related work on query-agnostic selection: EPIC
    recomputes a fixed number of boundary tokens of every stitched chunk,
    the first tokens of a chunk acting as attention sinks): the first n
    positions of every chunk.  kind "seam_tail" (KVBoost section 4.6.1,
    SelectiveRecompute): for every seam p -- the start of a chunk that follows
    another chunk -- the positions max(0, p - n) .. p - 1.  Chunks are given
    in position order; the selection is the union, read off a mask over the
    request's positions."""
    mask = np.zeros(n_ctx, dtype=bool)
    for c, (s, ln) in enumerate(zip(chunk_starts, chunk_lens)):
        if kind == "chunk_head":
            mask[s:s + min(n, ln)] = True
        elif kind == "seam_tail":
            if c > 0:
                mask[max(0, s - n):s] = True
        else:
            raise ValueError(kind)
    return np.nonzero(mask)[0].astype(np.int64)


# --------------------------------------------------------------------------
# Query-aware attention mass (QCFuse section 3.2.1, Eqs. 9-10; Eq. 20)
# --------------------------------------------------------------------------

def attention_mass_scores(H_query: np.ndarray, Wq, K_ctx: np.ndarray,
                          n_q_heads: int, n_kv_heads: int, head_dim: int, base: float,
                          store=None) -> np.ndarray:
    """Importance ``I(t)`` of every context token of one request at one layer:
    the attention the user query pays to it (QCFuse Eq. 10 for one layer;
    Eq. 20 adds this quantity over the critical layers L*).

    ``H_query`` ``[Qn, D]`` holds the query tokens' inputs to the layer; query
    token u sits at request position ``N + u`` with ``N = K_ctx.shape[0]``,
    so its state is ``q_{u,h} = R^{N+u} W_Q x_u`` (head h of the projection,
    the same projection the recomputation uses).  ``K_ctx`` ``[N, Hkv, d]``
    holds the stitched PIC keys of the N context tokens (QCFuse Eq. 4).
    For every (u, h) the weights over the context keys are
    ``softmax_t(q_{u,h} . K[t, h // g] / sqrt(d))``, ``g = Hq / Hkv``, and
    ``I(t)`` is the sum of the weight of t over all (u, h): each (u, h)
    contributes a total of exactly 1.  ``store`` (the layer's storage
    rounding) is applied to q where it is materialised.
    """
    X = np.asarray(H_query, F64)
    K = np.asarray(K_ctx, F64)
    n_query = X.shape[0]
    n = K.shape[0]
    out = np.zeros(n, dtype=F64)
    if n == 0 or n_query == 0:
        return out
    g = n_q_heads // n_kv_heads
    q = (X @ np.asarray(Wq, F64).T).reshape(n_query, n_q_heads, head_dim)
    q = rope_rotate(q, (n + np.arange(n_query))[:, None], base)
    if store is not None:
        q = store(q)
    scale = 1.0 / math.sqrt(head_dim)
    for h in range(n_q_heads):
        logits = np.matmul(q[:, h, :], K[:, h // g, :].T) * scale       # [Qn, N]
        m = logits.max(axis=1, keepdims=True)
        w = np.exp(logits - m)
        w /= w.sum(axis=1, keepdims=True)
        out += w.sum(axis=0)
    return out


def selected_rows(idx: np.ndarray, n_ctx: int, n_tok: int) -> np.ndarray:
    """``S``: the selected context rows followed by every query row, ascending."""
    return np.concatenate([np.asarray(idx, np.int64), np.arange(n_ctx, n_tok, dtype=np.int64)])


# --------------------------------------------------------------------------
# Recomputation of the selected rows (QCFuse Eqs. 6-7; KVBoost Eqs. 1-3)
# --------------------------------------------------------------------------

def project_rows(H_rows: np.ndarray, Wq, Wk, Wv, pos: np.ndarray,
                 n_q_heads: int, n_kv_heads: int, head_dim: int, base: float):
    """Fresh ``q, k, v`` of some rows at their request positions ``pos``:
    ``q = R^p W_Q x``, ``k = R^p W_K x``, ``v = W_V x``."""
    X = np.asarray(H_rows, F64)
    r = X.shape[0]
    q = (X @ np.asarray(Wq, F64).T).reshape(r, n_q_heads, head_dim)
    k = (X @ np.asarray(Wk, F64).T).reshape(r, n_kv_heads, head_dim)
    v = (X @ np.asarray(Wv, F64).T).reshape(r, n_kv_heads, head_dim)
    p = np.asarray(pos)[:, None]
    return rope_rotate(q, p, base), rope_rotate(k, p, base), v


def recompute_selected(H: np.ndarray, Wq, Wk, Wv, idx: np.ndarray, n_ctx: int,
                       K_fused: np.ndarray, V_fused: np.ndarray,
                       n_q_heads: int, n_kv_heads: int, head_dim: int, base: float,
                       out_rows: Optional[np.ndarray] = None, store=None):
    """Selective recomputation of one request at one layer.

    ``H`` is ``[T, D]`` (context then query), ``K_fused``/``V_fused`` are
    ``[T, Hkv, d]`` whose context rows hold the stitched cache (query rows
    are overwritten).  Rows ``S = idx U {N..T-1}`` get fresh ``q, k, v`` at
    position ``p = s``; their k and v replace the fused entries (Eq. 7).
    Then each row of S attends causally over ``j <= p`` of the fused cache
    (KVBoost Eq. 2, scale ``1/sqrt(d)``; query head h reads KV head
    ``h // (Hq/Hkv)``), two-pass softmax with the maximum subtracted.

    ``out_rows`` (indices into S) limits which attention rows are evaluated.
    ``store`` (the storage rounding of the layer, if any) is applied to the
    fresh q, k, v as they are materialised.
    Returns ``(K_fused', V_fused', O [len(out_rows), Hq, d], S)``.
    """
    T = H.shape[0]
    d = head_dim
    S = selected_rows(idx, n_ctx, T)
    q, k, v = project_rows(np.asarray(H, F64)[S], Wq, Wk, Wv, S,
                           n_q_heads, n_kv_heads, d, base)
    if store is not None:
        q, k, v = store(q), store(k), store(v)
    Kf = np.array(K_fused, dtype=F64, copy=True)
    Vf = np.array(V_fused, dtype=F64, copy=True)
    Kf[S] = k
    Vf[S] = v
    rows = np.arange(S.shape[0]) if out_rows is None else np.asarray(out_rows)
    O = causal_attention(q, Kf, Vf, S, rows, n_q_heads, n_kv_heads, d)
    return Kf, Vf, O, S


def causal_attention(q: np.ndarray, K_fused: np.ndarray, V_fused: np.ndarray, S: np.ndarray,
                     rows: np.ndarray, n_q_heads: int, n_kv_heads: int, head_dim: int):
    """Causal GQA attention rows over a fused cache (KVBoost Eq. 2).

    For each ``r`` in ``rows`` (indices into S), the row at position
    ``p = S[r]`` with query ``q[r]`` (``[Hq, d]``) attends over ``j <= p`` of
    ``K_fused``/``V_fused`` (``[T, Hkv, d]``) with scale ``1/sqrt(d)``; query
    head h reads KV head ``h // (Hq/Hkv)``; two-pass softmax with the maximum
    subtracted.  Returns ``O [len(rows), Hq, d]``.
    """
    d = head_dim
    g = n_q_heads // n_kv_heads
    Kt = np.ascontiguousarray(np.asarray(K_fused, F64).transpose(1, 0, 2))     # [Hkv, T, d]
    Vt = np.ascontiguousarray(np.asarray(V_fused, F64).transpose(1, 0, 2))
    rows = np.asarray(rows)
    O = np.zeros((rows.shape[0], n_q_heads, d), dtype=F64)
    scale = 1.0 / math.sqrt(d)
    for o, r in enumerate(rows):
        p = int(S[r])
        qr = q[r].reshape(n_kv_heads, g, d)                 # [Hkv, g, d]
        logits = np.matmul(qr, Kt[:, :p + 1, :].transpose(0, 2, 1)) * scale   # [Hkv, g, p+1]
        m = logits.max(axis=-1, keepdims=True)
        w = np.exp(logits - m)
        w /= w.sum(axis=-1, keepdims=True)
        O[o] = np.matmul(w, Vt[:, :p + 1, :]).reshape(n_q_heads, d)
    return O


def layer_step(H: np.ndarray, Wq, Wk, Wv, K_chunks, V_chunks, ratio: float,
               n_q_heads: int, n_kv_heads: int, head_dim: int, base: float,
               score: bool = True, idx: Optional[np.ndarray] = None,
               out_rows: Optional[np.ndarray] = None, store=None):
    """One layer-step for one request: stitch -> deviation -> top-k ->
    recompute, in the order of KVBoost Alg. 2 (probe, deviation, select,
    patch) on the cache stitched by QCFuse Eq. 4.

    With ``score=False`` the given ``idx`` is reused (a selection made at
    another layer).  Returns a dict with the fused cache, scores, idx, S, O.
    """
    T = H.shape[0]
    Kc, Vc = stitch_rerotate(K_chunks, V_chunks, base, store)
    n_ctx = Kc.shape[0]
    Kf = np.zeros((T, n_kv_heads, head_dim), F64)
    Vf = np.zeros((T, n_kv_heads, head_dim), F64)
    Kf[:n_ctx] = Kc
    Vf[:n_ctx] = Vc
    sc = None
    if score:
        sc = deviation_scores(np.asarray(H, F64)[:n_ctx], Wv, Vc, n_kv_heads, head_dim)
        idx = select_topk(sc, k_from_ratio(ratio, n_ctx))
    Kf2, Vf2, O, S = recompute_selected(H, Wq, Wk, Wv, idx, n_ctx, Kf, Vf,
                                        n_q_heads, n_kv_heads, head_dim, base, out_rows,
                                        store)
    return {"K_stitched": Kc, "V_stitched": Vc, "score": sc, "idx": idx, "S": S,
            "K_fused": Kf2, "V_fused": Vf2, "O": O}
