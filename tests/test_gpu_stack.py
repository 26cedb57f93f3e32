"""GPU parity of fuse_stack_step: several layers sharing one selection made
at a scoring layer (the layer loop of the 36-layer stack workload), each
layer with its own draws, weights and chunk caches."""

import numpy as np
import pytest

from oracle import fusion as orc
from rag_kv_cache_rerotate_gb300 import fusekv as fk
from rag_kv_cache_rerotate_gb300 import synth

import rounding
from harness import buffers, f64, make_case, max_rel, max_row_rel, request_slices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rag_kv_cache_rerotate_gb300 import _build
    _build.build()
    fk.load()


def test_stack_shares_the_scoring_layers_selection():
    cfg = synth.scaled(synth.CONFIGS["qwen3_8b_stack36"], chunks_per_request=3, chunk_len=256,
                       query_len=32, n_layers=3, score_layer=1)
    layouts = synth.draw_layouts(cfg)
    cases = [make_case(cfg, layouts, layer=l) for l in range(cfg.n_layers)]
    bufs = [buffers(c) for c in cases]
    b0 = bufs[cfg.score_layer]
    fk.stack_step(b0.desc, b0.reqs, bufs, cfg.score_layer, b0.idx, b0.score, b0.ws)
    fk.check_errors(b0.ws)
    q = b0.reqs[0]
    n, T = q.n_ctx, q.n_ctx + q.n_query
    idx = b0.idx.cpu().numpy()[:q.k].astype(np.int64)
    score = b0.score.cpu().numpy()[:n]
    store = orc.round_bf16
    # the selection: a bit-exact top-k of the scoring layer's GPU scores, and a
    # valid top-k of the oracle's scores of that layer
    assert orc.select_topk(score, q.k).tolist() == idx.tolist()
    cs = cases[cfg.score_layer]
    Kc, Vc = orc.stitch_rerotate(cs.K_cached, cs.V_cached, cfg.rope_base, store)
    s_orc = orc.deviation_scores(f64(cs.draws.H)[:n], f64(cs.draws.Wv), Vc, cfg.n_kv_heads,
                                 cfg.head_dim)
    assert np.max(np.abs(score - s_orc)) <= 1e-3
    rest = np.setdiff1d(np.arange(n), idx)
    assert s_orc[idx].min() >= s_orc[rest].max() - 2e-3
    # every layer: recomputed with that selection over its own stitched cache
    for l, (case, b) in enumerate(zip(cases, bufs)):
        H = f64(b.H)
        Kc, Vc = orc.stitch_rerotate(case.K_cached, case.V_cached, cfg.rope_base, store)
        Kf0 = np.zeros((T, cfg.n_kv_heads, cfg.head_dim))
        Vf0 = np.zeros_like(Kf0)
        Kf0[:n], Vf0[:n] = Kc, Vc
        S = orc.selected_rows(idx, n, T)
        rows = np.arange(len(S))
        Ko, Vo, Oo, _ = orc.recompute_selected(H, f64(b.Wq), f64(b.Wk), f64(b.Wv), idx, n, Kf0, Vf0,
                                               cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                                               cfg.rope_base, out_rows=rows, store=store)
        Kf, Vf, O = f64(b.Kf), f64(b.Vf), f64(b.O)
        assert max_rel(Kf[S], Ko[S]) <= 2e-2, l
        assert max_rel(Vf[S], Vo[S]) <= 2e-2, l
        keep = np.setdiff1d(np.arange(n), S)
        assert max_row_rel(Kf[keep], Ko[keep]) <= 2.0 ** -7, l
        st = rounding.stitched_bounds(case.K_cached, case.V_cached, cfg.rope_base, False)
        rounding.check_rows(f"stack_step[layer {l}]", O[q.out0 + rows], H, f64(b.Wq), f64(b.Wk),
                            f64(b.Wv), S, Ko, Vo, Oo, rows, cfg.n_q_heads, cfg.n_kv_heads,
                            cfg.head_dim, cfg.rope_base, 2e-2, stitched=st)
