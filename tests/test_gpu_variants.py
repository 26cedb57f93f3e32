"""Deviation variants on the GPU: KVBoost's Alg. 2 step 2 as printed, the
cosine of the keys averaged over key heads and layers
(fuse_score_key_deviation), against the oracle on the same stitched cache
(the oracle's, written into the device cache).

Tolerance: 1e-3 absolute, as for the value deviation.  A bf16 layer rounds
the fresh keys to bf16, which the oracle does not.  An emulation of that
(keys accumulated in fp32, rotated and rounded) on these cases moves a score
by at most 1.5e-4.  The top-k of the scores is bit-exact against the
oracle's selection from the same fp32 array."""

import numpy as np
import pytest
import torch

from oracle import fusion as orc
from rag_kv_cache_rerotate_gb300 import fusekv as fk
from rag_kv_cache_rerotate_gb300 import synth

from harness import buffers, f64, make_case, request_slices
import test_gpu_parity as parity

pytestmark = pytest.mark.gpu

# fp32 and bf16 d = 64 (CUDA-core projection), three paged requests and the
# Qwen3-8B-shaped layer (tensor-core projection)
CASES = ["tiny_fp32", "ragged_paged_bf16_d64", "paged3", "qwen3_8b_layer"]


@pytest.mark.parametrize("name", CASES)
def test_key_deviation_one_layer_matches_oracle(name):
    case = parity.case_of(name)
    cfg = case.cfg
    b = buffers(case)
    parity._load_oracle_stitched(case, b)
    fk.score_key_deviation(b.desc, b.reqs, b.H, b.Wk, b.Kf, b.score, b.ws)
    fk.check_errors(b.ws)
    score = b.score.cpu().numpy()
    H, Wk = f64(b.H), f64(b.Wk)
    for (r, row0, n, T, cis), (K, V) in zip(request_slices(case),
                                            parity._oracle_stitched(case, parity._store(cfg))):
        if n == 0:
            continue
        q = b.reqs[r]
        want = orc.key_deviation_scores([H[row0:row0 + n]], [Wk], [K], cfg.n_kv_heads,
                                        cfg.head_dim, cfg.rope_base)
        got = score[q.score0:q.score0 + n].astype(np.float64)
        assert np.max(np.abs(got - want)) <= 1e-3, r
    idx = torch.full((max(1, b.reqs.totals().n_sel),), -1, dtype=torch.int32, device="cuda")
    fk.select_topk(b.reqs, b.score, idx, b.ws)
    fk.check_errors(b.ws)
    sel = idx.cpu().numpy()
    for (r, row0, n, T, cis) in request_slices(case):
        q = b.reqs[r]
        want = orc.select_topk(score[q.score0:q.score0 + n], q.k)
        assert sel[q.sel0:q.sel0 + q.k].tolist() == want.tolist()


def test_key_deviation_averages_over_layers():
    # two layers with their own draws, weights and caches: weight 1/2 each,
    # the second call accumulating, gives the printed average over layers
    cfg = synth.scaled(synth.CONFIGS["qwen3_8b_layer"], chunks_per_request=3, chunk_len=200,
                       query_len=24, seed=17)
    layouts = synth.draw_layouts(cfg)
    cases = [make_case(cfg, layouts, layer=l) for l in range(2)]
    bufs = [buffers(c) for c in cases]
    for c, b in zip(cases, bufs):
        parity._load_oracle_stitched(c, b)
    out = bufs[0].score
    for l, b in enumerate(bufs):
        fk.score_key_deviation(b.desc, b.reqs, b.H, b.Wk, b.Kf, out, b.ws, weight=0.5,
                               accumulate=l > 0)
        fk.check_errors(b.ws)
    got = out.cpu().numpy().astype(np.float64)
    (r, row0, n, T, cis), = request_slices(cases[0])
    Ks = [parity._oracle_stitched(c, parity._store(cfg))[0][0] for c in cases]
    want = orc.key_deviation_scores([f64(b.H)[:n] for b in bufs], [f64(b.Wk) for b in bufs], Ks,
                                    cfg.n_kv_heads, cfg.head_dim, cfg.rope_base)
    assert np.max(np.abs(got[:n] - want)) <= 1e-3
