"""Query-aware attention mass on the GPU (QCFuse section 3.2.1, Eqs. 9-10;
section 3.4.2, Eq. 20), through the C ABI, against the oracle on the same
stitched cache (the oracle's, written into the device cache).

Tolerances: scores within 1e-4 relative in fp32 layers.  In bf16 layers q is
materialised in bf16 on both sides; the two sides round the same fp32 or
fp64 value, so a rounding can land one bf16 step apart where the fp32
accumulation differs from fp64.  An fp32 emulation of that on these cases
moves a score by at most 2.1e-5 relative, and the bound taken is 2e-3.  A
floor of 1e-6 of the mean score covers the fp32 underflow of negligible
weights.  The top-k of the scores is bit-exact against the oracle's
selection from the same fp32 array."""

import numpy as np
import pytest
import torch

from oracle import fusion as orc
from rag_kv_cache_rerotate_gb300 import fusekv as fk

from harness import buffers, f64, request_slices
import test_gpu_parity as parity

pytestmark = pytest.mark.gpu

# fp32 (SIMT projection), bf16 d = 64 ragged/paged with empty queries (SIMT
# projection in bf16); the tensor-core scorer: three requests of the batched
# paged workload (172 query rows: the layer GEMM's pair tiles split over K),
# the Qwen3-8B-shaped layer (64 rows), four 1024-token chunks of the
# Llama-3-70B shape (eight query heads per KV head: four 128-vector tiles per
# KV head) and 70 query rows (a partial second group of 64 rows) -- up to 128
# rows the projection is formed transposed, rows on the MMA's short side
CASES = ["tiny_fp32", "ragged_fp32", "ragged_paged_bf16_d64", "paged3", "qwen3_8b_layer",
         "int8_4x1024", "qwen3_q70"]


def _tol(cfg):
    return 2e-3 if cfg.dtype == "bf16" else 1e-4


def _run(case, accumulate=False, score=None):
    b = buffers(case)
    parity._load_oracle_stitched(case, b)
    out = b.score if score is None else score
    fk.score_attention_mass(b.desc, b.reqs, b.H, b.Wq, b.Kf, out, b.ws, accumulate=accumulate)
    fk.check_errors(b.ws)
    return b, out


def _oracle(case, b):
    cfg = case.cfg
    H, Wq = f64(b.H), f64(b.Wq)
    out = []
    for (r, row0, n, T, cis), (K, V) in zip(request_slices(case),
                                            parity._oracle_stitched(case, parity._store(cfg))):
        out.append(orc.attention_mass_scores(H[row0 + n:row0 + T], Wq, K, cfg.n_q_heads,
                                             cfg.n_kv_heads, cfg.head_dim, cfg.rope_base,
                                             parity._store(cfg)))
    return out


@pytest.mark.parametrize("name", CASES)
def test_attention_mass_matches_oracle(name):
    case = parity.case_of(name)
    cfg = case.cfg
    b, score = _run(case)
    got_all = score.cpu().numpy()
    tol = _tol(cfg)
    for (r, row0, n, T, cis), want in zip(request_slices(case), _oracle(case, b)):
        q = b.reqs[r]
        got = got_all[q.score0:q.score0 + n].astype(np.float64)
        if n == 0:
            continue
        total = (T - n) * cfg.n_q_heads
        if total == 0:
            assert np.array_equal(got, np.zeros(n)), r          # no query: nothing spread
            continue
        floor = 1e-6 * total / n
        assert np.all(np.abs(got - want) <= tol * want + floor), (
            r, float(np.max(np.abs(got - want) / (want + floor))))
        # every (query token, head) spreads a total weight of 1
        assert abs(got.sum() - total) <= 1e-4 * total
    # the selection from these scores
    idx = torch.full((max(1, b.reqs.totals().n_sel),), -1, dtype=torch.int32, device="cuda")
    fk.select_topk(b.reqs, score, idx, b.ws)
    fk.check_errors(b.ws)
    sel = idx.cpu().numpy()
    for (r, row0, n, T, cis) in request_slices(case):
        q = b.reqs[r]
        want = orc.select_topk(got_all[q.score0:q.score0 + n], q.k)
        assert sel[q.sel0:q.sel0 + q.k].tolist() == want.tolist()


def test_attention_mass_accumulates_over_layers():
    # Eq. 20: the critical layers' terms are added into one score array
    case = parity.case_of("paged3")
    b, once = _run(case)
    first = once.clone()
    fk.score_attention_mass(b.desc, b.reqs, b.H, b.Wq, b.Kf, once, b.ws, accumulate=True)
    fk.check_errors(b.ws)
    assert torch.equal(once, 2 * first)                          # the same term, added exactly


def test_attention_mass_edges():
    # a request without query tokens scores 0; one without context is skipped;
    # entries of the score array outside every request are left untouched
    cfg = parity.SMALL["tiny_fp32"]
    desc = fk.layer_desc(cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rope_base,
                         fk.FUSE_F32)
    n_ctx, n_query = [37, 0, 5, 64], [3, 4, 0, 1]
    reqs = fk.plan_requests(n_ctx, n_query, 0.25)
    t = reqs.totals()
    g = torch.Generator().manual_seed(4)
    H = torch.randn(t.n_tok, cfg.hidden, generator=g).cuda()
    Wq = (torch.randn(cfg.n_q_heads * cfg.head_dim, cfg.hidden, generator=g) * 0.05).cuda()
    Kf = torch.randn(t.n_tok, cfg.n_kv_heads, cfg.head_dim, generator=g).cuda()
    score = torch.full((t.n_ctx + 3,), 7.0, device="cuda")
    ws = fk.alloc_workspace(desc, reqs)
    fk.score_attention_mass(desc, reqs, H, Wq, Kf, score, ws)
    fk.check_errors(ws)
    got = score.cpu().numpy().astype(np.float64)
    Hn, Wn, Kn = f64(H), f64(Wq), f64(Kf)
    row = 0
    for i, (n, qn) in enumerate(zip(n_ctx, n_query)):
        q = reqs[i]
        want = orc.attention_mass_scores(Hn[row + n:row + n + qn], Wn, Kn[row:row + n],
                                         cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                                         cfg.rope_base)
        g_r = got[q.score0:q.score0 + n]
        if qn == 0:
            assert np.array_equal(g_r, np.zeros(n))
        else:
            assert np.all(np.abs(g_r - want) <= 1e-4 * want + 1e-6), i
        row += n + qn
    assert np.array_equal(got[t.n_ctx:], [7.0, 7.0, 7.0])


def test_attention_mass_tensor_core_edges():
    # the tensor-core path (bf16, head_dim 128): a request with no query
    # scores 0, one with no context is skipped, ragged vector and key tiles
    # (160 vectors: two 128-vector tiles; 300 keys: a partial key tile), and
    # entries outside every request are left untouched
    desc = fk.layer_desc(512, 8, 2, 128, 5e5, fk.FUSE_BF16)
    n_ctx, n_query = [300, 0, 5, 129, 77], [40, 4, 0, 1, 32]
    reqs = fk.plan_requests(n_ctx, n_query, 0.25)
    t = reqs.totals()
    g = torch.Generator().manual_seed(5)
    H = torch.randn(t.n_tok, 512, generator=g).to(torch.bfloat16).cuda()
    Wq = (torch.randn(8 * 128, 512, generator=g) / 22.6).to(torch.bfloat16).cuda()
    Kf = torch.randn(t.n_tok, 2, 128, generator=g).to(torch.bfloat16).cuda()
    score = torch.full((t.n_ctx + 3,), 7.0, device="cuda")
    ws = fk.alloc_workspace(desc, reqs)
    fk.score_attention_mass(desc, reqs, H, Wq, Kf, score, ws)
    fk.check_errors(ws)
    got = score.cpu().numpy().astype(np.float64)
    Hn, Wn, Kn = f64(H), f64(Wq), f64(Kf)
    row = 0
    for i, (n, qn) in enumerate(zip(n_ctx, n_query)):
        q = reqs[i]
        g_r = got[q.score0:q.score0 + n]
        if qn == 0:
            assert np.array_equal(g_r, np.zeros(n))
        elif n:
            want = orc.attention_mass_scores(Hn[row + n:row + n + qn], Wn, Kn[row:row + n], 8, 2,
                                             128, 5e5, orc.round_bf16)
            floor = 1e-6 * qn * 8 / n
            assert np.all(np.abs(g_r - want) <= 2e-3 * want + floor), i
            assert abs(g_r.sum() - qn * 8) <= 1e-4 * qn * 8
        row += n + qn
    assert np.array_equal(got[t.n_ctx:], [7.0, 7.0, 7.0])
