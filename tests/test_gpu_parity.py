"""GPU parity: every entry point of the C ABI against the oracle on the same
seeded inputs.

Tolerances (stated for the method): selected indices bit-exact given the
same score array; scores within 1e-3 absolute; re-rotated keys within 1e-5
relative (per row, normwise) in fp32 mode; attention outputs and refreshed
K/V within 2e-2 max relative (normwise) in bf16.  Stitched bf16 keys are
rounded to bf16 on output, so they get 2^-8 per row."""

import numpy as np
import pytest
import torch

from oracle import fusion as orc
from rag_kv_cache_rerotate_gb300 import fusekv as fk
from rag_kv_cache_rerotate_gb300 import synth, workload

import rounding
from harness import buffers, f64, make_case, max_rel, max_row_rel, request_slices, stitch_tol

pytestmark = pytest.mark.gpu

C = synth.CONFIGS
SMALL = {
    "tiny_fp32": C["tiny_fp32"],
    "qwen3_8b_layer": C["qwen3_8b_layer"],
    # three requests of the batched paged workload (same per-request recipe)
    "paged3": synth.scaled(C["llama3_8b_paged_batch16"], n_requests=3),
    # four 1024-token chunks of the int8 long-context workload
    "int8_4x1024": synth.scaled(C["llama3_70b_int8_long"], chunks_per_request=4, query_len=64),
    # 8192 context tokens, 1 % selected: row tiles span thousands of positions,
    # so the attention plan splits their key ranges into up to five pieces and
    # some rows lie wholly before the first key of a piece
    "sparse_long_bf16": synth.scaled(C["qwen3_8b_layer"], chunks_per_request=16, ratio=0.01,
                                     seed=21),
    # hidden 9216: the row gather copies a row in more than one round of
    # 16-byte loads per thread
    "wide_hidden_bf16": synth.scaled(C["qwen3_8b_layer"], hidden=9216, chunks_per_request=3,
                                     chunk_len=96, query_len=8, ratio=0.2, seed=23),
    # ragged: odd chunk lengths, 1-token chunks, a short query, fp32
    "ragged_fp32": synth.scaled(C["tiny_fp32"], chunks_per_request=None, chunk_len=None,
                                query_len=None, chunk_count_range=(1, 6),
                                chunk_len_range=(1, 45), query_len_range=(1, 9), n_requests=4,
                                ratio=0.35, seed=11),
    # ragged bf16, d = 64, paged with a partial tail block
    "ragged_paged_bf16_d64": synth.scaled(C["tiny_fp32"], dtype="bf16", kv_storage="bf16",
                                          kv_layout="paged", chunks_per_request=None,
                                          chunk_len=None, query_len=None,
                                          chunk_count_range=(2, 5), chunk_len_range=(3, 70),
                                          query_len_range=(0, 7), n_requests=3, ratio=0.5,
                                          seed=12),
}

# Cases whose storage type only the stitch sees (it dequantises into the fused
# cache; everything after reads that cache): the stitch and score/top-k tests
# take them, the recompute tests (which share the oracle's stitched cache)
# gain nothing from them.
STORAGE = {
    # four 1024-token chunks of the int8 long-context workload with KIVI's
    # 4-bit codes (two per byte)
    "int4_4x1024": synth.scaled(C["llama3_70b_int8_long"], chunks_per_request=4, query_len=64,
                                kv_storage="u4", seed=8),
    # two requests of the batched paged workload with 4-bit codes in the
    # block pool (d / 2 bytes per token and head, partial tail blocks)
    "int4_paged2": synth.scaled(C["llama3_8b_paged_batch16"], n_requests=2, kv_storage="u4"),
    # int8 codes in the block pool (16-token blocks, partial tail blocks)
    "int8_paged2": synth.scaled(C["llama3_8b_paged_batch16"], n_requests=2, kv_storage="u8",
                                seed=9),
    # int8, d = 64, ragged chunks of 1..70 tokens: partial row tiles of the
    # int8 stitch and 1-token chunks
    "int8_ragged_d64": synth.scaled(C["llama3_70b_int8_long"], hidden=1024, n_q_heads=16,
                                    head_dim=64, w_std=1.0 / 32.0, chunks_per_request=None,
                                    chunk_len=None, query_len=None, chunk_count_range=(2, 6),
                                    chunk_len_range=(1, 70), query_len_range=(1, 9),
                                    n_requests=3, ratio=0.3, seed=13),
    # 70 query rows: the scorer's short-side query projection with a partial
    # second group of 64 rows
    "qwen3_q70": synth.scaled(C["qwen3_8b_layer"], chunks_per_request=2, query_len=70, seed=16),
    # int8 with 4 KV heads: eight rows per stitch tile instead of four
    "int8_hkv4": synth.scaled(C["llama3_70b_int8_long"], hidden=1024, n_q_heads=8, n_kv_heads=4,
                              w_std=1.0 / 32.0, chunks_per_request=3, chunk_len=100, query_len=8,
                              seed=14),
}

# Requests of 16 384 tokens and more: the attention takes its tiles in pairs
# on clusters of two CTAs.  Two such requests with few selected rows (the
# oracle's attention stays cheap) and a GQA group of 2 (64-row tiles): pairs
# inside a request share their K/V fetches, pairs across the two requests do
# not, and an odd tile count leaves one tile without a partner.
LONG = {
    "long_pairs2": synth.scaled(C["llama3_70b_int8_long"], hidden=1024, n_q_heads=16,
                                w_std=1.0 / 32.0, n_requests=2, chunks_per_request=None,
                                chunk_count_range=(16, 17), chunk_len=1024, query_len=16,
                                ratio=0.0029, seed=15),
}

_CASES = {}


def case_of(name):
    if name not in _CASES:
        cfg = SMALL.get(name) or STORAGE.get(name) or LONG[name]
        _CASES[name] = make_case(cfg)
    return _CASES[name]


def _rows_for_attention(S):
    """Attention rows the oracle evaluates: every recomputed row."""
    return np.arange(len(S))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rag_kv_cache_rerotate_gb300 import _build
    _build.build()
    fk.load()


def _store(cfg):
    """Storage rounding of the layer's fused cache and Q (bf16 layers)."""
    return orc.round_bf16 if cfg.dtype == "bf16" else None


def _oracle_stitched(case, store=None):
    """Per request: oracle stitched K, V of its context rows."""
    out = []
    for (r, row0, n, T, cis) in request_slices(case):
        K, V = orc.stitch_rerotate([case.K_cached[i] for i in cis], [case.V_cached[i] for i in cis],
                                   case.cfg.rope_base, store)
        out.append((K, V))
    return out


@pytest.mark.parametrize("name", list(SMALL) + list(STORAGE))
def test_stitch_rerotate(name):
    case = case_of(name)
    b = buffers(case)
    fk.stitch_rerotate(b.desc, b.chunks, b.Kf, b.Vf, b.ws)
    fk.check_errors(b.ws)
    Kf, Vf = f64(b.Kf), f64(b.Vf)
    tol = stitch_tol(case.cfg)
    starts = np.cumsum([0] + [len(k) for k in case.K_cached])
    for (r, row0, n, T, cis), (K, V) in zip(request_slices(case), _oracle_stitched(case)):
        if n == 0:
            continue
        assert max_row_rel(Kf[row0:row0 + n], K) <= tol
        if case.cfg.kv_storage in ("u8", "u4"):
            assert max_row_rel(Vf[row0:row0 + n], V) <= tol
        else:
            assert np.array_equal(Vf[row0:row0 + n], V)
        if case.cfg.kv_storage == case.cfg.dtype:
            # the first chunk (offset 0) is copied bit for bit
            n0 = case.layouts[r].chunk_lens[0]
            c0 = int(starts[cis[0]])
            assert torch.equal(b.Kf[row0:row0 + n0].cpu(), case.caches.K[c0:c0 + n0])


def test_stitch_large_positions_fp32():
    cfg = synth.scaled(C["tiny_fp32"], rope_base=5e5, head_dim=128, n_kv_heads=2, n_q_heads=4)
    rng = np.random.default_rng(5)
    poss = [0, 1, 999, 16383, 31999, 33023, (1 << 20) + 7, (1 << 24) - 70]
    lens = [16, 3, 64, 17, 32, 1, 40, 64]
    Ks = [rng.standard_normal((n, 2, 128)) for n in lens]
    Vs = [rng.standard_normal((n, 2, 128)) for n in lens]
    caches = workload.ChunkCaches(torch.from_numpy(np.concatenate(Ks)).float(),
                                  torch.from_numpy(np.concatenate(Vs)).float())
    rows = []
    dst = 0
    for p, n in zip(poss, lens):
        rows.append((0, len(rows), dst, p, n))
        dst += n
    table, store = workload._contiguous_storage(cfg, rows, caches, "cuda")
    Kf = torch.zeros(dst, 2, 128, device="cuda")
    Vf = torch.zeros_like(Kf)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    fk.stitch_rerotate(workload.desc_of(cfg), table, Kf, Vf, ws)
    fk.check_errors(ws)
    Kc = f64(caches.K)
    got = f64(Kf)
    for (_, _, d0, p, n) in rows:
        want = orc.rope_rotate(Kc[d0:d0 + n], p, 5e5)
        assert max_row_rel(got[d0:d0 + n], want) <= 1e-5, p
    assert np.array_equal(f64(Vf), f64(caches.V))


@pytest.mark.parametrize("name", list(SMALL) + list(STORAGE))
def test_score_and_topk(name):
    case = case_of(name)
    b = buffers(case)
    fk.stitch_rerotate(b.desc, b.chunks, b.Kf, b.Vf, b.ws)
    fk.score_deviation(b.desc, b.reqs, b.H, b.Wv, b.Vf, b.score, b.ws)
    fk.select_topk(b.reqs, b.score, b.idx, b.ws)
    fk.check_errors(b.ws)
    H = f64(b.H)
    Wv = f64(b.Wv)
    score = b.score.cpu().numpy()
    idx = b.idx.cpu().numpy()
    cfg = case.cfg
    for (r, row0, n, T, cis), (K, V) in zip(request_slices(case), _oracle_stitched(case, _store(cfg))):
        q = b.reqs[r]
        s_gpu = score[q.score0:q.score0 + n]
        if n > 0:
            s_orc = orc.deviation_scores(H[row0:row0 + n], Wv, V, cfg.n_kv_heads, cfg.head_dim)
            assert np.max(np.abs(s_gpu - s_orc)) <= 1e-3
        want = orc.select_topk(s_gpu, q.k)           # same fp32 array -> bit-exact
        assert idx[q.sel0:q.sel0 + q.k].tolist() == want.tolist()


def test_topk_ties_and_edges():
    rng = np.random.default_rng(9)
    # the first group keeps keys in shared memory, the second (max N > 40960) in the workspace
    for sizes in ([1, 2, 7, 64, 1000, 4097, 33024], [3, 50000, 129]):
        vals = []
        for n in sizes:
            v = (rng.integers(-3, 4, size=n) * 0.125).astype(np.float32)   # many ties
            v[rng.integers(0, n)] = -0.0
            vals.append(v)
        for ratio in (0.0, 0.13, 0.5, 1.0):
            reqs = fk.plan_requests(sizes, [0] * len(sizes), ratio)
            tot = reqs.totals()
            score = torch.from_numpy(np.concatenate(vals)).cuda()
            idx = torch.full((max(tot.n_sel, 1),), -1, dtype=torch.int32, device="cuda")
            ws = torch.zeros(256 + 4 * tot.n_ctx + 256, dtype=torch.uint8, device="cuda")
            fk.select_topk(reqs, score, idx, ws)
            fk.check_errors(ws)
            got = idx.cpu().numpy()
            for i, v in enumerate(vals):
                q = reqs[i]
                assert got[q.sel0:q.sel0 + q.k].tolist() == orc.select_topk(v, q.k).tolist()


def _recompute_and_compare(case, b, idx_np, label, gpu_stitched=False):
    """The recomputed rows of every request against the oracle on its own
    stitched cache.  gpu_stitched: the device cache was stitched by the GPU
    (else both sides hold the oracle's), so the rounding allowance also
    covers stitched entries either side may round the other way."""
    cfg = case.cfg
    H = f64(b.H)
    Wq, Wk, Wv = f64(b.Wq), f64(b.Wk), f64(b.Wv)
    Kf, Vf, O = f64(b.Kf), f64(b.Vf), f64(b.O)
    store = _store(cfg)
    quant = cfg.kv_storage in ("u8", "u4")
    for (r, row0, n, T, cis), (Ks, Vs) in zip(request_slices(case), _oracle_stitched(case, store)):
        q = b.reqs[r]
        idx = idx_np[q.sel0:q.sel0 + q.k].astype(np.int64)
        Kf0 = np.zeros((T, cfg.n_kv_heads, cfg.head_dim))
        Vf0 = np.zeros_like(Kf0)
        Kf0[:n], Vf0[:n] = Ks, Vs
        S = orc.selected_rows(idx, n, T)
        rows = _rows_for_attention(S)
        Ko, Vo, Oo, S = orc.recompute_selected(H[row0:row0 + T], Wq, Wk, Wv, idx, n, Kf0, Vf0,
                                               cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                                               cfg.rope_base, out_rows=rows, store=store)
        if len(S) == 0:
            continue
        tol = 2e-2 if cfg.dtype == "bf16" else 1e-4
        assert max_rel(Kf[row0 + S], Ko[S]) <= tol
        assert max_rel(Vf[row0 + S], Vo[S]) <= tol
        if store is None:
            assert max_rel(O[q.out0 + rows], Oo) <= tol
        else:
            # bf16: the stated tolerance, widened per (row, head) only by what
            # equally correct bf16 roundings of q, k, v (and, when the GPU
            # stitched the cache, of the stitched entries) can move that row
            st = None
            if gpu_stitched and n:
                st = rounding.stitched_bounds([case.K_cached[i] for i in cis],
                                              [case.V_cached[i] for i in cis], cfg.rope_base,
                                              quant)
            rounding.check_rows(f"{label}[req {r}]", O[q.out0 + rows], H[row0:row0 + T], Wq, Wk,
                                Wv, S, Ko, Vo, Oo, rows, cfg.n_q_heads, cfg.n_kv_heads,
                                cfg.head_dim, cfg.rope_base, tol, stitched=st)
        keep = np.setdiff1d(np.arange(n), S)
        if keep.size:
            # both sides hold bf16-rounded values here: two roundings of values
            # that differ by fp32 arithmetic error can land one ulp (2^-7) apart
            keep_tol = 2.0 ** -7 if store is not None else stitch_tol(cfg)
            assert max_row_rel(Kf[row0 + keep], Ko[keep]) <= keep_tol
            if quant:
                assert max_row_rel(Vf[row0 + keep], Vo[keep]) <= keep_tol


def _load_oracle_stitched(case, b):
    """Write the oracle's stitched cache (in the layer's storage type) into the
    context rows of the device fused cache: the shared input of a unit test
    of the recompute entry point."""
    dt = b.Kf.dtype
    for (r, row0, n, T, cis), (K, V) in zip(request_slices(case), _oracle_stitched(case, _store(case.cfg))):
        if n:
            b.Kf[row0:row0 + n] = torch.from_numpy(K).to(dt).cuda()
            b.Vf[row0:row0 + n] = torch.from_numpy(V).to(dt).cuda()


@pytest.mark.parametrize("name", list(SMALL))
def test_recompute_selected(name):
    # Unit test of fuse_recompute_selected on a fused cache both sides share
    # (the oracle's stitched cache); the stitch has its own parity test.
    case = case_of(name)
    b = buffers(case)
    _load_oracle_stitched(case, b)
    fk.score_deviation(b.desc, b.reqs, b.H, b.Wv, b.Vf, b.score, b.ws)
    fk.select_topk(b.reqs, b.score, b.idx, b.ws)
    fk.recompute_selected(b.desc, b.reqs, b.H, b.Wq, b.Wk, b.Wv, b.idx, b.Kf, b.Vf, b.O, b.ws)
    fk.check_errors(b.ws)
    _recompute_and_compare(case, b, b.idx.cpu().numpy(), f"recompute_selected[{name}]")


# End to end through fuse_layer_step, on the cache the GPU stitched.  The int8
# long-context recipe draws its perturbation scales from LogNormal(-3, 2);
# some of its attention rows have logits so large that a one-ulp bf16
# difference in a stitched key (fp32 versus fp64 dequantise-and-rotate) moves
# them by more than 2e-2: the allowance covers exactly those flips.
@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_8b_layer", "paged3", "ragged_fp32",
                                  "ragged_paged_bf16_d64", "sparse_long_bf16", "int8_4x1024",
                                  "wide_hidden_bf16", "long_pairs2"])
def test_layer_step(name):
    case = case_of(name)
    b = buffers(case)
    fk.layer_step(b.desc, b.chunks, b.reqs, b.H, b.Wq, b.Wk, b.Wv, True, b.idx, b.Kf, b.Vf, b.O,
                  b.score, b.ws)
    fk.check_errors(b.ws)
    idx = b.idx.cpu().numpy()
    score = b.score.cpu().numpy()
    H, Wv = f64(b.H), f64(b.Wv)
    cfg = case.cfg
    for (r, row0, n, T, cis), (K, V) in zip(request_slices(case), _oracle_stitched(case, _store(cfg))):
        q = b.reqs[r]
        sel = idx[q.sel0:q.sel0 + q.k]
        assert np.all(np.diff(sel) > 0) and (q.k == 0 or (sel[0] >= 0 and sel[-1] < n))
        if n and 0 < q.k < n:
            # the selection is a valid top-k of the oracle's scores, up to score tolerance
            s_orc = orc.deviation_scores(H[row0:row0 + n], Wv, V, cfg.n_kv_heads, cfg.head_dim)
            rest = np.setdiff1d(np.arange(n), sel)
            assert s_orc[sel].min() >= s_orc[rest].max() - 2e-3
            assert orc.select_topk(score[q.score0:q.score0 + n], q.k).tolist() == sel.tolist()
    _recompute_and_compare(case, b, idx, f"layer_step[{name}]", gpu_stitched=True)


def _offset16(t):
    """A copy of t whose storage starts 16 bytes past a 256-byte boundary:
    aligned as the ABI requires (16 bytes) but not to 32 bytes."""
    flat = torch.zeros(t.numel() * t.element_size() + 256, dtype=torch.uint8, device=t.device)
    base = (-flat.data_ptr()) % 256 + 16
    v = flat[base:base + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 32 == 16
    return v


# The Q/K/V scatter and the attention output use 256-bit stores when their
# destinations are 32-byte aligned; fused caches and O that are only 16-byte
# aligned take the 16-byte stores instead and must give the same results.
@pytest.mark.parametrize("name", ["qwen3_8b_layer", "sparse_long_bf16"])
def test_layer_step_16_byte_aligned_outputs(name):
    case = case_of(name)
    b = buffers(case)
    b.Kf, b.Vf, b.O = _offset16(b.Kf), _offset16(b.Vf), _offset16(b.O)
    fk.layer_step(b.desc, b.chunks, b.reqs, b.H, b.Wq, b.Wk, b.Wv, True, b.idx, b.Kf, b.Vf, b.O,
                  b.score, b.ws)
    fk.check_errors(b.ws)
    _recompute_and_compare(case, b, b.idx.cpu().numpy(), f"layer_step_16B[{name}]",
                           gpu_stitched=True)


@pytest.mark.parametrize("ratio", [0.0, 1.0])
def test_ratio_endpoints(ratio):
    cfg = synth.scaled(C["tiny_fp32"], ratio=ratio)
    case = make_case(cfg)
    b = buffers(case)
    fk.layer_step(b.desc, b.chunks, b.reqs, b.H, b.Wq, b.Wk, b.Wv, True, b.idx, b.Kf, b.Vf, b.O,
                  b.score, b.ws)
    fk.check_errors(b.ws)
    q = b.reqs[0]
    assert q.k == (0 if ratio == 0.0 else 256)
    _recompute_and_compare(case, b, b.idx.cpu().numpy(), f"ratio[{ratio}]", gpu_stitched=True)
    if ratio == 1.0:
        # full prefill: every row recomputed
        assert b.idx.cpu().tolist() == list(range(256))


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_8b_layer"])
def test_pic_precompute(name):
    cfg = SMALL[name]
    case = case_of(name)
    d = case.draws
    caches = workload.gpu_pic_caches(cfg, case.layouts, d.H_clean, d.Wk, d.Wv)
    tol = 1e-5 if cfg.dtype == "f32" else 2.0 ** -8
    # oracle caches before storage rounding
    Hc, Wk, Wv = f64(d.H_clean), f64(d.Wk), f64(d.Wv)
    got_K, got_V = f64(caches.K), f64(caches.V)
    c0 = 0
    for (_, _, row, _p, n) in synth.chunk_token_rows(case.layouts):
        K, V = orc.pic_precompute(Hc[row:row + n], Wk, Wv, cfg.n_kv_heads, cfg.head_dim, cfg.rope_base)
        assert max_row_rel(got_K[c0:c0 + n], K) <= tol
        assert max_row_rel(got_V[c0:c0 + n], V) <= tol
        c0 += n


def test_device_detects_bad_indices():
    case = case_of("tiny_fp32")
    b = buffers(case)
    fk.stitch_rerotate(b.desc, b.chunks, b.Kf, b.Vf, b.ws)
    fk.check_errors(b.ws)
    k = b.reqs[0].k
    bad = torch.arange(k, dtype=torch.int32, device="cuda")
    bad[3] = 10_000                                        # out of range
    fk.recompute_selected(b.desc, b.reqs, b.H, b.Wq, b.Wk, b.Wv, bad, b.Kf, b.Vf, b.O, b.ws)
    with pytest.raises(fk.FuseError) as e:
        fk.check_errors(b.ws)
    assert e.value.status == fk.FUSE_ERR_DEVICE_BOUNDS
    bad = torch.arange(k, dtype=torch.int32, device="cuda").flip(0).contiguous()   # descending
    fk.recompute_selected(b.desc, b.reqs, b.H, b.Wq, b.Wk, b.Wv, bad, b.Kf, b.Vf, b.O, b.ws)
    with pytest.raises(fk.FuseError) as e:
        fk.check_errors(b.ws)
    assert e.value.status == fk.FUSE_ERR_DEVICE_BOUNDS
    fk.check_errors(b.ws)                                  # cleared after reading


def test_device_detects_bad_block_id():
    case = case_of("paged3")
    b = buffers(case)
    tables = b.storage["block_tables"]
    tables[1][0] = 1 << 30                                 # outside the pool
    fk.stitch_rerotate(b.desc, b.chunks, b.Kf, b.Vf, b.ws)
    with pytest.raises(fk.FuseError) as e:
        fk.check_errors(b.ws)
    assert e.value.status == fk.FUSE_ERR_DEVICE_BOUNDS
