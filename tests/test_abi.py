"""The C ABI without a GPU: the library loads, exports every function the
header declares, and its host-side logic (k from ratio, request planning,
workspace sizing, argument validation) behaves as documented.  No call here
reaches a kernel launch."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fk():
    from rag_kv_cache_rerotate_gb300 import _build, fusekv
    _build.build()
    fusekv.load()
    return fusekv


def _declared():
    src = open(os.path.join(ROOT, "include", "fusekv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fuse_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(fk):
    names = _declared()
    assert "fuse_layer_step" in names and len(names) >= 13
    lib = fk.load()
    for n in names:
        assert hasattr(lib, n), n


def test_k_from_ratio_host(fk):
    assert fk.k_from_ratio(0.30, 256) == 76
    assert fk.k_from_ratio(0.15, 4096) == 614
    assert fk.k_from_ratio(0.29, 100) == 29
    assert fk.k_from_ratio(0.0, 10) == 0 and fk.k_from_ratio(1.0, 10) == 10
    assert fk.k_from_ratio(2.0, 10) == 10 and fk.k_from_ratio(-1.0, 10) == 0
    assert fk.k_from_ratio(float("nan"), 10) == 0


def test_plan_requests_offsets(fk):
    t = fk.plan_requests([100, 0, 37], [5, 3, 0], 0.2, device=None)
    r = [t[i] for i in range(3)]
    assert [x.row0 for x in r] == [0, 105, 108]
    assert [x.score0 for x in r] == [0, 100, 100]
    assert [x.k for x in r] == [20, 0, 7]
    assert [x.sel0 for x in r] == [0, 20, 20]
    assert [x.out0 for x in r] == [0, 25, 28]
    tot = t.totals()
    assert (tot.n_tok, tot.n_ctx, tot.n_sel, tot.n_out) == (145, 137, 27, 35)


def _desc(fk, **kw):
    a = dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, rope_base=1e4, dtype=fk.FUSE_F32)
    a.update(kw)
    return fk.layer_desc(**a)


def test_workspace_size_and_validation(fk):
    t = fk.plan_requests([256], [16], 0.3, device=None)
    n = fk.workspace_size(_desc(fk), t)
    assert n > 256 and n % 256 == 0
    for bad, code in [(dict(head_dim=96), fk.FUSE_ERR_UNSUPPORTED),
                      (dict(n_q_heads=6, n_kv_heads=4), fk.FUSE_ERR_INVALID_ARG),
                      (dict(n_q_heads=12, n_kv_heads=1), fk.FUSE_ERR_UNSUPPORTED),
                      (dict(hidden=200), fk.FUSE_ERR_UNSUPPORTED),
                      (dict(rope_base=1.0), fk.FUSE_ERR_INVALID_ARG),
                      (dict(pos_encoding=7), fk.FUSE_ERR_UNSUPPORTED),
                      (dict(dtype=fk.FUSE_U8_ASYM), fk.FUSE_ERR_UNSUPPORTED)]:
        with pytest.raises(fk.FuseError) as e:
            fk.workspace_size(_desc(fk, **bad), t)
        assert e.value.status == code, bad


def test_invalid_requests_rejected_before_launch(fk):
    bad = fk.Request()
    bad.n_ctx, bad.n_query, bad.k = 10, 2, 11          # k > N
    t = fk.RequestTable([bad], device=None)
    t.c.d_req = 16                                      # a non-null stand-in, never dereferenced
    with pytest.raises(fk.FuseError) as e:
        fk.workspace_size(_desc(fk), t)
    assert e.value.status == fk.FUSE_ERR_INVALID_ARG


def test_stitch_argument_errors(fk):
    lib = fk.load()
    desc = _desc(fk)
    e = fk.Chunk()
    e.k, e.v, e.dst_row, e.pos, e.len = 4096, 4096, 10, 10, 8
    tab = fk.ChunkTable([e], fk.FUSE_KV_CONTIGUOUS, fk.FUSE_F32, device=None)
    tab.c.d_chunks = 4096
    ws = ctypes.c_void_p(1 << 20)
    # rows past the fused cache
    st = lib.fuse_stitch_rerotate(ctypes.byref(desc), ctypes.byref(tab.c), 4096, 4096, 12, ws, 1 << 20, None)
    assert st == fk.FUSE_ERR_INVALID_ARG
    # misaligned chunk pointer
    e2 = fk.Chunk()
    e2.k, e2.v, e2.dst_row, e2.pos, e2.len = 4100, 4096, 0, 0, 8
    tab2 = fk.ChunkTable([e2], fk.FUSE_KV_CONTIGUOUS, fk.FUSE_F32, device=None)
    tab2.c.d_chunks = 4096
    st = lib.fuse_stitch_rerotate(ctypes.byref(desc), ctypes.byref(tab2.c), 4096, 4096, 64, ws, 1 << 20, None)
    assert st == fk.FUSE_ERR_MISALIGNED
    # missing workspace
    st = lib.fuse_stitch_rerotate(ctypes.byref(desc), ctypes.byref(tab.c), 4096, 4096, 64, None, 0, None)
    assert st == fk.FUSE_ERR_WORKSPACE
    # paged without a block table / pool size
    tab3 = fk.ChunkTable([e], fk.FUSE_KV_PAGED, fk.FUSE_F32, block_size=16, n_pool_blocks=0, device=None)
    tab3.c.d_chunks = 4096
    st = lib.fuse_stitch_rerotate(ctypes.byref(desc), ctypes.byref(tab3.c), 4096, 4096, 64, ws, 1 << 20, None)
    assert st == fk.FUSE_ERR_INVALID_ARG
    # int8 storage without its scales
    tab4 = fk.ChunkTable([e], fk.FUSE_KV_CONTIGUOUS, fk.FUSE_U8_ASYM, device=None)
    tab4.c.d_chunks = 4096
    e.dst_row = 0
    st = lib.fuse_stitch_rerotate(ctypes.byref(desc), ctypes.byref(tab4.c), 4096, 4096, 64, ws, 1 << 20, None)
    assert st == fk.FUSE_ERR_INVALID_ARG


def test_status_strings(fk):
    for s in range(8):
        assert fk.status_string(s)
    assert fk.load().fuse_version() >= 100


def test_struct_layouts_match_header(fk):
    # sizes implied by the header's field order under the platform C ABI
    assert ctypes.sizeof(fk.LayerDesc) == 32
    assert ctypes.sizeof(fk.Chunk) == 72
    assert ctypes.sizeof(fk.Chunks) == 40
    assert ctypes.sizeof(fk.Request) == 48
    assert ctypes.sizeof(fk.Requests) == 24
    assert ctypes.sizeof(fk.Totals) == 40


def _static_layout(fk, seed):
    """Five requests of 1-6 chunks (1-59 tokens each) and 0-8 query rows,
    packed back to back, with host-only tables."""
    import numpy as np
    rng = np.random.default_rng(seed)
    reqs, chunks, layouts, row = [], [], [], 0
    for _ in range(5):
        lens = [int(x) for x in rng.integers(1, 60, size=int(rng.integers(1, 7)))]
        starts = [sum(lens[:i]) for i in range(len(lens))]
        n_ctx, nq = sum(lens), int(rng.integers(0, 9))
        for s0, ln in zip(starts, lens):
            e = fk.Chunk()
            e.dst_row, e.pos, e.len = row + s0, s0, ln
            chunks.append(e)
        reqs.append(fk.Request(row, 0, 0, 0, n_ctx, nq, 0, 0))
        layouts.append((starts, lens, n_ctx))
        row += n_ctx + nq
    return (fk.RequestTable(reqs, device=None), fk.ChunkTable(chunks, 0, 1, device=None), layouts)


@pytest.mark.parametrize("kind,name", [(0, "chunk_head"), (1, "seam_tail")])
def test_static_select_count_matches_oracle(fk, kind, name):
    from oracle import fusion as orc
    for seed in range(4):
        rt, ct, layouts = _static_layout(fk, 11 * seed + kind)
        for n in (0, 1, 3, 16, 100):
            want = [len(orc.static_select(s, l, nc, name, n)) for s, l, nc in layouts]
            assert fk.static_select_count(rt, ct, kind, n) == want


def test_static_select_rejects_bad_tables(fk):
    rt, ct, layouts = _static_layout(fk, 5)
    with pytest.raises(fk.FuseError):
        fk.static_select_count(rt, ct, 2, 16)                        # unknown kind
    with pytest.raises(fk.FuseError):
        fk.static_select_count(rt, ct, 0, -1)                        # negative n
    entries = list(ct.entries)
    entries[0], entries[1] = entries[1], entries[0]                  # not sorted by row
    with pytest.raises(fk.FuseError):
        fk.static_select_count(rt, fk.ChunkTable(entries, 0, 1, device=None), 0, 4)
    orphan = fk.Chunk()
    orphan.dst_row, orphan.len = 10 ** 9, 4                          # outside every request
    with pytest.raises(fk.FuseError):
        fk.static_select_count(rt, fk.ChunkTable(list(ct.entries) + [orphan], 0, 1, device=None), 0, 4)
    # k of the request table must equal the count (checked before any launch)
    k = fk.static_select_count(rt, ct, 1, 16)
    wrong = fk.requests_with_k(rt, [x + 1 for x in k], device=None)
    with pytest.raises(fk.FuseError):
        fk.static_select(wrong, ct, 1, 16, None)


def test_attention_mass_argument_errors(fk):
    # every call below carries one error, found on the host before any launch
    lib = fk.load()
    desc = _desc(fk)
    t = fk.plan_requests([256], [16], 0.3, device=None)
    t.c.d_req = 16                                      # a non-null stand-in, never dereferenced
    need = fk.workspace_size(desc, t)

    def call(H, Wq, Kf, score, ws, nbytes):
        return lib.fuse_score_attention_mass(ctypes.byref(desc), ctypes.byref(t.c), H, Wq, Kf, 0,
                                             score, ws, nbytes, None)

    A = 1 << 20                                         # aligned stand-ins, never dereferenced
    assert call(None, A, A, A, A, need) == fk.FUSE_ERR_INVALID_ARG
    assert call(A, A, None, A, A, need) == fk.FUSE_ERR_INVALID_ARG
    assert call(A + 8, A, A, A, A, need) == fk.FUSE_ERR_MISALIGNED
    assert call(A, A, A, A + 4, A, need) == fk.FUSE_ERR_MISALIGNED
    assert call(A, A, A, A, A, need - 1) == fk.FUSE_ERR_WORKSPACE
    assert call(A, A, A, A, A + 16, need) == fk.FUSE_ERR_MISALIGNED     # workspace: 256 bytes
    assert call(A, A, A, A, None, need) == fk.FUSE_ERR_WORKSPACE
    # the packed query rows (Q, RoPE table, tile statistics) need workspace
    t0 = fk.plan_requests([256], [0], 0.3, device=None)
    assert need > fk.workspace_size(desc, t0)


def test_stack_step_streamed_argument_errors(fk):
    # one valid layer built from aligned stand-in pointers; each call below
    # carries one error in its uploads, found before any copy or launch
    lib = fk.load()
    desc = _desc(fk)
    t = fk.plan_requests([64], [8], 0.25, device=None)
    t.c.d_req = 16
    e = fk.Chunk()
    e.k, e.v, e.dst_row, e.pos, e.len = 4096, 4096, 0, 0, 64
    tab = fk.ChunkTable([e], fk.FUSE_KV_CONTIGUOUS, fk.FUSE_F32, device=None)
    tab.c.d_chunks = 4096
    A = 1 << 20
    layers = (fk.LayerIO * 1)(fk.LayerIO(ctypes.addressof(tab.c), A, A, A, A, A, A, A))
    need = fk.workspace_size(desc, t)

    def call(uploads, n_slots):
        return lib.fuse_stack_step_streamed(ctypes.byref(desc), ctypes.byref(t.c), 1, 0, layers,
                                            uploads, n_slots, None, A, A, A, need, None)

    assert call(None, 1) == fk.FUSE_ERR_INVALID_ARG
    bad = (fk.Copy * 1)(fk.Copy(A, None, 256))                      # no source
    ups = (fk.LayerUpload * 1)(fk.LayerUpload(0, 1, ctypes.addressof(bad)))
    assert call(ups, 1) == fk.FUSE_ERR_INVALID_ARG
    ups2 = (fk.LayerUpload * 1)(fk.LayerUpload(0, 2, None))           # copies missing
    assert call(ups2, 1) == fk.FUSE_ERR_INVALID_ARG
    ok = (fk.Copy * 1)(fk.Copy(A, A, 256))
    ups3 = (fk.LayerUpload * 1)(fk.LayerUpload(1, 1, ctypes.addressof(ok)))   # slot 1 of 1
    assert call(ups3, 1) == fk.FUSE_ERR_INVALID_ARG
    ups4 = (fk.LayerUpload * 1)(fk.LayerUpload(0, 1, ctypes.addressof(ok)))
    assert call(ups4, 0) == fk.FUSE_ERR_INVALID_ARG                   # no slot at all


def test_key_deviation_argument_errors(fk):
    # every call below carries one error, found on the host before any launch
    lib = fk.load()
    desc = _desc(fk)
    t = fk.plan_requests([128], [8], 0.3, device=None)
    t.c.d_req = 16
    need = fk.workspace_size(desc, t)
    A = 1 << 20

    def call(H, Wk, Kf, weight, score, ws, nbytes):
        return lib.fuse_score_key_deviation(ctypes.byref(desc), ctypes.byref(t.c), H, Wk, Kf,
                                            weight, 0, score, ws, nbytes, None)

    assert call(None, A, A, 1.0, A, A, need) == fk.FUSE_ERR_INVALID_ARG
    assert call(A, A, A, float("nan"), A, A, need) == fk.FUSE_ERR_INVALID_ARG
    assert call(A, A, A, float("inf"), A, A, need) == fk.FUSE_ERR_INVALID_ARG
    assert call(A, A + 2, A, 1.0, A, A, need) == fk.FUSE_ERR_MISALIGNED
    assert call(A, A, A, 1.0, A, A, need - 1) == fk.FUSE_ERR_WORKSPACE
    # the fresh keys of every packed row need workspace
    t2 = fk.plan_requests([256], [8], 0.3, device=None)
    assert fk.workspace_size(desc, t2) > need


def test_more_than_65535_requests_are_unsupported(fk):
    ok = fk.plan_requests([1] * 65535, [0] * 65535, 0.5, device=None)
    assert fk.workspace_size(_desc(fk), ok) > 0
    big = fk.plan_requests([1] * 65536, [0] * 65536, 0.5, device=None)
    with pytest.raises(fk.FuseError) as e:
        fk.workspace_size(_desc(fk), big)
    assert e.value.status == fk.FUSE_ERR_UNSUPPORTED


def test_noalloc_topk_request_table_limit(fk):
    lib = fk.load()
    fn = lib.fuse_select_topk_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 4
    big = fk.plan_requests([1] * 65536, [0] * 65536, 0.5, device=None)
    big.c.d_req = 4096                                  # a non-null stand-in, never dereferenced
    assert fn(ctypes.byref(big.c), 4096, 4096, None) == fk.FUSE_ERR_UNSUPPORTED


def test_kivi_quantize_argument_errors(fk):
    lib = fk.load()
    desc = fk.layer_desc(256, 4, 2, 64, 1e4, fk.FUSE_BF16)

    def table(storage, lens, scales=True):
        es = []
        for n in lens:
            e = fk.Chunk()
            e.k, e.v, e.len = 4096, 4096, n
            if scales:
                e.k_scale, e.k_zero, e.v_scale, e.v_zero = 4096, 4096, 4096, 4096
            es.append(e)
        t = fk.ChunkTable(es, fk.FUSE_KV_CONTIGUOUS, storage, device=None)
        t.c.d_chunks = 4096
        return t

    def call(src, dst):
        return lib.fuse_kivi_quantize(ctypes.byref(desc), ctypes.byref(src.c), ctypes.byref(dst.c),
                                      None)

    src = table(fk.FUSE_BF16, [8, 3], scales=False)
    assert call(src, table(fk.FUSE_U8_ASYM, [8, 4])) == fk.FUSE_ERR_INVALID_ARG     # lengths differ
    assert call(src, table(fk.FUSE_U8_ASYM, [8])) == fk.FUSE_ERR_INVALID_ARG        # chunk counts
    assert call(src, table(fk.FUSE_U8_ASYM, [8, 3], scales=False)) == fk.FUSE_ERR_INVALID_ARG
    assert call(src, table(fk.FUSE_BF16, [8, 3])) == fk.FUSE_ERR_UNSUPPORTED        # not codes
    assert call(table(fk.FUSE_F32, [8, 3]), table(fk.FUSE_U4_ASYM, [8, 3])) == fk.FUSE_ERR_UNSUPPORTED
    empty = table(fk.FUSE_BF16, [0, 0], scales=False)
    assert call(empty, table(fk.FUSE_U8_ASYM, [0, 0])) == fk.FUSE_OK                # nothing to do
