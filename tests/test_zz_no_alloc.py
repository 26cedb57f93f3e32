"""fuse_select_topk_noalloc: the top-k for callers that cannot allocate
device memory (all HBM already handed to a KV-cache pool, or running where
the allocator must not be touched).  Its key scratch is a fixed array inside
the library; this test checks, through the C ABI, that two calls in a row
select exactly what fuse_select_topk (with a caller workspace) selects, and
what the oracle's top-k selects from the same scores.

Kept in a file of its own that pytest collects last; it passes alone in a
fresh process and after the other tests."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import fusion as orc
from rag_kv_cache_rerotate_gb300 import _build
from rag_kv_cache_rerotate_gb300 import fusekv as fk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    _build.build()
    lib = fk.load()
    fn = lib.fuse_select_topk_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return lib


def _scores(rng, sizes):
    vals = []
    for n in sizes:
        v = (rng.integers(-4, 5, size=n) * 0.25).astype(np.float32)   # many ties
        v[: max(1, n // 3)] = rng.standard_normal(max(1, n // 3)).astype(np.float32)
        vals.append(v)
    return torch.from_numpy(np.concatenate(vals)).cuda()


def test_noalloc_topk_matches_workspace_topk_twice(lib):
    rng = np.random.default_rng(21)
    sizes = [4096, 1, 777, 50000, 129, 33024]
    reqs = fk.plan_requests(sizes, [0] * len(sizes), 0.15)
    tot = reqs.totals()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):                          # two calls in a row share the scratch
        score = _scores(rng, sizes)
        want = torch.full((tot.n_sel,), -1, dtype=torch.int32, device="cuda")
        ws = torch.zeros(256 + 4 * tot.n_ctx + 256, dtype=torch.uint8, device="cuda")
        fk.select_topk(reqs, score, want, ws)
        fk.check_errors(ws)
        got = torch.full((tot.n_sel,), -2, dtype=torch.int32, device="cuda")
        st = lib.fuse_select_topk_noalloc(ctypes.byref(reqs.c), score.data_ptr(), got.data_ptr(),
                                          stream)
        assert st == fk.FUSE_OK, fk.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"call {call}"
        # and each request's selection is the oracle's top-k of its scores
        got_h, score_h = got.cpu().numpy(), score.cpu().numpy()
        for i in range(len(sizes)):
            q = reqs[i]
            ref = orc.select_topk(score_h[q.score0:q.score0 + q.n_ctx], q.k)
            assert got_h[q.sel0:q.sel0 + q.k].tolist() == ref.tolist(), (call, i)


def test_noalloc_topk_rejects_oversize(lib):
    n = (1 << 19) + 1
    reqs = fk.plan_requests([n], [0], 0.1)
    score = torch.zeros(n, dtype=torch.float32, device="cuda")
    idx = torch.zeros(reqs.totals().n_sel, dtype=torch.int32, device="cuda")
    st = lib.fuse_select_topk_noalloc(ctypes.byref(reqs.c), score.data_ptr(), idx.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
    assert st == fk.FUSE_ERR_WORKSPACE
