"""Static selectors on the GPU (QCFuse related work, EPIC boundary tokens;
KVBoost section 4.6.1, SelectiveRecompute seam windows): the kernel's indices
equal the oracle's definition bit for bit, and a layer recomputed from them
matches the oracle's recomputation."""

import dataclasses

import numpy as np
import pytest
import torch

from oracle import fusion as orc
from rag_kv_cache_rerotate_gb300 import fusekv as fk
from rag_kv_cache_rerotate_gb300 import synth

from harness import buffers, make_case, request_slices
import test_gpu_parity as parity

pytestmark = pytest.mark.gpu

KINDS = [(fk.SEL_CHUNK_HEAD, "chunk_head"), (fk.SEL_SEAM_TAIL, "seam_tail")]


def _layouts(case):
    """(chunk starts, chunk lengths, N_r) per request, in request order."""
    out = []
    for l in case.layouts:
        lens = [int(x) for x in l.chunk_lens]
        out.append(([sum(lens[:i]) for i in range(len(lens))], lens, int(l.n_ctx)))
    return out


def _select(b, kind, n):
    k = fk.static_select_count(b.reqs, b.chunks, kind, n)
    reqs = fk.requests_with_k(b.reqs, k)
    idx = torch.zeros(max(1, sum(k)), dtype=torch.int32, device="cuda")
    fk.static_select(reqs, b.chunks, kind, n, idx)
    torch.cuda.synchronize()
    return reqs, idx


@pytest.mark.parametrize("name", ["paged3", "qwen3_8b_layer", "ragged_paged_bf16_d64",
                                  "sparse_long_bf16"])
def test_static_select_matches_oracle(name):
    case = parity.case_of(name)
    b = buffers(case)
    lay = _layouts(case)
    for kind, kname in KINDS:
        for n in (0, 1, 16, 37, 700):
            reqs, idx = _select(b, kind, n)
            got = idx.cpu().numpy()
            for r, (s, l, nc) in enumerate(lay):
                q = reqs[r]
                want = orc.static_select(s, l, nc, kname, n)
                assert q.k == len(want)
                assert got[q.sel0:q.sel0 + q.k].tolist() == want.tolist(), (kname, n, r)


@pytest.mark.parametrize("name", ["tiny_fp32", "paged3"])
@pytest.mark.parametrize("kind", [fk.SEL_CHUNK_HEAD, fk.SEL_SEAM_TAIL])
def test_recompute_from_static_selection(name, kind):
    case = parity.case_of(name)
    b = buffers(case)
    reqs, idx = _select(b, kind, 16)
    t = reqs.totals()
    ws = torch.zeros(fk.workspace_size(b.desc, reqs), dtype=torch.uint8, device="cuda")
    O = torch.zeros(max(t.n_out, 1), b.O.shape[1], b.O.shape[2], dtype=b.O.dtype, device="cuda")
    b2 = dataclasses.replace(b, reqs=reqs, idx=idx, O=O, ws=ws)
    fk.stitch_rerotate(b2.desc, b2.chunks, b2.Kf, b2.Vf, b2.ws)
    fk.recompute_selected(b2.desc, b2.reqs, b2.H, b2.Wq, b2.Wk, b2.Wv, b2.idx, b2.Kf, b2.Vf, b2.O,
                          b2.ws)
    fk.check_errors(b2.ws)
    parity._recompute_and_compare(case, b2, idx.cpu().numpy(), f"static_select[{name},{kind}]",
                                  gpu_stitched=True)
