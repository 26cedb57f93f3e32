"""GPU parity of fuse_stack_step_streamed (QCFuse Figure 9, pipeline cache
fusion; PCR, layer-wise overlapping): every layer's chunk caches are
uploaded from pinned host memory into a ring of staging slots on a copy
stream while the previous layers compute.  The layers share only the
selection, so every output -- the selection, the scoring layer's scores,
and each layer's fused cache and attention rows -- must equal
fuse_stack_step's on the same data, bit for bit (the kernels are
deterministic).  fuse_stack_step itself is checked against the oracle in
test_gpu_stack.py."""

import pytest
import torch

from rag_kv_cache_rerotate_gb300 import fusekv as fk
from rag_kv_cache_rerotate_gb300 import synth

from harness import buffers, make_case

pytestmark = pytest.mark.gpu

_STATE = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rag_kv_cache_rerotate_gb300 import _build
    _build.build()
    fk.load()


def _cases():
    if "cases" not in _STATE:
        cfg = synth.scaled(synth.CONFIGS["qwen3_8b_stack36"], chunks_per_request=3, chunk_len=256,
                           query_len=32, n_layers=4, score_layer=1)
        layouts = synth.draw_layouts(cfg)
        _STATE["cfg"] = cfg
        _STATE["cases"] = [make_case(cfg, layouts, layer=l) for l in range(cfg.n_layers)]
    return _STATE["cfg"], _STATE["cases"]


def _reference():
    if "ref" not in _STATE:
        cfg, cases = _cases()
        bufs = [buffers(c) for c in cases]
        b0 = bufs[cfg.score_layer]
        fk.stack_step(b0.desc, b0.reqs, bufs, cfg.score_layer, b0.idx, b0.score, b0.ws)
        fk.check_errors(b0.ws)
        torch.cuda.synchronize()
        _STATE["ref"] = bufs
    return _STATE["ref"]


class _Layer:
    """A layer of the streamed stack: its own H, weights and outputs, and the
    chunk table of the staging slot its caches are uploaded into."""

    def __init__(self, own, slot_bufs):
        self.chunks = slot_bufs.chunks
        self.H, self.Wq, self.Wk, self.Wv = own.H, own.Wq, own.Wk, own.Wv
        self.Kf, self.Vf, self.O = own.Kf, own.Vf, own.O


@pytest.mark.parametrize("n_slots", [1, 2, 3])
def test_streamed_stack_equals_the_resident_stack(n_slots):
    cfg, cases = _cases()
    ref = _reference()
    own = [buffers(c) for c in cases]
    # the staging slots: the device chunk storage of the first n_slots layers'
    # buffers (every layer has the same layout, so a slot's chunk table serves
    # any layer uploaded into it); it is overwritten before every use
    slots = own[:n_slots]
    order = [cfg.score_layer] + [l for l in range(cfg.n_layers) if l != cfg.score_layer]
    slot_of = {l: i % n_slots for i, l in enumerate(order)}
    host = []
    for b in own:
        pinned = {}
        for name, t in b.storage.items():
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            pinned[name] = h
        host.append(pinned)
    torch.cuda.synchronize()             # the pinned copies above are host work
    for b in slots:                      # nothing of the slots' own data may survive
        for t in b.storage.values():
            t.zero_()                    # on the compute stream: the uploads follow it
    layers = [_Layer(own[l], slots[slot_of[l]]) for l in range(cfg.n_layers)]
    uploads = [(slot_of[l], [(slots[slot_of[l]].storage[name], host[l][name])
                             for name in host[l]]) for l in range(cfg.n_layers)]
    s = own[cfg.score_layer]
    copy_stream = torch.cuda.Stream()
    fk.stack_step_streamed(s.desc, s.reqs, layers, cfg.score_layer, uploads, n_slots, s.idx,
                           s.score, s.ws, copy_stream)
    fk.check_errors(s.ws)
    torch.cuda.synchronize()
    r = ref[cfg.score_layer]
    assert torch.equal(s.idx, r.idx)
    assert torch.equal(s.score, r.score)
    for l in range(cfg.n_layers):
        assert torch.equal(own[l].Kf, ref[l].Kf), l
        assert torch.equal(own[l].Vf, ref[l].Vf), l
        assert torch.equal(own[l].O, ref[l].O), l


def test_streamed_stack_back_to_back_calls():
    # Two calls in a row on one stream, sharing two staging slots, with no
    # ordering added by the caller: the second call uploads other layers'
    # caches into the slots the first call's last layers still read.  The
    # first call's outputs must still equal the resident stack's.
    cfg, cases = _cases()
    ref = _reference()
    n_slots = 2
    first = [buffers(c) for c in cases]
    second = [buffers(c) for c in cases]
    slots = first[:n_slots]
    order = [cfg.score_layer] + [l for l in range(cfg.n_layers) if l != cfg.score_layer]
    slot_of = {l: i % n_slots for i, l in enumerate(order)}
    host = []
    for b in first:
        pinned = {}
        for name, t in b.storage.items():
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            pinned[name] = h
        host.append(pinned)
    torch.cuda.synchronize()
    L = cfg.n_layers

    def run(outs, src_of):
        layers = [_Layer(outs[l], slots[slot_of[l]]) for l in range(L)]
        uploads = [(slot_of[l], [(slots[slot_of[l]].storage[name], host[src_of(l)][name])
                                 for name in host[l]]) for l in range(L)]
        s = outs[cfg.score_layer]
        fk.stack_step_streamed(s.desc, s.reqs, layers, cfg.score_layer, uploads, n_slots, s.idx,
                               s.score, s.ws, torch.cuda.Stream())

    run(first, lambda l: l)                  # the layers' own caches
    run(second, lambda l: (l + 1) % L)       # another layer's caches, at once
    fk.check_errors(first[cfg.score_layer].ws)
    fk.check_errors(second[cfg.score_layer].ws)
    torch.cuda.synchronize()
    r = ref[cfg.score_layer]
    assert torch.equal(first[cfg.score_layer].idx, r.idx)
    assert torch.equal(first[cfg.score_layer].score, r.score)
    for l in range(L):
        assert torch.equal(first[l].Kf, ref[l].Kf), l
        assert torch.equal(first[l].Vf, ref[l].Vf), l
        assert torch.equal(first[l].O, ref[l].O), l
