"""fuse_stack_graph_create / fuse_graph_launch: the layer stack of
fuse_stack_step captured once as a CUDA graph and replayed.  Every replay
must equal the eager stack bit for bit (the kernels are deterministic), also
after the inputs' contents change between replays (the graph reads the
buffers when it runs, not when it was captured).  fuse_stack_step itself is
checked against the oracle in test_gpu_stack.py."""

import pytest
import torch

from rag_kv_cache_rerotate_gb300 import fusekv as fk
from rag_kv_cache_rerotate_gb300 import synth

from harness import buffers, make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rag_kv_cache_rerotate_gb300 import _build
    _build.build()
    fk.load()


def _outputs(bufs, b0):
    return [t.clone() for b in bufs for t in (b.Kf, b.Vf, b.O)] + [b0.idx.clone(),
                                                                   b0.score.clone()]


def _clear(bufs, b0):
    for b in bufs:
        b.Kf.zero_()
        b.Vf.zero_()
        b.O.zero_()
    b0.idx.zero_()
    b0.score.zero_()


@pytest.mark.parametrize("name", ["qwen3_8b_stack36", "tiny_fp32"])
def test_graph_replay_equals_the_eager_stack(name):
    base = synth.CONFIGS[name]
    if name == "qwen3_8b_stack36":
        cfg = synth.scaled(base, chunks_per_request=3, chunk_len=256, query_len=32, n_layers=4,
                           score_layer=1)
    else:
        cfg = synth.scaled(base, n_layers=3, score_layer=2)
    layouts = synth.draw_layouts(cfg)
    cases = [make_case(cfg, layouts, layer=l) for l in range(cfg.n_layers)]
    bufs = [buffers(c) for c in cases]
    b0 = bufs[cfg.score_layer]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        fk.stack_step(b0.desc, b0.reqs, bufs, cfg.score_layer, b0.idx, b0.score, b0.ws)
    fk.check_errors(b0.ws, stream)
    want = _outputs(bufs, b0)

    graph = fk.StackGraph(b0.desc, b0.reqs, bufs, cfg.score_layer, b0.idx, b0.score, b0.ws,
                          stream=stream)
    try:
        for rep in range(2):
            _clear(bufs, b0)
            torch.cuda.synchronize()
            graph.launch(stream)
            fk.check_errors(b0.ws, stream)
            got = _outputs(bufs, b0)
            for i, (g, w) in enumerate(zip(got, want)):
                assert torch.equal(g, w), (rep, i)

        # new contents in the same buffers: the replay follows them
        for b in bufs:
            b.H.mul_(-1)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            fk.stack_step(b0.desc, b0.reqs, bufs, cfg.score_layer, b0.idx, b0.score, b0.ws)
        fk.check_errors(b0.ws, stream)
        want2 = _outputs(bufs, b0)
        _clear(bufs, b0)
        torch.cuda.synchronize()
        graph.launch(stream)
        fk.check_errors(b0.ws, stream)
        for i, (g, w) in enumerate(zip(_outputs(bufs, b0), want2)):
            assert torch.equal(g, w), i
    finally:
        graph.close()
