"""Device-side failure detection without a GPU fault: a bounded wait that
runs out is reported through the workspace's error word and leaves the
context usable (the library's one-second mbarrier wait, on a barrier that
nothing arrives on).  No trap, no bad address, no endless wait."""

import time

import pytest
import torch

from rag_kv_cache_rerotate_gb300 import fusekv as fk

from harness import buffers, make_case
from rag_kv_cache_rerotate_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rag_kv_cache_rerotate_gb300 import _build
    _build.build()
    fk.load()


def test_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.monotonic()
    fk.selftest_wait_timeout(ws)
    with pytest.raises(fk.FuseError) as ex:
        fk.check_errors(ws)
    elapsed = time.monotonic() - t0
    assert ex.value.status == fk.FUSE_ERR_TIMEOUT
    assert 0.5 < elapsed < 30.0            # the wait gave up after its limit, not at once
    fk.check_errors(ws)                    # the word was read and cleared
    # the context still runs work: a small layer-step afterwards is error-free
    cfg = synth.scaled(synth.CONFIGS["tiny_fp32"], n_layers=1)
    case = make_case(cfg, synth.draw_layouts(cfg))
    b = buffers(case)
    fk.layer_step(b.desc, b.chunks, b.reqs, b.H, b.Wq, b.Wk, b.Wv, True, b.idx, b.Kf, b.Vf, b.O,
                  b.score, b.ws)
    fk.check_errors(b.ws)
    assert torch.isfinite(b.O).all()


def test_selftest_rejects_a_missing_or_short_workspace():
    with pytest.raises(fk.FuseError):
        fk.selftest_wait_timeout(torch.zeros(0, dtype=torch.uint8, device="cuda"))
    with pytest.raises(fk.FuseError):
        fk.selftest_wait_timeout(torch.zeros(128, dtype=torch.uint8, device="cuda"))
