"""GPU parity of fuse_kivi_quantize (KVBoost section 4.5, Eq. 7): the codes
and the fp16 scale / zero it writes for layer-type chunk caches must equal,
bit for bit, the oracle's KIVI quantisation of the same values (both form
the codes in fp64 with round-half-even and round scale / zero to fp16 once).
The quantiser prepares the int8 / int4 inputs of the benchmark; the parity
tests of the stitch take their int8 caches from the oracle."""

import numpy as np
import pytest
import torch

from oracle import fusion as orc
from rag_kv_cache_rerotate_gb300 import fusekv as fk
from rag_kv_cache_rerotate_gb300 import synth, workload

from harness import f64

pytestmark = pytest.mark.gpu
C = synth.CONFIGS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rag_kv_cache_rerotate_gb300 import _build
    _build.build()
    fk.load()


def _unpack(q, bits):
    q = q.astype(np.uint8)
    if bits == 8:
        return q
    out = np.empty(q.shape[:-1] + (2 * q.shape[-1],), np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


CASES = {
    "u8_bf16_d128": synth.scaled(C["llama3_70b_int8_long"], chunks_per_request=3, chunk_len=None,
                                 chunk_len_range=(1, 300), query_len=8, seed=31),
    "u4_bf16_d128": synth.scaled(C["llama3_70b_int8_long"], chunks_per_request=3, chunk_len=None,
                                 chunk_len_range=(1, 300), query_len=8, kv_storage="u4", seed=32),
    "u8_f32_d64": synth.scaled(C["tiny_fp32"], kv_storage="u8", chunks_per_request=None,
                               chunk_len=None, chunk_count_range=(2, 5),
                               chunk_len_range=(1, 70), seed=33),
    "u4_f32_d64": synth.scaled(C["tiny_fp32"], kv_storage="u4", seed=34),
}


@pytest.mark.parametrize("name", list(CASES))
def test_kivi_quantize_matches_oracle(name):
    cfg = CASES[name]
    bits = 8 if cfg.kv_storage == "u8" else 4
    layouts = synth.draw_layouts(cfg)
    gen = torch.Generator().manual_seed(cfg.seed)
    rows = synth.chunk_token_rows(layouts)
    n_tot = sum(n for (*_, n) in rows)
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    K = (3.0 * torch.randn(n_tot, cfg.n_kv_heads, cfg.head_dim, generator=gen)).to(dt)
    V = torch.randn(n_tot, cfg.n_kv_heads, cfg.head_dim, generator=gen).to(dt)
    # a constant key channel and a constant value group: scale 0, codes 0
    n0 = rows[0][4]
    K[:n0, 0, 5] = 1.25
    V[0, 1, :] = -0.5
    out = workload.gpu_kivi_caches(cfg, layouts, workload.ChunkCaches(K.cuda(), V.cuda()))
    gK, gV = out.K.cpu().numpy(), out.V.cpu().numpy()
    Kn, Vn = f64(K), f64(V)
    c0 = 0
    for ci, (_, _, _, _, n) in enumerate(rows):
        qk, sk, zk = orc.kivi_quantize_key(Kn[c0:c0 + n], bits)
        qv, sv, zv = orc.kivi_quantize_value(Vn[c0:c0 + n], bits)
        assert np.array_equal(_unpack(gK[c0:c0 + n], bits), qk), ci
        assert np.array_equal(_unpack(gV[c0:c0 + n], bits), qv), ci
        assert np.array_equal(out.k_scale[ci].cpu().numpy(), sk.astype(np.float16)), ci
        assert np.array_equal(out.k_zero[ci].cpu().numpy(), zk.astype(np.float16)), ci
        assert np.array_equal(out.v_scale[c0:c0 + n].cpu().numpy(), sv.astype(np.float16)), ci
        assert np.array_equal(out.v_zero[c0:c0 + n].cpu().numpy(), zv.astype(np.float16)), ci
        c0 += n
    assert out.k_scale[0, 0, 5].item() == 0.0
    assert out.v_scale[0, 1].item() == 0.0
