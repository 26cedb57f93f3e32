"""Device buffers of one cache-fusion layer: chunk caches laid out as the
library expects (contiguous per chunk, a shared paged pool, or KIVI int8
codes with fp16 scale/zero), the request and chunk tables, and the fused
cache, score, index, output and workspace buffers.

Layout and bookkeeping only: the chunk caches themselves are produced
elsewhere (by ``fusekv.pic_precompute`` on the GPU, or handed in).
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import torch

from . import fusekv as fk
from .synth import FusionConfig, RequestLayout, chunk_token_rows, draw_block_permutation

_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "u8": torch.uint8, "u4": torch.uint8}
_FUSE = {"f32": fk.FUSE_F32, "bf16": fk.FUSE_BF16, "u8": fk.FUSE_U8_ASYM, "u4": fk.FUSE_U4_ASYM}


def desc_of(cfg: FusionConfig) -> fk.LayerDesc:
    return fk.layer_desc(cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rope_base,
                         _FUSE[cfg.dtype])


@dataclasses.dataclass
class ChunkCaches:
    """Per-chunk cached K/V in storage form, concatenated over all chunks in
    chunk order (``[sum len, Hkv, d]``).  For int8 storage also the KIVI
    parameters: k_scale/k_zero ``[n_chunks, Hkv, d]`` (per channel) and
    v_scale/v_zero ``[sum len, Hkv]`` (per token), fp16."""

    K: torch.Tensor
    V: torch.Tensor
    k_scale: Optional[torch.Tensor] = None
    k_zero: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None
    v_zero: Optional[torch.Tensor] = None


@dataclasses.dataclass
class LayerBuffers:
    cfg: FusionConfig
    layouts: List[RequestLayout]
    desc: fk.LayerDesc
    reqs: fk.RequestTable
    chunks: fk.ChunkTable
    H: torch.Tensor
    Wq: torch.Tensor
    Wk: torch.Tensor
    Wv: torch.Tensor
    Kf: torch.Tensor
    Vf: torch.Tensor
    O: torch.Tensor
    score: torch.Tensor
    idx: torch.Tensor
    ws: torch.Tensor
    chunk_rows: list          # (request, chunk, packed row, position, len) per chunk
    storage: dict             # the tensors the chunk table points at


def plan(cfg: FusionConfig, layouts: Sequence[RequestLayout], device="cuda") -> fk.RequestTable:
    return fk.plan_requests([l.n_ctx for l in layouts], [l.query_len for l in layouts], cfg.ratio,
                            device=device)


def _contiguous_storage(cfg, rows, caches: ChunkCaches, device):
    Kst = caches.K.to(device).contiguous()
    Vst = caches.V.to(device).contiguous()
    store = {"K": Kst, "V": Vst}
    quant = cfg.kv_storage in ("u8", "u4")
    if quant:
        for name in ("k_scale", "k_zero", "v_scale", "v_zero"):
            store[name] = getattr(caches, name).to(device).contiguous()
    row_bytes_k = Kst[0].numel() * Kst.element_size()
    entries = []
    c0 = 0
    for ci, (_, _, row, pos, n) in enumerate(rows):
        e = fk.Chunk()
        e.k = Kst.data_ptr() + c0 * row_bytes_k
        e.v = Vst.data_ptr() + c0 * row_bytes_k
        if quant:
            hd = cfg.n_kv_heads * cfg.head_dim
            e.k_scale = store["k_scale"].data_ptr() + ci * hd * 2
            e.k_zero = store["k_zero"].data_ptr() + ci * hd * 2
            e.v_scale = store["v_scale"].data_ptr() + c0 * cfg.n_kv_heads * 2
            e.v_zero = store["v_zero"].data_ptr() + c0 * cfg.n_kv_heads * 2
        e.dst_row = row
        e.pos = pos
        e.len = n
        entries.append(e)
        c0 += n
    table = fk.ChunkTable(entries, fk.FUSE_KV_CONTIGUOUS, _FUSE[cfg.kv_storage],
                          keep=list(store.values()), device=device)
    return table, store


def _paged_storage(cfg, rows, caches: ChunkCaches, device, layer=0):
    bs = cfg.block_size
    nblk_per = [(n + bs - 1) // bs for (_, _, _, _, n) in rows]
    n_blocks = sum(nblk_per)
    perm = draw_block_permutation(cfg, n_blocks, layer)
    Hkv, d = cfg.n_kv_heads, cfg.head_dim
    dt = caches.K.dtype
    dk = caches.K.shape[-1]               # d, or d / 2 bytes of packed 4-bit codes
    Kpool = torch.zeros(n_blocks, bs, Hkv, dk, dtype=dt, device=device)
    Vpool = torch.zeros(n_blocks, bs, Hkv, dk, dtype=dt, device=device)
    quant = cfg.kv_storage in ("u8", "u4")
    store = {"K": Kpool, "V": Vpool}
    if quant:
        store["k_scale"] = caches.k_scale.to(device).contiguous()
        store["k_zero"] = caches.k_zero.to(device).contiguous()
        store["v_scale"] = torch.zeros(n_blocks, bs, Hkv, dtype=torch.float16, device=device)
        store["v_zero"] = torch.zeros(n_blocks, bs, Hkv, dtype=torch.float16, device=device)
    K = caches.K.to(device)
    V = caches.V.to(device)
    # pool slot of every cached token: block perm[b0 + r // bs], row r % bs
    slots = []
    b0 = 0
    for ci, (_, _, _, _, n) in enumerate(rows):
        r = torch.arange(n)
        slots.append(perm[b0 + r // bs].to(torch.int64) * bs + r % bs)
        b0 += nblk_per[ci]
    slots = torch.cat(slots).to(device) if slots else torch.zeros(0, dtype=torch.int64, device=device)
    Kpool.view(-1, Hkv, dk)[slots] = K
    Vpool.view(-1, Hkv, dk)[slots] = V
    if quant:
        store["v_scale"].view(-1, Hkv)[slots] = caches.v_scale.to(device)
        store["v_zero"].view(-1, Hkv)[slots] = caches.v_zero.to(device)
    tables = []
    entries = []
    b0 = 0
    for ci, (_, _, row, pos, n) in enumerate(rows):
        nb = nblk_per[ci]
        ids = perm[b0:b0 + nb].to(device)
        tables.append(ids)
        e = fk.Chunk()
        e.k = Kpool.data_ptr()
        e.v = Vpool.data_ptr()
        e.block_table = ids.data_ptr()
        if quant:
            hd = Hkv * d
            e.k_scale = store["k_scale"].data_ptr() + ci * hd * 2
            e.k_zero = store["k_zero"].data_ptr() + ci * hd * 2
            e.v_scale = store["v_scale"].data_ptr()
            e.v_zero = store["v_zero"].data_ptr()
        e.dst_row = row
        e.pos = pos
        e.len = n
        entries.append(e)
        b0 += nb
    store["block_tables"] = tables
    table = fk.ChunkTable(entries, fk.FUSE_KV_PAGED, _FUSE[cfg.kv_storage], block_size=bs,
                          n_pool_blocks=n_blocks, keep=list(store.values()) + tables, device=device)
    return table, store


def chunk_table(cfg: FusionConfig, layouts, caches: ChunkCaches, device="cuda", layer=0):
    rows = chunk_token_rows(layouts)
    if cfg.kv_layout == "paged":
        return _paged_storage(cfg, rows, caches, device, layer) + (rows,)
    return _contiguous_storage(cfg, rows, caches, device) + (rows,)


def layer_buffers(cfg: FusionConfig, layouts, H, Wq, Wk, Wv, caches: ChunkCaches,
                  device="cuda", layer=0) -> LayerBuffers:
    """Everything one ``fuse_layer_step`` call needs, on the device."""
    reqs = plan(cfg, layouts, device)
    tot = reqs.totals()
    chunks, store, rows = chunk_table(cfg, layouts, caches, device, layer)
    dt = _TORCH[cfg.dtype]
    Hkv, Hq, d = cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim
    desc = desc_of(cfg)
    return LayerBuffers(
        cfg=cfg, layouts=list(layouts), desc=desc, reqs=reqs, chunks=chunks,
        H=H.to(device).contiguous(), Wq=Wq.to(device).contiguous(), Wk=Wk.to(device).contiguous(),
        Wv=Wv.to(device).contiguous(),
        Kf=torch.zeros(tot.n_tok, Hkv, d, dtype=dt, device=device),
        Vf=torch.zeros(tot.n_tok, Hkv, d, dtype=dt, device=device),
        O=torch.zeros(max(tot.n_out, 1), Hq, d, dtype=dt, device=device),
        score=torch.zeros(max(tot.n_ctx, 1), dtype=torch.float32, device=device),
        idx=torch.zeros(max(tot.n_sel, 1), dtype=torch.int32, device=device),
        ws=fk.alloc_workspace(desc, reqs, device),
        chunk_rows=rows, storage=store)


def gpu_pic_caches(cfg: FusionConfig, layouts, H_clean, Wk, Wv, device="cuda") -> ChunkCaches:
    """Chunk caches computed on the GPU by ``fuse_pic_precompute`` (each chunk
    alone, at local positions), in the compute dtype.  Contiguous storage."""
    rows = chunk_token_rows(layouts)
    n_tot = sum(n for (*_, n) in rows)
    dt = _TORCH[cfg.dtype]
    K = torch.empty(n_tot, cfg.n_kv_heads, cfg.head_dim, dtype=dt, device=device)
    V = torch.empty_like(K)
    row_bytes = K[0].numel() * K.element_size()
    entries = []
    c0 = 0
    for (_, _, row, pos, n) in rows:
        e = fk.Chunk()
        e.k = K.data_ptr() + c0 * row_bytes
        e.v = V.data_ptr() + c0 * row_bytes
        e.dst_row = row
        e.pos = pos
        e.len = n
        entries.append(e)
        c0 += n
    table = fk.ChunkTable(entries, fk.FUSE_KV_CONTIGUOUS, _FUSE[cfg.dtype], keep=[K, V], device=device)
    desc = desc_of(cfg)
    ws = torch.zeros(256, dtype=torch.uint8, device=device)
    fk.pic_precompute(desc, table, H_clean.to(device).contiguous(), Wk.to(device).contiguous(),
                      Wv.to(device).contiguous(), ws)
    fk.check_errors(ws)
    return ChunkCaches(K, V)


def gpu_kivi_caches(cfg: FusionConfig, layouts, caches: ChunkCaches, device="cuda") -> ChunkCaches:
    """KIVI codes of layer-type chunk caches (``fuse_kivi_quantize``), in the
    storage ``cfg.kv_storage`` ("u8" or "u4"), laid out as ``ChunkCaches``
    expects: codes ``[sum len, Hkv, d]`` (``d / 2`` bytes for 4 bits), key
    scale / zero ``[n_chunks, Hkv, d]`` and value scale / zero
    ``[sum len, Hkv]`` in fp16."""
    rows = chunk_token_rows(layouts)
    Hkv, d = cfg.n_kv_heads, cfg.head_dim
    n_tot = sum(n for (*_, n) in rows)
    dk = d // 2 if cfg.kv_storage == "u4" else d
    f16 = torch.float16
    out = ChunkCaches(torch.empty(n_tot, Hkv, dk, dtype=torch.uint8, device=device),
                      torch.empty(n_tot, Hkv, dk, dtype=torch.uint8, device=device),
                      torch.empty(len(rows), Hkv, d, dtype=f16, device=device),
                      torch.empty(len(rows), Hkv, d, dtype=f16, device=device),
                      torch.empty(n_tot, Hkv, dtype=f16, device=device),
                      torch.empty(n_tot, Hkv, dtype=f16, device=device))
    K, V = caches.K.to(device).contiguous(), caches.V.to(device).contiguous()
    src_row = K[0].numel() * K.element_size()
    src, dst = [], []
    c0 = 0
    for ci, (_, _, row, pos, n) in enumerate(rows):
        e = fk.Chunk()
        e.k = K.data_ptr() + c0 * src_row
        e.v = V.data_ptr() + c0 * src_row
        e.dst_row, e.pos, e.len = row, pos, n
        src.append(e)
        q = fk.Chunk()
        q.k = out.K.data_ptr() + c0 * Hkv * dk
        q.v = out.V.data_ptr() + c0 * Hkv * dk
        q.k_scale = out.k_scale.data_ptr() + ci * Hkv * d * 2
        q.k_zero = out.k_zero.data_ptr() + ci * Hkv * d * 2
        q.v_scale = out.v_scale.data_ptr() + c0 * Hkv * 2
        q.v_zero = out.v_zero.data_ptr() + c0 * Hkv * 2
        q.dst_row, q.pos, q.len = row, pos, n
        dst.append(q)
        c0 += n
    t_src = fk.ChunkTable(src, fk.FUSE_KV_CONTIGUOUS, _FUSE[cfg.dtype], keep=[K, V], device=device)
    t_dst = fk.ChunkTable(dst, fk.FUSE_KV_CONTIGUOUS, _FUSE[cfg.kv_storage], device=device)
    fk.kivi_quantize(desc_of(cfg), t_src, t_dst)
    torch.cuda.synchronize()
    return out
