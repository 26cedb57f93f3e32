"""Seeded synthetic inputs for one layer-step of RAG KV-cache fusion.

This module draws random numbers and lays out structure (chunk lengths,
request sizes, paged block ids).  It holds none of the method's arithmetic:
no projection, no rotary embedding, no deviation, no selection.  Both the
CPU oracle (through the tests) and the CUDA path consume what it returns.

The recipe follows the workloads described for cache fusion:

* retrieved context ``C = [c_1; ...; c_m]`` of ``N`` tokens with the user
  query ``U`` appended after it (QCFuse, section 2.1.1, Eq. 1);
* a "clean" hidden state ``H_clean ~ N(0, 1)`` from which the chunk caches
  are precomputed independently (QCFuse, section 2.1.2, Eq. 3), and the
  current hidden state ``H = H_clean + e_t * N(0, 1)`` with a per-token
  scale ``e_t ~ LogNormal(mu, sigma)`` standing in for the cross-chunk
  context that the independent caches miss (QCFuse, Eq. 5; KVBoost,
  section 3.3 "seam error");
* projection weights ``W ~ N(0, 1/hidden)``.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class FusionConfig:
    """Shape and distribution parameters of one synthetic workload."""

    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    rope_base: float
    dtype: str                    # "f32" or "bf16": activations, weights, fused cache
    kv_storage: str               # "f32", "bf16", "u8" or "u4" (KIVI asymmetric int8 / int4)
    kv_layout: str                # "contiguous" or "paged"
    ratio: float                  # recompute ratio rho
    w_std: float                  # std of the projection weights
    e_mu: float                   # LogNormal mu of the per-token perturbation scale
    e_sigma: float                # LogNormal sigma
    seed: int
    n_requests: int = 1
    chunks_per_request: Optional[int] = None       # fixed chunk count
    chunk_len: Optional[int] = None                # fixed chunk length
    query_len: Optional[int] = None                # fixed query length
    chunk_count_range: Optional[tuple] = None      # inclusive uniform range
    chunk_len_range: Optional[tuple] = None        # inclusive uniform range
    query_len_range: Optional[tuple] = None        # inclusive uniform range
    block_size: int = 16                           # paged pool block (tokens)
    n_layers: int = 1
    score_layer: int = 0


CONFIGS = {
    # 4 chunks x 64 tokens + 16 query tokens, fp32 throughout.
    "tiny_fp32": FusionConfig(
        name="tiny_fp32", hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
        rope_base=1e4, dtype="f32", kv_storage="f32", kv_layout="contiguous",
        ratio=0.30, w_std=1.0 / 16.0, e_mu=-3.0, e_sigma=1.5, seed=0,
        chunks_per_request=4, chunk_len=64, query_len=16),
    # Qwen3-8B-shaped single layer: 8 chunks x 512 + 64 query tokens, bf16.
    "qwen3_8b_layer": FusionConfig(
        name="qwen3_8b_layer", hidden=4096, n_q_heads=32, n_kv_heads=8,
        head_dim=128, rope_base=1e6, dtype="bf16", kv_storage="bf16",
        kv_layout="contiguous", ratio=0.15, w_std=1.0 / 64.0, e_mu=-3.0,
        e_sigma=1.5, seed=1, chunks_per_request=8, chunk_len=512, query_len=64),
    # Qwen3-8B-shaped 36-layer attention-only stack: 20 chunks x 512 + 128.
    "qwen3_8b_stack36": FusionConfig(
        name="qwen3_8b_stack36", hidden=4096, n_q_heads=32, n_kv_heads=8,
        head_dim=128, rope_base=1e6, dtype="bf16", kv_storage="bf16",
        kv_layout="contiguous", ratio=0.30, w_std=1.0 / 64.0, e_mu=-3.0,
        e_sigma=1.5, seed=2, chunks_per_request=20, chunk_len=512,
        query_len=128, n_layers=36, score_layer=2),
    # 16 requests, Llama-3-8B-shaped layer, K/V in a paged pool of 16-token blocks.
    "llama3_8b_paged_batch16": FusionConfig(
        name="llama3_8b_paged_batch16", hidden=4096, n_q_heads=32,
        n_kv_heads=8, head_dim=128, rope_base=5e5, dtype="bf16",
        kv_storage="bf16", kv_layout="paged", ratio=0.20, w_std=1.0 / 64.0,
        e_mu=-3.0, e_sigma=1.5, seed=3, n_requests=16,
        chunk_count_range=(4, 16), chunk_len_range=(128, 512),
        query_len_range=(32, 128)),
    # 32 chunks x 1024 + 256 query tokens, Llama-3-70B-shaped layer, int8 cache.
    "llama3_70b_int8_long": FusionConfig(
        name="llama3_70b_int8_long", hidden=8192, n_q_heads=64, n_kv_heads=8,
        head_dim=128, rope_base=5e5, dtype="bf16", kv_storage="u8",
        kv_layout="contiguous", ratio=0.10, w_std=1.0 / math.sqrt(8192.0),
        e_mu=-3.0, e_sigma=2.0, seed=4, chunks_per_request=32,
        chunk_len=1024, query_len=256),
}


def scaled(cfg: FusionConfig, **overrides) -> FusionConfig:
    """A copy of ``cfg`` with some fields replaced (smaller test cases)."""
    return dataclasses.replace(cfg, **overrides)


@dataclasses.dataclass
class RequestLayout:
    """Token structure of one request: chunk lengths then the query."""

    chunk_lens: List[int]
    query_len: int

    @property
    def n_ctx(self) -> int:
        return int(sum(self.chunk_lens))

    @property
    def n_tok(self) -> int:
        return self.n_ctx + self.query_len


def draw_layouts(cfg: FusionConfig) -> List[RequestLayout]:
    """Chunk and query lengths of every request (integer draws, seeded)."""
    g = torch.Generator().manual_seed(cfg.seed * 7919 + 17)
    out = []
    for _ in range(cfg.n_requests):
        if cfg.chunks_per_request is not None:
            m = cfg.chunks_per_request
        else:
            lo, hi = cfg.chunk_count_range
            m = int(torch.randint(lo, hi + 1, (1,), generator=g))
        if cfg.chunk_len is not None:
            lens = [cfg.chunk_len] * m
        else:
            lo, hi = cfg.chunk_len_range
            lens = [int(v) for v in torch.randint(lo, hi + 1, (m,), generator=g)]
        if cfg.query_len is not None:
            q = cfg.query_len
        else:
            lo, hi = cfg.query_len_range
            q = int(torch.randint(lo, hi + 1, (1,), generator=g))
        out.append(RequestLayout(lens, q))
    return out


def _cast(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "f32":
        return x.to(torch.float32)
    raise ValueError(dtype)


@dataclasses.dataclass
class LayerDraws:
    """Random tensors of one layer (all requests packed along tokens).

    ``H_clean`` and ``H`` are ``[sum T_r, hidden]``: request r owns rows
    ``[tok0[r], tok0[r] + T_r)``, context first then query.  Query rows are
    not perturbed (they have no cache).  Weights are ``[out, hidden]``.
    """

    H_clean: torch.Tensor
    H: torch.Tensor
    Wq: torch.Tensor
    Wk: torch.Tensor
    Wv: torch.Tensor
    e: torch.Tensor            # [sum T_r] per-token perturbation scale (0 on query rows)


def draw_layer(cfg: FusionConfig, layouts: List[RequestLayout], layer: int = 0,
               device: str = "cpu", e_scale: float = 1.0) -> LayerDraws:
    """Draw ``H_clean``, the perturbed ``H`` and the weights of one layer.

    ``e_scale`` multiplies the perturbation (0 gives ``H == H_clean``).
    On ``device="cuda"`` the draws use a CUDA generator: same recipe,
    different numbers than on the CPU.
    """
    g = torch.Generator(device=device).manual_seed(cfg.seed * 1000003 + layer * 7 + 1)
    D = cfg.hidden
    d = cfg.head_dim
    T = sum(l.n_tok for l in layouts)
    f32 = torch.float32
    H_clean = torch.randn(T, D, generator=g, device=device, dtype=f32)
    noise = torch.randn(T, D, generator=g, device=device, dtype=f32)
    e = torch.exp(cfg.e_mu + cfg.e_sigma * torch.randn(T, generator=g, device=device, dtype=f32))
    ctx_mask = torch.zeros(T, dtype=torch.bool, device=device)
    row = 0
    for l in layouts:
        ctx_mask[row:row + l.n_ctx] = True
        row += l.n_tok
    e = torch.where(ctx_mask, e * e_scale, torch.zeros_like(e))
    H = H_clean + e[:, None] * noise
    del noise
    Wq = torch.randn(cfg.n_q_heads * d, D, generator=g, device=device, dtype=f32) * cfg.w_std
    Wk = torch.randn(cfg.n_kv_heads * d, D, generator=g, device=device, dtype=f32) * cfg.w_std
    Wv = torch.randn(cfg.n_kv_heads * d, D, generator=g, device=device, dtype=f32) * cfg.w_std
    return LayerDraws(_cast(H_clean, cfg.dtype), _cast(H, cfg.dtype), _cast(Wq, cfg.dtype),
                      _cast(Wk, cfg.dtype), _cast(Wv, cfg.dtype), e)


def draw_block_permutation(cfg: FusionConfig, n_blocks: int, layer: int = 0) -> torch.Tensor:
    """A random permutation of pool block ids (paged layout), seeded."""
    g = torch.Generator().manual_seed(cfg.seed * 31337 + layer)
    return torch.randperm(n_blocks, generator=g).to(torch.int32)


def chunk_token_rows(layouts: List[RequestLayout]):
    """(request, chunk, first packed row, first request-local position, length)
    of every chunk, in order.  Pure bookkeeping of the packed layout."""
    out = []
    row = 0
    for r, l in enumerate(layouts):
        pos = 0
        for c, n in enumerate(l.chunk_lens):
            out.append((r, c, row + pos, pos, n))
            pos += n
        row += l.n_tok
    return out
