"""Test glue: seeded draws -> oracle-made chunk caches -> device buffers,
and the comparisons used by the GPU parity tests.

Chunk caches for parity tests are produced by the oracle (fp64, then stored
in the configuration's storage type), never by the CUDA path."""

from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

from oracle import fusion as orc
from rag_kv_cache_rerotate_gb300 import synth, workload


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


@dataclasses.dataclass
class Case:
    cfg: synth.FusionConfig
    layouts: List[synth.RequestLayout]
    draws: synth.LayerDraws
    caches: workload.ChunkCaches       # storage form (CPU tensors)
    K_cached: List[np.ndarray]         # per chunk, the values the cache holds (fp64)
    V_cached: List[np.ndarray]


def _pack(q: np.ndarray, bits: int) -> np.ndarray:
    """Codes as the library stores them: uint8, or for 4 bits two per byte
    along the last axis (element 2m in the low nibble of byte m)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    if bits == 8:
        return q
    return np.ascontiguousarray(q[..., 0::2] | (q[..., 1::2] << 4))


def make_case(cfg: synth.FusionConfig, layouts=None, layer: int = 0, e_scale: float = 1.0) -> Case:
    layouts = layouts if layouts is not None else synth.draw_layouts(cfg)
    draws = synth.draw_layer(cfg, layouts, layer=layer, e_scale=e_scale)
    Hc = f64(draws.H_clean)
    Wk, Wv = f64(draws.Wk), f64(draws.Wv)
    Hkv, d = cfg.n_kv_heads, cfg.head_dim
    Ks, Vs, Kc, Vc = [], [], [], []
    kq_s, kq_z, vq_s, vq_z = [], [], [], []
    for (_, _, row, _pos, n) in synth.chunk_token_rows(layouts):
        K, V = orc.pic_precompute(Hc[row:row + n], Wk, Wv, Hkv, d, cfg.rope_base)
        if cfg.kv_storage in ("u8", "u4"):
            bits = 8 if cfg.kv_storage == "u8" else 4
            qk, sk, zk = orc.kivi_quantize_key(K, bits)
            qv, sv, zv = orc.kivi_quantize_value(V, bits)
            sk16, zk16 = sk.astype(np.float16), zk.astype(np.float16)
            sv16, zv16 = sv.astype(np.float16), zv.astype(np.float16)
            Ks.append(torch.from_numpy(_pack(qk, bits)))
            Vs.append(torch.from_numpy(_pack(qv, bits)))
            kq_s.append(torch.from_numpy(sk16))
            kq_z.append(torch.from_numpy(zk16))
            vq_s.append(torch.from_numpy(sv16))
            vq_z.append(torch.from_numpy(zv16))
            Kc.append(orc.kivi_dequantize(qk, sk16[None].astype(np.float64), zk16[None].astype(np.float64)))
            Vc.append(orc.kivi_dequantize(qv, sv16[..., None].astype(np.float64),
                                          zv16[..., None].astype(np.float64)))
        else:
            dt = torch.bfloat16 if cfg.kv_storage == "bf16" else torch.float32
            Kt = torch.from_numpy(K).to(dt)
            Vt = torch.from_numpy(V).to(dt)
            Ks.append(Kt)
            Vs.append(Vt)
            Kc.append(f64(Kt))
            Vc.append(f64(Vt))
    caches = workload.ChunkCaches(torch.cat(Ks), torch.cat(Vs))
    if cfg.kv_storage in ("u8", "u4"):
        caches.k_scale = torch.stack(kq_s)
        caches.k_zero = torch.stack(kq_z)
        caches.v_scale = torch.cat(vq_s)
        caches.v_zero = torch.cat(vq_z)
    return Case(cfg, layouts, draws, caches, Kc, Vc)


def buffers(case: Case, device="cuda") -> workload.LayerBuffers:
    d = case.draws
    return workload.layer_buffers(case.cfg, case.layouts, d.H, d.Wq, d.Wk, d.Wv, case.caches, device)


def request_slices(case: Case):
    """(request, packed row0, N_r, T_r, chunk indices) in order."""
    out = []
    row = 0
    ci = 0
    for r, l in enumerate(case.layouts):
        m = len(l.chunk_lens)
        out.append((r, row, l.n_ctx, l.n_tok, list(range(ci, ci + m))))
        row += l.n_tok
        ci += m
    return out


def max_rel(a: np.ndarray, b: np.ndarray) -> float:
    """Normwise relative error max|a - b| / max|b| over the whole tensor."""
    den = float(np.max(np.abs(b))) if b.size else 0.0
    return float(np.max(np.abs(a - b))) / den if den > 0 else float(np.max(np.abs(a - b), initial=0.0))


def max_row_rel(a: np.ndarray, b: np.ndarray) -> float:
    """Largest per-row normwise relative error (rows = leading axis)."""
    a = a.reshape(a.shape[0], -1)
    b = b.reshape(b.shape[0], -1)
    num = np.max(np.abs(a - b), axis=1)
    den = np.maximum(np.max(np.abs(b), axis=1), 1e-30)
    return float(np.max(num / den)) if a.shape[0] else 0.0


def stitch_tol(cfg) -> float:
    """Per-row normwise tolerance of the stitched keys: 1e-5 in fp32 mode; in
    bf16 mode the output is rounded to bf16 (unit roundoff 2^-9), so 2^-8."""
    return 1e-5 if cfg.dtype == "f32" else 2.0 ** -8
