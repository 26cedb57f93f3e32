"""Thin Python binding of libfusekv (the C ABI declared in include/fusekv.h).

Argument marshalling only: tensors are passed as raw device pointers, the
stream as the current torch stream handle.  Every computation runs in the
library's CUDA kernels; there is no Python or CPU fallback, and loading fails
loudly when the library has not been built.
"""

from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfusekv.so")

# status codes (fuse_status_t)
FUSE_OK = 0
FUSE_ERR_INVALID_ARG = 1
FUSE_ERR_MISALIGNED = 2
FUSE_ERR_UNSUPPORTED = 3
FUSE_ERR_WORKSPACE = 4
FUSE_ERR_CUDA = 5
FUSE_ERR_TIMEOUT = 6
FUSE_ERR_DEVICE_BOUNDS = 7

# fuse_dtype_t, fuse_kv_layout_t, fuse_pos_encoding_t
FUSE_F32, FUSE_BF16, FUSE_U8_ASYM, FUSE_U4_ASYM = 0, 1, 2, 3
FUSE_KV_CONTIGUOUS, FUSE_KV_PAGED = 0, 1
FUSE_ROPE_ROTATE_HALF = 0

_c = ctypes


class LayerDesc(_c.Structure):
    _fields_ = [("hidden", _c.c_int32), ("n_q_heads", _c.c_int32), ("n_kv_heads", _c.c_int32),
                ("head_dim", _c.c_int32), ("rope_base", _c.c_double),
                ("pos_encoding", _c.c_int32), ("dtype", _c.c_int32)]


class Chunk(_c.Structure):
    _fields_ = [("k", _c.c_void_p), ("v", _c.c_void_p), ("block_table", _c.c_void_p),
                ("k_scale", _c.c_void_p), ("k_zero", _c.c_void_p), ("v_scale", _c.c_void_p),
                ("v_zero", _c.c_void_p), ("dst_row", _c.c_int64), ("pos", _c.c_int32),
                ("len", _c.c_int32)]


class Chunks(_c.Structure):
    _fields_ = [("n_chunks", _c.c_int32), ("kv_layout", _c.c_int32), ("kv_storage", _c.c_int32),
                ("block_size", _c.c_int32), ("n_pool_blocks", _c.c_int64),
                ("h_chunks", _c.c_void_p), ("d_chunks", _c.c_void_p)]


class Request(_c.Structure):
    _fields_ = [("row0", _c.c_int64), ("score0", _c.c_int64), ("sel0", _c.c_int64),
                ("out0", _c.c_int64), ("n_ctx", _c.c_int32), ("n_query", _c.c_int32),
                ("k", _c.c_int32), ("reserved", _c.c_int32)]


class Requests(_c.Structure):
    _fields_ = [("n_req", _c.c_int32), ("h_req", _c.c_void_p), ("d_req", _c.c_void_p)]


class LayerIO(_c.Structure):
    _fields_ = [("chunks", _c.c_void_p), ("H", _c.c_void_p), ("Wq", _c.c_void_p),
                ("Wk", _c.c_void_p), ("Wv", _c.c_void_p), ("Kf", _c.c_void_p), ("Vf", _c.c_void_p),
                ("O", _c.c_void_p)]


class Copy(_c.Structure):
    _fields_ = [("dst", _c.c_void_p), ("src", _c.c_void_p), ("bytes", _c.c_size_t)]


class LayerUpload(_c.Structure):
    _fields_ = [("slot", _c.c_int32), ("n_copies", _c.c_int32), ("copies", _c.c_void_p)]


class PipelineOp(_c.Structure):
    _fields_ = [("kind", _c.c_int32), ("layer", _c.c_int32), ("slot", _c.c_int32)]


OP_WAIT_FREE, OP_COPY, OP_MARK_READY, OP_WAIT_READY, OP_COMPUTE, OP_MARK_FREE = range(6)


class Totals(_c.Structure):
    _fields_ = [("n_tok", _c.c_int64), ("n_ctx", _c.c_int64), ("n_sel", _c.c_int64),
                ("n_out", _c.c_int64), ("max_ctx", _c.c_int32), ("max_tok", _c.c_int32)]


class TraceEntry(_c.Structure):
    _fields_ = [("kernel", _c.c_char_p), ("ms", _c.c_float)]


class FuseError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None

_P = _c.c_void_p
_SIGS = {
    "fuse_k_from_ratio": (_c.c_int64, [_c.c_double, _c.c_int64]),
    "fuse_plan_requests": (_c.c_int, [_c.c_int32, _P, _P, _c.c_double, _P, _P]),
    "fuse_workspace_size": (_c.c_int, [_P, _P, _c.POINTER(_c.c_size_t)]),
    "fuse_workspace_reset": (_c.c_int, [_P, _c.c_size_t, _P]),
    "fuse_selftest_wait_timeout": (_c.c_int, [_P, _c.c_size_t, _P]),
    "fuse_stitch_rerotate": (_c.c_int, [_P, _P, _P, _P, _c.c_int64, _P, _c.c_size_t, _P]),
    "fuse_score_deviation": (_c.c_int, [_P, _P, _P, _P, _P, _P, _P, _c.c_size_t, _P]),
    "fuse_score_attention_mass": (_c.c_int, [_P, _P, _P, _P, _P, _c.c_int32, _P, _P,
                                             _c.c_size_t, _P]),
    "fuse_score_key_deviation": (_c.c_int, [_P, _P, _P, _P, _P, _c.c_float, _c.c_int32, _P,
                                            _P, _c.c_size_t, _P]),
    "fuse_select_topk": (_c.c_int, [_P, _P, _P, _P, _c.c_size_t, _P]),
    "fuse_recompute_selected": (_c.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                           _c.c_size_t, _P]),
    "fuse_layer_step": (_c.c_int, [_P, _P, _P, _P, _P, _P, _P, _c.c_int32, _P, _P, _P, _P, _P,
                                   _P, _c.c_size_t, _P]),
    "fuse_pic_precompute": (_c.c_int, [_P, _P, _P, _P, _P, _P, _c.c_size_t, _P]),
    "fuse_stack_step_streamed": (_c.c_int, [_P, _P, _c.c_int32, _c.c_int32, _P, _P, _c.c_int32,
                                            _P, _P, _P, _P, _c.c_size_t, _P]),
    "fuse_stack_pipeline_plan": (_c.c_int, [_c.c_int32, _c.c_int32, _P, _c.c_int32, _P,
                                            _c.c_int32, _c.POINTER(_c.c_int32)]),
    "fuse_stack_step": (_c.c_int, [_P, _P, _c.c_int32, _c.c_int32, _P, _P, _P, _P, _c.c_size_t, _P]),
    "fuse_kivi_quantize": (_c.c_int, [_P, _P, _P, _P]),
    "fuse_stack_graph_create": (_c.c_int, [_P, _P, _c.c_int32, _c.c_int32, _P, _P, _P, _P,
                                           _c.c_size_t, _P, _c.POINTER(_c.c_void_p)]),
    "fuse_graph_launch": (_c.c_int, [_c.c_void_p, _P]),
    "fuse_graph_destroy": (None, [_c.c_void_p]),
    "fuse_check_errors": (_c.c_int, [_P, _P, _c.POINTER(_c.c_uint32)]),
    "fuse_static_select_count": (_c.c_int, [_P, _P, _c.c_int32, _c.c_int32, _P]),
    "fuse_static_select": (_c.c_int, [_P, _P, _c.c_int32, _c.c_int32, _P, _P]),
    "fuse_trace_begin": (_c.c_int, [_c.c_int32]),
    "fuse_trace_end": (_c.c_int, [_P, _c.c_int32, _c.POINTER(_c.c_int32)]),
    "fuse_status_string": (_c.c_char_p, [_c.c_int]),
    "fuse_version": (_c.c_int32, []),
}


def load(path: str = LIB_PATH):
    """Load libfusekv.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libfusekv.so is not built ({path}); run __graft_entry__.build()")
    lib = _c.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().fuse_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != FUSE_OK:
        raise FuseError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream) -> Optional[int]:
    if stream is None:
        if not torch.cuda.is_available():
            return None
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ref(x):
    return _c.byref(x) if x is not None else None


# ---------------------------------------------------------------------------
# descriptors and tables
# ---------------------------------------------------------------------------

def layer_desc(hidden: int, n_q_heads: int, n_kv_heads: int, head_dim: int, rope_base: float,
               dtype: int, pos_encoding: int = FUSE_ROPE_ROTATE_HALF) -> LayerDesc:
    return LayerDesc(hidden, n_q_heads, n_kv_heads, head_dim, float(rope_base), pos_encoding, dtype)


def _to_device_bytes(arr, device) -> torch.Tensor:
    raw = bytes(arr)
    t = torch.frombuffer(bytearray(raw), dtype=torch.uint8) if raw else torch.zeros(0, dtype=torch.uint8)
    return t.to(device)


class RequestTable:
    """Host and device copies of a ``fuse_request_t`` array."""

    def __init__(self, reqs: Sequence[Request], device="cuda"):
        self.host = (Request * max(1, len(reqs)))(*reqs)
        self.n = len(reqs)
        self.dev = _to_device_bytes(self.host, device) if device is not None else None
        self.c = Requests(self.n, _c.addressof(self.host),
                          self.dev.data_ptr() if self.dev is not None and self.dev.numel() else None)

    def totals(self) -> Totals:
        t = Totals()
        for r in self.host[: self.n]:
            t.n_tok = max(t.n_tok, r.row0 + r.n_ctx + r.n_query)
            t.n_ctx = max(t.n_ctx, r.score0 + r.n_ctx)
            t.n_sel = max(t.n_sel, r.sel0 + r.k)
            t.n_out = max(t.n_out, r.out0 + r.k + r.n_query)
            t.max_ctx = max(t.max_ctx, r.n_ctx)
            t.max_tok = max(t.max_tok, r.n_ctx + r.n_query)
        return t

    def __getitem__(self, i) -> Request:
        return self.host[i]


def plan_requests(n_ctx: Sequence[int], n_query: Sequence[int], ratio: float,
                  device="cuda") -> RequestTable:
    """Requests laid out back to back; k_r = floor(ratio * N_r + 1e-9)."""
    n = len(n_ctx)
    a = (_c.c_int32 * max(1, n))(*[int(x) for x in n_ctx])
    b = (_c.c_int32 * max(1, n))(*[int(x) for x in n_query])
    out = (Request * max(1, n))()
    tot = Totals()
    _check(load().fuse_plan_requests(n, a, b, float(ratio), out, _c.byref(tot)), "fuse_plan_requests")
    return RequestTable(list(out)[:n], device)


class ChunkTable:
    """Host and device copies of a ``fuse_chunk_t`` array plus its storage mode.

    Keeps references to the tensors the entries point at."""

    def __init__(self, entries: Sequence[Chunk], kv_layout: int, kv_storage: int,
                 block_size: int = 0, n_pool_blocks: int = 0, keep=(), device="cuda"):
        self.entries = list(entries)
        self.host = (Chunk * max(1, len(entries)))(*entries)
        self.dev = _to_device_bytes(self.host, device) if device is not None else None
        self.keep = list(keep)
        self.c = Chunks(len(entries), kv_layout, kv_storage, block_size, n_pool_blocks,
                        _c.addressof(self.host),
                        self.dev.data_ptr() if self.dev is not None and self.dev.numel() else None)


def k_from_ratio(ratio: float, n_ctx: int) -> int:
    return int(load().fuse_k_from_ratio(float(ratio), int(n_ctx)))


def workspace_size(desc: LayerDesc, reqs: RequestTable) -> int:
    n = _c.c_size_t(0)
    _check(load().fuse_workspace_size(_c.byref(desc), _c.byref(reqs.c), _c.byref(n)),
           "fuse_workspace_size")
    return int(n.value)


def alloc_workspace(desc: LayerDesc, reqs: RequestTable, device="cuda") -> torch.Tensor:
    """A zeroed workspace tensor (256-byte aligned by the caching allocator)."""
    ws = torch.zeros(workspace_size(desc, reqs), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def stitch_rerotate(desc, chunks: ChunkTable, Kf, Vf, ws, stream=None):
    _check(load().fuse_stitch_rerotate(_c.byref(desc), _c.byref(chunks.c), _ptr(Kf), _ptr(Vf),
                                       Kf.shape[0], _ptr(ws), ws.numel(), _stream(stream)),
           "fuse_stitch_rerotate")


def score_deviation(desc, reqs: RequestTable, H, Wv, Vf, score, ws, stream=None):
    _check(load().fuse_score_deviation(_c.byref(desc), _c.byref(reqs.c), _ptr(H), _ptr(Wv),
                                       _ptr(Vf), _ptr(score), _ptr(ws), ws.numel(),
                                       _stream(stream)), "fuse_score_deviation")


def score_attention_mass(desc, reqs: RequestTable, H, Wq, Kf, score, ws, accumulate=False,
                         stream=None):
    """Query-aware attention mass of every context token (QCFuse Eqs. 9-10;
    ``accumulate=True`` adds this layer's term, Eq. 20)."""
    _check(load().fuse_score_attention_mass(_c.byref(desc), _c.byref(reqs.c), _ptr(H), _ptr(Wq),
                                            _ptr(Kf), int(bool(accumulate)), _ptr(score),
                                            _ptr(ws), ws.numel(), _stream(stream)),
           "fuse_score_attention_mass")


def score_key_deviation(desc, reqs: RequestTable, H, Wk, Kf, score, ws, weight=1.0,
                        accumulate=False, stream=None):
    """KVBoost Alg. 2 step 2 on the keys, one layer's term:
    ``score (+)= weight * (1 - mean_h cos(R^t W_K x_t, Kf[t]))``; ``weight=1/L``
    over L layers (accumulating after the first) gives the printed delta."""
    _check(load().fuse_score_key_deviation(_c.byref(desc), _c.byref(reqs.c), _ptr(H), _ptr(Wk),
                                           _ptr(Kf), float(weight), int(bool(accumulate)),
                                           _ptr(score), _ptr(ws), ws.numel(), _stream(stream)),
           "fuse_score_key_deviation")


SEL_CHUNK_HEAD, SEL_SEAM_TAIL = 0, 1


def static_select_count(reqs: RequestTable, chunks: ChunkTable, kind: int, n: int) -> list:
    """k_r of the static selector `kind` (SEL_CHUNK_HEAD / SEL_SEAM_TAIL) per request."""
    k = (_c.c_int32 * max(1, reqs.n))()
    _check(load().fuse_static_select_count(_c.byref(reqs.c), _c.byref(chunks.c), int(kind), int(n),
                                           k), "fuse_static_select_count")
    return [int(x) for x in k[:reqs.n]]


def static_select(reqs: RequestTable, chunks: ChunkTable, kind: int, n: int, idx, stream=None):
    _check(load().fuse_static_select(_c.byref(reqs.c), _c.byref(chunks.c), int(kind), int(n),
                                     _ptr(idx), _stream(stream)), "fuse_static_select")


def requests_with_k(reqs: RequestTable, k: Sequence[int], device="cuda") -> RequestTable:
    """The same requests with k_r replaced, idx and O offsets packed again in
    request order."""
    out, sel, row = [], 0, 0
    for r, kr in zip(reqs.host[: reqs.n], k):
        q = Request(r.row0, r.score0, sel, row, r.n_ctx, r.n_query, int(kr), 0)
        sel += int(kr)
        row += int(kr) + r.n_query
        out.append(q)
    return RequestTable(out, device=device)


def select_topk(reqs: RequestTable, score, idx, ws, stream=None):
    _check(load().fuse_select_topk(_c.byref(reqs.c), _ptr(score), _ptr(idx), _ptr(ws), ws.numel(),
                                   _stream(stream)), "fuse_select_topk")


def recompute_selected(desc, reqs: RequestTable, H, Wq, Wk, Wv, idx, Kf, Vf, O, ws, stream=None):
    _check(load().fuse_recompute_selected(_c.byref(desc), _c.byref(reqs.c), _ptr(H), _ptr(Wq),
                                          _ptr(Wk), _ptr(Wv), _ptr(idx), _ptr(Kf), _ptr(Vf),
                                          _ptr(O), _ptr(ws), ws.numel(), _stream(stream)),
           "fuse_recompute_selected")


def layer_step(desc, chunks: ChunkTable, reqs: RequestTable, H, Wq, Wk, Wv, score_this_layer,
               idx, Kf, Vf, O, score, ws, stream=None):
    _check(load().fuse_layer_step(_c.byref(desc), _c.byref(chunks.c), _c.byref(reqs.c), _ptr(H),
                                  _ptr(Wq), _ptr(Wk), _ptr(Wv), int(bool(score_this_layer)),
                                  _ptr(idx), _ptr(Kf), _ptr(Vf), _ptr(O), _ptr(score), _ptr(ws),
                                  ws.numel(), _stream(stream)), "fuse_layer_step")


def stack_step(desc, reqs: RequestTable, layers, score_layer: int, idx, score, ws, stream=None):
    """``layers``: objects with ``chunks`` (ChunkTable), ``H``, ``Wq``, ``Wk``, ``Wv``,
    ``Kf``, ``Vf``, ``O`` (one per layer)."""
    arr = (LayerIO * len(layers))()
    for i, b in enumerate(layers):
        arr[i] = LayerIO(_c.addressof(b.chunks.c), _ptr(b.H), _ptr(b.Wq), _ptr(b.Wk), _ptr(b.Wv),
                         _ptr(b.Kf), _ptr(b.Vf), _ptr(b.O))
    _check(load().fuse_stack_step(_c.byref(desc), _c.byref(reqs.c), len(layers), int(score_layer),
                                  arr, _ptr(idx), _ptr(score), _ptr(ws), ws.numel(),
                                  _stream(stream)), "fuse_stack_step")


class StackGraph:
    """``fuse_stack_step`` captured once as a CUDA graph (``fuse_stack_graph_create``)
    and replayed with ``launch()``; the buffers must stay where they are."""

    def __init__(self, desc, reqs: RequestTable, layers, score_layer: int, idx, score, ws,
                 stream=None):
        arr = (LayerIO * len(layers))()
        for i, b in enumerate(layers):
            arr[i] = LayerIO(_c.addressof(b.chunks.c), _ptr(b.H), _ptr(b.Wq), _ptr(b.Wk),
                             _ptr(b.Wv), _ptr(b.Kf), _ptr(b.Vf), _ptr(b.O))
        self.keep = (desc, reqs, layers, arr, idx, score, ws)
        h = _c.c_void_p(None)
        _check(load().fuse_stack_graph_create(_c.byref(desc), _c.byref(reqs.c), len(layers),
                                              int(score_layer), arr, _ptr(idx), _ptr(score),
                                              _ptr(ws), ws.numel(), _stream(stream), _c.byref(h)),
               "fuse_stack_graph_create")
        self.h = h

    def launch(self, stream=None):
        _check(load().fuse_graph_launch(self.h, _stream(stream)), "fuse_graph_launch")

    def close(self):
        if self.h:
            load().fuse_graph_destroy(self.h)
            self.h = _c.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def stack_pipeline_plan(n_layers: int, score_layer: int, slot_of_layer: Sequence[int],
                        n_slots: int) -> list:
    """The issue order of ``stack_step_streamed``: (kind, layer, slot) tuples."""
    slots = (_c.c_int32 * max(1, n_layers))(*[int(x) for x in slot_of_layer])
    n = _c.c_int32(0)
    st = load().fuse_stack_pipeline_plan(int(n_layers), int(score_layer), slots, int(n_slots),
                                         None, 0, _c.byref(n))
    if st not in (FUSE_OK, FUSE_ERR_WORKSPACE):
        _check(st, "fuse_stack_pipeline_plan")
    ops = (PipelineOp * max(1, n.value))()
    _check(load().fuse_stack_pipeline_plan(int(n_layers), int(score_layer), slots, int(n_slots),
                                           ops, n.value, _c.byref(n)), "fuse_stack_pipeline_plan")
    return [(o.kind, o.layer, o.slot) for o in ops[:n.value]]


def stack_step_streamed(desc, reqs: RequestTable, layers, score_layer: int, uploads, n_slots: int,
                        idx, score, ws, copy_stream, stream=None):
    """``uploads[l]``: (slot, [(dst tensor, src tensor), ...]) -- whole-tensor
    copies that fill layer l's staging slot.  ``copy_stream``: a
    ``torch.cuda.Stream`` other than ``stream``."""
    arr = (LayerIO * len(layers))()
    for i, b in enumerate(layers):
        arr[i] = LayerIO(_c.addressof(b.chunks.c), _ptr(b.H), _ptr(b.Wq), _ptr(b.Wk), _ptr(b.Wv),
                         _ptr(b.Kf), _ptr(b.Vf), _ptr(b.O))
    keep = []
    ups = (LayerUpload * len(layers))()
    for i, (slot, pairs) in enumerate(uploads):
        cs = (Copy * max(1, len(pairs)))()
        for j, (dst, src) in enumerate(pairs):
            nb = src.numel() * src.element_size()
            if dst.numel() * dst.element_size() != nb:
                raise ValueError("a copy's source and destination differ in size")
            cs[j] = Copy(_ptr(dst), _ptr(src), nb)
        keep.append(cs)
        ups[i] = LayerUpload(int(slot), len(pairs), _c.addressof(cs))
    _check(load().fuse_stack_step_streamed(_c.byref(desc), _c.byref(reqs.c), len(layers),
                                           int(score_layer), arr, ups, int(n_slots),
                                           _stream(copy_stream), _ptr(idx), _ptr(score),
                                           _ptr(ws), ws.numel(), _stream(stream)),
           "fuse_stack_step_streamed")


def pic_precompute(desc, chunks: ChunkTable, H_clean, Wk, Wv, ws, stream=None):
    _check(load().fuse_pic_precompute(_c.byref(desc), _c.byref(chunks.c), _ptr(H_clean),
                                      _ptr(Wk), _ptr(Wv), _ptr(ws), ws.numel(), _stream(stream)),
           "fuse_pic_precompute")


def kivi_quantize(desc, src: ChunkTable, dst: ChunkTable, stream=None):
    """KIVI codes and fp16 scale / zero of layer-type chunk caches (KVBoost
    Eq. 7): input preparation for the int8 / int4 storage modes."""
    _check(load().fuse_kivi_quantize(_c.byref(desc), _c.byref(src.c), _c.byref(dst.c),
                                     _stream(stream)), "fuse_kivi_quantize")


def check_errors(ws, stream=None):
    """Synchronise, read and clear the device error word; raise if set."""
    detail = _c.c_uint32(0)
    st = load().fuse_check_errors(_ptr(ws), _stream(stream), _c.byref(detail))
    if st != FUSE_OK:
        raise FuseError(st, f"device (site {detail.value >> 24}, info {detail.value & 0xFFFFFF})")


def selftest_wait_timeout(ws, stream=None):
    """Launch the library's failure-detection self-test: a bounded wait on a
    barrier nothing arrives on, reported as FUSE_ERR_TIMEOUT in ws's error
    word after the wait's one-second limit (read it with check_errors)."""
    _check(load().fuse_selftest_wait_timeout(_ptr(ws), ws.numel(), _stream(stream)),
           "fuse_selftest_wait_timeout")


def workspace_reset(ws, stream=None):
    _check(load().fuse_workspace_reset(_ptr(ws), ws.numel(), _stream(stream)), "fuse_workspace_reset")


def trace_begin(max_records: int = 4096):
    """Start recording CUDA events around every library kernel launch."""
    _check(load().fuse_trace_begin(int(max_records)), "fuse_trace_begin")


def trace_end():
    """Stop recording; returns [(kernel name, ms)] in launch order."""
    cap = 1 << 16
    buf = (TraceEntry * cap)()
    n = _c.c_int32(0)
    _check(load().fuse_trace_end(buf, cap, _c.byref(n)), "fuse_trace_end")
    return [(buf[i].kernel.decode(), float(buf[i].ms)) for i in range(n.value)]
