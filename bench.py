#!/usr/bin/env python
"""Benchmark of one layer-step of RAG KV-cache fusion on GB300.

Headline workload (the largest single-GPU configuration): the long-context
int8 layer -- 32 chunks x 1024 context tokens + 256 query tokens
(T = 33 024), Llama-3-70B shape (hidden 8192, 64 query / 8 KV heads,
head_dim 128, RoPE base 5e5), bf16 compute, chunk caches stored as KIVI
int8 codes (keys per channel, values per token, fp16 scale / zero)
dequantised in the stitch, recompute ratio 0.1 -- with synthetic inputs.

A step is one ``fuse_layer_step``: stitch + dequantise + re-rotate,
deviation score, top-k, gathered QKV projection with RoPE and scatter,
selected-row causal attention.  The metric is fused (context + query)
tokens per second per layer-step.  Inputs are resident in HBM and larger
than the L2; two independent input sets alternate.  The timed region (K
steps between CUDA events) is repeated and its median reported.

The same line carries the other workloads as extra keys (``workloads``):
the Qwen3-8B-shaped layer, the 16-request paged batch and the 36-layer
stack (36 * T tokens per stack step), each timed the same way.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

``--impl reference`` times the CPU oracle (fp64 numpy) on the machine's host
cores on the headline workload.  Under torchrun (N > 1) every rank runs its
own independent copy of the workload (weak scaling, no collective on the
data path); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "llama3_70b_int8_long"
EXTRA_WORKLOADS = ("qwen3_8b_layer", "llama3_8b_paged_batch16", "qwen3_8b_stack36")
AUX_WORKLOAD = "qwen3_8b_layer"          # scorer, key deviation and streamed stack
METRIC = "cache-fusion fused tokens/s per layer-step"
UNIT = "fused tokens/s"
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return (float(j["hbm_gbs"]), float(j["bf16_tflops"]),
                float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


# ncu DRAM traffic per launch recorded under profiles/, valid only while the
# kernel's sources are unchanged (hash of the files that define it)
_KSRC = {
    "attention_tc": ["attention_tc.cu", "tc_ptx.cuh", "common.cuh", "launch.h"],
    "qkv_gemm_tc": ["gemm_tc.cu", "tc_ptx.cuh", "common.cuh", "launch.h"],
    "deviation_gemm_tc": ["gemm_tc.cu", "tc_ptx.cuh", "common.cuh", "launch.h"],
    "stitch_rerotate": ["stitch.cu", "tc_ptx.cuh", "common.cuh", "launch.h"],
}
_PROFILED = {
    ("attention_tc", "qwen3_8b_layer"): "attn_tc_kernel_qwen3_8b_layer.md",
    ("qkv_gemm_tc", "qwen3_8b_layer"): "gemm_tc_kernel_qwen3_8b_layer.md",
    ("deviation_gemm_tc", "qwen3_8b_layer"): "gemm_tc_kernel_qwen3_8b_layer.md",
    ("attention_tc", "llama3_70b_int8_long"): "attn_tc_kernel_llama3_70b_int8_long.md",
    ("stitch_rerotate", "llama3_70b_int8_long"): "stitch_kernel_llama3_70b_int8_long.md",
    ("qkv_gemm_tc", "llama3_70b_int8_long"): "gemm_tc_kernel_llama3_70b_int8_long.md",
    ("deviation_gemm_tc", "llama3_70b_int8_long"): "gemm_tc_kernel_llama3_70b_int8_long.md",
    ("stitch_rerotate", "qwen3_8b_layer"): "stitch_topk_prepare_qwen3_8b_layer.md",
}


def _traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from its committed ncu
    summary, or None when there is none or its sources changed since."""
    import hashlib
    md = _PROFILED.get((kernel, workload))
    if md is None:
        return None
    path = os.path.join(ROOT, "profiles", md)
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in _KSRC[kernel]:
        with open(os.path.join(ROOT, "rag_kv_cache_rerotate_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    vals = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("sources_sha256_16") != h.hexdigest()[:16]:
        return None
    v = vals.get("traffic_bytes_per_launch." + kernel, vals.get("traffic_bytes_per_launch"))
    return float(v) if v is not None else None


def max_over_ranks(ms: float, ws: int, device) -> float:
    """The slowest rank's time: every rank contributes its own and all get the
    maximum (one all-reduce of a single number; nothing on the data path)."""
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(ws: int, units_per_step: float, steps: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (each rank runs its own copy of the workload)."""
    return ws * units_per_step * steps / (ms / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# workload description (the same for both arms)
# ---------------------------------------------------------------------------

_ELEM = {"f32": 4, "bf16": 2, "u8": 1, "u4": 0.5}


def _set_bytes(cfg, layouts):
    """Bytes of one input set of a layer (H, weights, chunk caches), from the
    shapes alone."""
    D, Hq, Hkv, d = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    es = _ELEM[cfg.dtype]
    T = sum(l.n_tok for l in layouts)
    N = sum(l.n_ctx for l in layouts)
    n = T * D * es + (Hq + 2 * Hkv) * d * D * es + 2 * N * Hkv * d * _ELEM[cfg.kv_storage]
    if cfg.kv_storage in ("u8", "u4"):
        n += 2 * N * Hkv * 2 + 2 * sum(len(l.chunk_lens) for l in layouts) * Hkv * d * 2
    return int(n)


def _n_sets(cfg, layouts):
    return max(2, math.ceil(2 * L2_BYTES / _set_bytes(cfg, layouts)) + 1)


def config_json(cfg, layouts, ws):
    T = sum(l.n_tok for l in layouts)
    N = sum(l.n_ctx for l in layouts)
    from rag_kv_cache_rerotate_gb300 import synth  # noqa: F401
    k = sum(int(math.floor(cfg.ratio * l.n_ctx + 1e-9)) for l in layouts)
    R = k + sum(l.query_len for l in layouts)
    l0 = layouts[0]
    if len(layouts) == 1:
        shape = f"{len(l0.chunk_lens)} chunks x {l0.chunk_lens[0]} context + {l0.query_len} query tokens"
    else:
        shape = (f"{len(layouts)} requests, {sum(len(l.chunk_lens) for l in layouts)} chunks, "
                 f"{N} context + {T - N} query tokens")
    store = {"u8": "KIVI int8", "u4": "KIVI int4", "bf16": "bf16", "f32": "fp32"}[cfg.kv_storage]
    layers = f", {cfg.n_layers} layers scored at layer {cfg.score_layer}" if cfg.n_layers > 1 else ""
    n_sets = _n_sets(cfg, layouts) if cfg.n_layers == 1 else 1
    sb = _set_bytes(cfg, layouts)
    l2 = (f"{n_sets} independent input sets of {sb / 2**20:.0f} MiB alternate "
          f"({n_sets * sb / 2**20:.0f} MiB > 2x the 129 MB L2)" if cfg.n_layers == 1 else
          f"every layer has its own inputs ({cfg.n_layers} x {sb / 2**20:.0f} MiB > 2x the 129 MB L2)")
    return {
        "workload": (f"{cfg.name}: {shape}, hidden {cfg.hidden}, {cfg.n_q_heads}/{cfg.n_kv_heads} "
                     f"heads, head_dim {cfg.head_dim}, RoPE base {cfg.rope_base:g}, ratio "
                     f"{cfg.ratio}, {store} chunk caches{layers}"),
        "tokens_per_step": T * cfg.n_layers,
        "context_tokens": N,
        "recomputed_rows": R,
        "kv_storage": cfg.kv_storage,
        "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
        "l2": l2,
    }


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (every 50 ms) of the SM clock, the power draw and
    the throttle reasons; stop() keeps the samples taken inside the timed
    window when it is given one."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.proc = None
        self.path = os.path.join("/tmp", f"fusekv_clocks_{os.getpid()}.csv")
        sel = []
        try:
            pr = torch.cuda.get_device_properties(device_index)
            bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
            sel = ["-i", bus]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi"] + sel + ["--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                           "-lms", "50"]

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(self.cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    @staticmethod
    def _when(stamp):
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self, window=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((self._when(parts[0]), float(parts[1]), float(parts[2]),
                                 float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        inside = [r for r in rows if window and r[0] is not None and window[0] <= r[0] <= window[1]]
        use = inside or rows
        reasons = set()
        for r in use:
            for n, v in zip(names, r[4]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_min_mhz": min(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "power_w": statistics.median(r[3] for r in use) if use else None,
                "reasons": sorted(reasons), "samples": len(use),
                "window": "timed regions" if inside else "whole sampling period"}


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline object)
# ---------------------------------------------------------------------------

def _blas_lib():
    """The BLAS library numpy loaded, with its thread-count setter and
    getter, or None (the oracle's matrix products run on its threads)."""
    try:
        with open("/proc/self/maps") as f:
            libs = sorted(set(re.findall(r"(/\S*blas\S*\.so\S*)", f.read())))
    except OSError:
        return None
    for path in libs:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sfx in ("scipy_openblas_{}64_", "scipy_openblas_{}", "openblas_{}64_", "openblas_{}"):
            try:
                st = getattr(lib, sfx.format("set_num_threads"))
                gt = getattr(lib, sfx.format("get_num_threads"))
            except AttributeError:
                continue
            st.restype = None
            st.argtypes = [ctypes.c_int]
            gt.restype = ctypes.c_int
            return st, gt
    return None


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_inputs(cfg):
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import harness  # noqa: E402  (test glue: oracle-made chunk caches)
    case = harness.make_case(cfg)
    f = harness.f64
    return case, f(case.draws.H), f(case.draws.Wq), f(case.draws.Wk), f(case.draws.Wv)


def _grow(fn, full, budget_s, start):
    """Time fn(n) on samples of n units, n = start, 4*start, ... up to
    `full`, until one run takes budget_s; returns seconds per unit of the
    last run and its sample size."""
    n = max(1, min(full, start))
    while True:
        t0 = time.perf_counter()
        fn(n)
        dt = time.perf_counter() - t0
        if n >= full or dt >= budget_s / 2:
            return dt / n, n
        n = min(full, max(n + 1, int(n * min(8.0, budget_s / max(dt, 1e-4)))))


def oracle_step_estimate(orc, cfg, case, H, Wq, Wk, Wv, budget_s):
    """Seconds of one oracle layer-step of a single-request workload, from
    the oracle's own functions run on bounded samples: the stitch and the
    top-k in full, the deviation scores of a sample of context rows (scaled
    by N), the projection of a sample of recomputed rows (scaled by R) and the
    attention of a sample of rows (scaled by the keys they read).  Returns
    (seconds, description of the sample)."""
    Hkv, Hq, d, base = cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim, cfg.rope_base
    t0 = time.perf_counter()
    Kc, Vc = orc.stitch_rerotate(case.K_cached, case.V_cached, base)
    t_stitch = time.perf_counter() - t0
    N, T = Kc.shape[0], H.shape[0]
    sc = {}

    def dev(n):
        sc["s"] = orc.deviation_scores(H[:n], Wv, Vc[:n], Hkv, d)
    per_dev, n_dev = _grow(dev, N, budget_s / 4, 64)
    # the selection: the oracle's top-k of full-length scores (the sampled
    # scores repeated over N: the same k and a spread of positions)
    full = np.resize(sc["s"], N)
    t0 = time.perf_counter()
    idx = orc.select_topk(full, orc.k_from_ratio(cfg.ratio, N))
    t_topk = time.perf_counter() - t0
    S = orc.selected_rows(idx, N, T)
    R = len(S)
    proj = {}

    def prj(m):
        rows = S[np.linspace(0, R - 1, m).astype(int)]
        proj["q"] = orc.project_rows(H[rows], Wq, Wk, Wv, rows, Hq, Hkv, d, base)
    per_proj, n_proj = _grow(prj, R, budget_s / 4, 8)
    Kf = np.zeros((T, Hkv, d))
    Vf = np.zeros_like(Kf)
    Kf[:N], Vf[:N] = Kc, Vc
    q = np.zeros((R, Hq, d))
    keys_all = float(np.sum(S + 1))
    att = {}
    # the call's fixed part (the fused cache laid out per head), once per step
    fixed = []
    for _ in range(2):
        t0 = time.perf_counter()
        orc.causal_attention(q, Kf, Vf, S, np.zeros(0, np.int64), Hq, Hkv, d)
        fixed.append(time.perf_counter() - t0)
    t_fixed = min(fixed)

    def attn(m):
        rows = np.unique(np.linspace(0, R - 1, m).astype(int))
        att["keys"] = float(np.sum(S[rows] + 1))
        att["n"] = len(rows)
        t0 = time.perf_counter()
        orc.causal_attention(q, Kf, Vf, S, rows, Hq, Hkv, d)
        att["t"] = time.perf_counter() - t0
    _grow(attn, R, budget_s / 4, 4)
    n_att = att["n"]
    t_attn = t_fixed + max(0.0, att["t"] - t_fixed) * keys_all / att["keys"]
    total = t_stitch + per_dev * N + t_topk + per_proj * R + t_attn
    sample = (f"stitch and top-k in full; deviation of {n_dev}/{N} context rows, projection of "
              f"{n_proj}/{R} and attention of {n_att}/{R} recomputed rows, each scaled to the "
              f"full step (attention by keys read)")
    return total, sample


def cpu_oracle_run(cfg, steps, warmup, budget_s, threads=None, inputs=None):
    """Oracle seconds per step on the host cores; `threads` sets the BLAS
    thread count for the timed part (None: as numpy starts); `inputs` are
    those of _oracle_inputs (made here when None)."""
    from oracle import fusion as orc
    case, H, Wq, Wk, Wv = inputs if inputs is not None else _oracle_inputs(cfg)
    T = H.shape[0] * cfg.n_layers
    blas = _blas_lib()
    used = blas[1]() if blas else None
    old = used
    if threads is not None:
        if blas is None:
            return {"unavailable": "no BLAS thread control found in this numpy"}
        blas[0](int(threads))
        used = blas[1]()
    per_step = budget_s / max(1, steps + warmup)
    try:
        for _ in range(warmup):
            oracle_step_estimate(orc, cfg, case, H, Wq, Wk, Wv, per_step)
        secs, sample = [], ""
        for _ in range(max(1, steps)):
            s, sample = oracle_step_estimate(orc, cfg, case, H, Wq, Wk, Wv, per_step)
            secs.append(s)
    finally:
        if threads is not None and blas is not None and old is not None:
            blas[0](int(old))
    mean = float(np.mean(secs))
    if cfg.n_layers > 1:
        sample += f"; one layer, times {cfg.n_layers}"
        mean *= cfg.n_layers
    return {"value": T / mean, "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "threads": used, "cpu_model": _cpu_model(),
            "sample": sample + f" ({cfg.name}, {max(1, steps)} step(s), fp64 numpy)",
            "ms_per_step": mean * 1e3}


# ---------------------------------------------------------------------------
# native (CUDA) arm
# ---------------------------------------------------------------------------

def make_set(cfg, layouts, layer):
    """One input set on the device: GPU draws, chunk caches from
    fuse_pic_precompute (KIVI-quantised by fuse_kivi_quantize for the int8 /
    int4 workloads)."""
    from rag_kv_cache_rerotate_gb300 import synth, workload
    d = synth.draw_layer(cfg, layouts, layer=layer, device="cuda")
    caches = workload.gpu_pic_caches(cfg, layouts, d.H_clean, d.Wk, d.Wv)
    if cfg.kv_storage in ("u8", "u4"):
        caches = workload.gpu_kivi_caches(cfg, layouts, caches)
    b = workload.layer_buffers(cfg, layouts, d.H, d.Wq, d.Wk, d.Wv, caches, device="cuda",
                               layer=layer)
    del d, caches
    return b


def build_sets(cfg, layouts):
    """The input sets of a workload: one per layer of a stack, else enough
    alternating sets to exceed twice the L2."""
    n = cfg.n_layers if cfg.n_layers > 1 else _n_sets(cfg, layouts)
    return [make_set(cfg, layouts, l) for l in range(n)]


def step_fn(fk, cfg, sets):
    """One step of the workload: a layer-step on the next input set, or the
    whole stack for the 36-layer workload."""
    if cfg.n_layers > 1:
        b0 = sets[cfg.score_layer]

        def stack(i):
            fk.stack_step(b0.desc, b0.reqs, sets, cfg.score_layer, b0.idx, b0.score, b0.ws)
        return stack

    def layer(i):
        b = sets[i % len(sets)]
        fk.layer_step(b.desc, b.chunks, b.reqs, b.H, b.Wq, b.Wk, b.Wv, True, b.idx, b.Kf, b.Vf,
                      b.O, b.score, b.ws)
    return layer


def work_per_launch(cfg, b):
    """Algorithmic work of one launch of each kernel of a layer-step on
    buffers `b` (after a step wrote its selection): bytes for the HBM-bound
    kernels, flops for the contractions."""
    Hkv, Hq, d, D = cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim, cfg.hidden
    es = _ELEM[cfg.dtype]
    idx = b.idx.cpu().numpy().astype(np.int64)
    N = R = 0
    keys = 0.0
    for r in range(b.reqs.n):
        q = b.reqs[r]
        S = np.concatenate([idx[q.sel0:q.sel0 + q.k], np.arange(q.n_ctx, q.n_ctx + q.n_query)])
        keys += float(np.sum(S + 1))
        N += q.n_ctx
        R += q.k + q.n_query
    n_chunks = sum(len(l.chunk_lens) for l in b.layouts)
    stitch = N * Hkv * d * (2 * _ELEM[cfg.kv_storage] + 2 * es)
    if cfg.kv_storage in ("u8", "u4"):
        stitch += 2 * N * Hkv * 2 + 2 * n_chunks * Hkv * d * 2
    return {
        "stitch_rerotate": ("hbm", float(stitch)),
        "deviation_gemm_tc": ("tensor", 2.0 * N * D * Hkv * d),
        "deviation_gemm_simt": ("tensor", 2.0 * N * D * Hkv * d),
        "prepare_rows": ("hbm", 2.0 * R * D * es),
        "qkv_gemm_tc": ("tensor", 2.0 * R * D * (Hq + 2 * Hkv) * d),
        "qkv_gemm_simt": ("tensor", 2.0 * R * D * (Hq + 2 * Hkv) * d),
        "attention_tc": ("tensor", 4.0 * d * Hq * keys),
        "attention_simt": ("tensor", 4.0 * d * Hq * keys),
    }, {"N": N, "R": R, "keys_read": keys}


def time_regions(fn, steps, regions, stream):
    """Milliseconds of `regions` timed regions of `steps` steps each (CUDA
    events on the launching stream, synchronised on both sides)."""
    out = []
    i = 0
    for _ in range(regions):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn(i)
            i += 1
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


def trace_kernels(fk, fn, steps):
    """Per-kernel launches and total ms over `steps` steps with the library's
    kernel trace on (CUDA events around every launch on its stream)."""
    fk.trace_begin(steps * 512 + 64)
    for i in range(steps):
        fn(i)
    torch.cuda.synchronize()
    per = {}
    n = 0
    for name, kms in fk.trace_end():
        c, tot = per.get(name, (0, 0.0))
        per[name] = (c + 1, tot + kms)
        n += 1
    return per, n / max(1, steps)


def kernel_table(per, work, hbm_gbs, bf16_tf, wl=None):
    kernels = {}
    for n, (c, tot) in per.items():
        kernels[n] = {"launches": c, "avg_us": 1e3 * tot / c}
        t = _traffic(n, wl) if wl else None
        if t is not None:
            kernels[n]["traffic"] = t
        if n in work:
            bound, amount = work[n]
            avg_s = tot / c / 1e3
            if bound == "hbm":
                kernels[n]["GB/s"] = amount / avg_s / 1e9
                kernels[n]["frac_hbm"] = kernels[n]["GB/s"] / hbm_gbs
            else:
                kernels[n]["TFLOP/s"] = amount / avg_s / 1e12
                kernels[n]["frac_bf16"] = kernels[n]["TFLOP/s"] / bf16_tf
    return kernels


def roofline(per, work, wl, hbm_gbs, bf16_tf, peak_src):
    dom = max(per.items(), key=lambda kv: kv[1][1])[0] if per else None
    if dom not in work:
        return None
    bound, amount = work[dom]
    c, tot = per[dom]
    avg_s = tot / c / 1e3
    if bound == "hbm":
        ach, peak, unit = amount / avg_s / 1e9, hbm_gbs, "GB/s"
    else:
        ach, peak, unit = amount / avg_s / 1e12, bf16_tf, "TFLOP/s"
    return {"bound": bound, "kernel": dom, "achieved": ach, "peak": peak, "unit": unit,
            "frac": ach / peak, "traffic": _traffic(dom, wl),
            "algorithmic_per_launch": amount, "avg_launch_us": avg_s * 1e6,
            "peak_source": f"{peak_src} ({'bf16 burst' if bound == 'tensor' else 'HBM copy'})"}


def run_workload(fk, name, args, ws, stream, peaks, keep=False):
    """Build, time and trace one workload; returns (result dict, sets)."""
    from rag_kv_cache_rerotate_gb300 import synth
    hbm_gbs, bf16_tf, _, peak_src = peaks
    cfg = synth.CONFIGS[name]
    layouts = synth.draw_layouts(cfg)
    sets = build_sets(cfg, layouts)
    fn = step_fn(fk, cfg, sets)
    for i in range(args.warmup):
        fn(i)
    for b in sets:
        fk.check_errors(b.ws)
    regions = time_regions(fn, args.steps, args.regions, stream)
    for b in sets:
        fk.check_errors(b.ws)
    per, per_step = trace_kernels(fk, fn, args.steps)
    b0 = sets[cfg.score_layer] if cfg.n_layers > 1 else sets[0]
    work, counts = work_per_launch(cfg, b0)
    T = sum(l.n_tok for l in layouts) * cfg.n_layers
    ms = statistics.median(regions)
    res = {"value": job_rate(ws, T, args.steps, ms), "unit": UNIT,
           "ms_per_step": ms / args.steps, "regions_ms": regions,
           "config": config_json(cfg, layouts, ws), "counts": counts,
           "kernels": kernel_table(per, work, hbm_gbs, bf16_tf, name),
           "roofline": roofline(per, work, name, hbm_gbs, bf16_tf, peak_src),
           "launches_per_step": per_step}
    res["graph"] = graph_timing(fk, cfg, sets, args, stream, T, ws)
    if not keep:
        del sets, fn
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        return res, None
    return res, sets


def graph_timing(fk, cfg, sets, args, stream, T, ws):
    """The same steps replayed from CUDA graphs: the stack captured once
    (fuse_stack_graph_create), or for a single layer one graph per input set
    (a one-layer stack that scores its layer is the layer-step), replayed in
    the same alternation.  Reported, not fatal."""
    graphs = []
    try:
        if cfg.n_layers > 1:
            b0 = sets[cfg.score_layer]
            graphs = [fk.StackGraph(b0.desc, b0.reqs, sets, cfg.score_layer, b0.idx, b0.score,
                                    b0.ws, stream=torch.cuda.Stream())]
            what = "fuse_stack_step captured once (fuse_stack_graph_create), replayed per step"
        else:
            # captured on a stream of its own (the legacy stream cannot be
            # captured), replayed on the timing stream
            cap = torch.cuda.Stream()
            graphs = [fk.StackGraph(b.desc, b.reqs, [b], 0, b.idx, b.score, b.ws, stream=cap)
                      for b in sets]
            what = ("fuse_layer_step of each input set captured once as a one-layer "
                    "fuse_stack_graph_create, replayed alternately")
        n = len(graphs)
        for i in range(args.warmup):
            graphs[i % n].launch(stream)
        gms = statistics.median(time_regions(lambda i: graphs[i % n].launch(stream), args.steps,
                                             args.regions, stream))
        for b in sets:
            fk.check_errors(b.ws)
        return {"value": job_rate(ws, T, args.steps, gms), "unit": UNIT,
                "ms_per_step": gms / args.steps, "what": what}
    except Exception as ex:
        return {"error": f"{type(ex).__name__}: {ex}"}
    finally:
        for g in graphs:
            g.close()


def e2e_run(fk, bufs, args, ws, stream, T):
    """End to end through the C ABI with host buffers: every step uploads its
    inputs (chunk caches and H) from pinned host memory and reads its result
    (O and idx) back; two input sets alternate so that one step's upload runs
    on a copy stream while the previous step computes; every copy of every
    step lies inside the timed region."""
    host_in, host_out = [], []
    for b in bufs:
        pairs = []
        for tsr in [b.H] + [v for k, v in b.storage.items()
                            if k in ("K", "V", "k_scale", "k_zero", "v_scale", "v_zero")]:
            h = torch.empty(tsr.shape, dtype=tsr.dtype, pin_memory=True)
            h.copy_(tsr)
            pairs.append((h, tsr))
        host_in.append(pairs)
        host_out.append((torch.empty(b.O.shape, dtype=b.O.dtype, pin_memory=True),
                         torch.empty(b.idx.shape, dtype=b.idx.dtype, pin_memory=True)))
    h2d = sum(h.numel() * h.element_size() for h, _ in host_in[0])
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    up = torch.cuda.Stream()
    down = torch.cuda.Stream()
    computed = [torch.cuda.Event() for _ in bufs]
    uploaded = [torch.cuda.Event() for _ in bufs]
    read = [torch.cuda.Event() for _ in bufs]

    def e2e_step(i):
        s = i % 2
        b = bufs[s]
        up.wait_event(computed[s])                   # the last step on set s read its inputs
        with torch.cuda.stream(up):
            for h, dv in host_in[s]:
                dv.copy_(h, non_blocking=True)
        uploaded[s].record(up)
        stream.wait_event(uploaded[s])
        stream.wait_event(read[s])                   # its previous results are out
        fk.layer_step(b.desc, b.chunks, b.reqs, b.H, b.Wq, b.Wk, b.Wv, True, b.idx, b.Kf, b.Vf,
                      b.O, b.score, b.ws)
        computed[s].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(computed[s])
            O_h, idx_h = host_out[s]
            O_h.copy_(b.O, non_blocking=True)
            idx_h.copy_(b.idx, non_blocking=True)
            read[s].record(down)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(up)                                    # before the first upload
    for u in (stream, down):
        u.wait_event(e0)
    for i in range(args.e2e_steps):
        e2e_step(i)
    for s in range(2):
        stream.wait_event(read[s])                   # after the last read-back
    e1.record(stream)
    torch.cuda.synchronize()
    ems = max_over_ranks(e0.elapsed_time(e1), ws, "cuda")
    for b in bufs:
        fk.check_errors(b.ws)
    return {"value": job_rate(ws, T, args.e2e_steps, ems), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": args.e2e_steps, "ms_per_step": ems / args.e2e_steps,
            "what": "pinned-host chunk caches (int8 codes, fp16 scale / zero) and H copied in, "
                    "fuse_layer_step, O and idx copied out; two input sets alternate, uploads "
                    "overlap the previous step"}


def aux_blocks(fk, args, stream, sets):
    """The scorers and the streamed stack, timed apart from the step on the
    Qwen3-8B-shaped layer's input sets; a failure in one is reported in the
    line instead of ending the run."""
    from rag_kv_cache_rerotate_gb300 import synth
    cfg = synth.CONFIGS[AUX_WORKLOAD]
    out = {}
    n_sets = len(sets)
    q = sets[0].reqs[0]
    T, N, Qn = q.n_ctx + q.n_query, q.n_ctx, q.n_query
    Hkv, Hq, d, D = cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim, cfg.hidden

    def timed_calls(fn, calls):
        for i in range(3):
            fn(sets[i % n_sets])
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for i in range(calls):
            fn(sets[i % n_sets])
        s1.record(stream)
        torch.cuda.synchronize()
        us = 1e3 * s0.elapsed_time(s1) / calls
        fk.trace_begin(calls * 8 + 8)
        for i in range(calls):
            fn(sets[i % n_sets])
        torch.cuda.synchronize()
        per = {}
        for name, kms in fk.trace_end():
            c, tot = per.get(name, (0, 0.0))
            per[name] = (c + 1, tot + kms)
        for b in sets:
            fk.check_errors(b.ws)
        return us, {n: {"launches": c, "avg_us": 1e3 * tot / c} for n, (c, tot) in per.items()}

    # the query-aware attention-mass scorer (QCFuse Eqs. 9-10)
    if args.scorer_calls > 0:
        try:
            us, sk = timed_calls(lambda b: fk.score_attention_mass(b.desc, b.reqs, b.H, b.Wq, b.Kf,
                                                                   b.score, b.ws),
                                 args.scorer_calls)
            s_work = {"query_gemm_tc": 2.0 * Qn * D * Hq * d,
                      "query_gemm_simt": 2.0 * Qn * D * Hq * d,
                      "attention_mass": 2.0 * Qn * Hq * N * d}
            for n, v in sk.items():
                if n in s_work:
                    v["TFLOP/s"] = s_work[n] / (v["avg_us"] / 1e6) / 1e12
            out["attention_mass_scorer"] = {
                "us_per_call": us, "calls": args.scorer_calls, "kernels": sk,
                "work": "query GEMM 2*Qn*D*Hq*d flop; attention mass one Q.K pass 2*Qn*Hq*N*d flop"}
        except Exception as ex:
            out["attention_mass_scorer"] = {"error": f"{type(ex).__name__}: {ex}"}

    # the key deviation over layers (KVBoost Alg. 2 step 2 as printed)
    if args.key_deviation_calls > 0:
        try:
            kus, kk = timed_calls(lambda b: fk.score_key_deviation(b.desc, b.reqs, b.H, b.Wk, b.Kf,
                                                                   b.score, b.ws),
                                  args.key_deviation_calls)
            for n_, v in kk.items():
                avg_s = v["avg_us"] / 1e6
                if n_ in ("key_gemm_tc", "key_gemm_simt"):
                    v["TFLOP/s"] = 2.0 * T * D * Hkv * d / avg_s / 1e12
                if n_ == "key_cosine":
                    v["GB/s"] = 2.0 * N * Hkv * d * 2 / avg_s / 1e9
            out["key_deviation"] = {"us_per_call": kus, "calls": args.key_deviation_calls,
                                    "kernels": kk,
                                    "work": "fresh keys 2*T*D*Hkv*d flop; cosines read 2*N*Hkv*d bf16"}
        except Exception as ex:
            out["key_deviation"] = {"error": f"{type(ex).__name__}: {ex}"}

    # layer-wise loading overlapped with fusion (QCFuse Figure 9; PCR
    # layer-wise overlapping): the input sets as the layers of a stack scored
    # at layer 0, timed three ways -- the resident stack, the uploads of every
    # layer's chunk caches from pinned host memory alone, and the streamed
    # stack through two staging slots (the first two sets' cache storage,
    # overwritten here)
    if args.streamed_layers > 1 and n_sets >= 2:
        try:
            import types
            nl = min(args.streamed_layers, n_sets)
            lay = sets[:nl]
            names = [k for k in lay[0].storage if k in ("K", "V")]
            host = []
            for b in lay:
                hb = {}
                for k in names:
                    h = torch.empty(b.storage[k].shape, dtype=b.storage[k].dtype, pin_memory=True)
                    h.copy_(b.storage[k])
                    hb[k] = h
                host.append(hb)
            up_bytes = sum(h.numel() * h.element_size() for hb in host for h in hb.values())
            b0 = lay[0]
            cstream = torch.cuda.Stream()

            def timed(fn):
                a0 = torch.cuda.Event(enable_timing=True)
                a1 = torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                cstream.wait_event(a0)
                fn()
                stream.wait_stream(cstream)
                a1.record(stream)
                torch.cuda.synchronize()
                return a0.elapsed_time(a1)

            def resident():
                fk.stack_step(b0.desc, b0.reqs, lay, 0, b0.idx, b0.score, b0.ws)

            slots = lay[:2]

            def uploads_only():
                with torch.cuda.stream(cstream):
                    for l in range(nl):
                        for k in names:
                            slots[l % 2].storage[k].copy_(host[l][k], non_blocking=True)

            layers = [types.SimpleNamespace(chunks=slots[l % 2].chunks, H=b.H, Wq=b.Wq, Wk=b.Wk,
                                            Wv=b.Wv, Kf=b.Kf, Vf=b.Vf, O=b.O)
                      for l, b in enumerate(lay)]
            ups = [(l % 2, [(slots[l % 2].storage[k], host[l][k]) for k in names])
                   for l in range(nl)]

            def streamed_stack():
                fk.stack_step_streamed(b0.desc, b0.reqs, layers, 0, ups, 2, b0.idx, b0.score,
                                       b0.ws, cstream)

            res = {}
            for name_, fn in (("resident_ms", resident), ("uploads_ms", uploads_only),
                              ("streamed_ms", streamed_stack)):
                timed(fn)
                res[name_] = statistics.median(timed(fn) for _ in range(args.streamed_reps))
            fk.check_errors(b0.ws)
            hidden = res["resident_ms"] + res["uploads_ms"] - res["streamed_ms"]
            out["streamed_stack"] = dict(
                res, layers=nl, slots=2, upload_bytes=int(up_bytes),
                upload_GBps=up_bytes / (res["uploads_ms"] / 1e3) / 1e9,
                hidden_fraction=hidden / min(res["resident_ms"], res["uploads_ms"]))
        except Exception as ex:
            out["streamed_stack"] = {"error": f"{type(ex).__name__}: {ex}"}
    return out


def native_run(args, ws, rank, local):
    from rag_kv_cache_rerotate_gb300 import _build, fusekv as fk, synth
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if rank == 0:
        _build.build()
    if ws > 1:
        dist.barrier()
    fk.load()
    peaks = _peaks()
    stream = torch.cuda.current_stream()
    cfg = synth.CONFIGS[args.workload]
    layouts = synth.draw_layouts(cfg)
    sets = build_sets(cfg, layouts)
    fn = step_fn(fk, cfg, sets)
    for i in range(args.warmup):
        fn(i)
    for b in sets:
        fk.check_errors(b.ws)
    torch.cuda.synchronize()

    # the headline: `regions` timed regions of K steps, clocks sampled
    # throughout, median region reported
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.5)
    if ws > 1:
        dist.barrier()
    t_win = time.time()
    regions = time_regions(fn, args.steps, args.regions, stream)
    if ws > 1:
        dist.barrier()
    t_win = (t_win, time.time())
    time.sleep(0.1)
    clocks = sampler.stop(t_win)
    ms = max_over_ranks(statistics.median(regions), ws, "cuda")
    for b in sets:
        fk.check_errors(b.ws)

    # per-kernel times: the same steps again with the library's kernel trace
    # on (a separate region, so the events do not perturb the throughput)
    hbm_gbs, bf16_tf, _, peak_src = peaks
    per, per_step = trace_kernels(fk, fn, args.steps)
    work, counts = work_per_launch(cfg, sets[cfg.score_layer] if cfg.n_layers > 1 else sets[0])
    kernels = kernel_table(per, work, hbm_gbs, bf16_tf, args.workload)
    roof = roofline(per, work, args.workload, hbm_gbs, bf16_tf, peak_src)
    T = sum(l.n_tok for l in layouts) * cfg.n_layers

    graph = None if args.profile else graph_timing(fk, cfg, sets, args, stream, T, ws)
    e2e = None
    if args.e2e_steps > 0 and not args.profile and cfg.n_layers == 1:
        e2e = e2e_run(fk, sets[:2], args, ws, stream, T)
    if args.profile and args.profile_scorer > 0:
        # a few query-aware scorer calls on the headline's sets (for a capture)
        for i in range(args.profile_scorer):
            b = sets[i % len(sets)]
            fk.score_attention_mass(b.desc, b.reqs, b.H, b.Wq, b.Kf, b.score, b.ws)
        for b in sets:
            fk.check_errors(b.ws)
    del sets, fn
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    extra, aux = {}, {}
    if not args.profile:
        for name in EXTRA_WORKLOADS:
            if name == args.workload:
                continue
            try:
                keep = name == AUX_WORKLOAD
                res, kept = run_workload(fk, name, args, ws, stream, peaks, keep=keep)
                extra[name] = res
                if kept is not None:
                    aux = aux_blocks(fk, args, stream, kept)
                    del kept
                    torch.cuda.synchronize()
                    torch.cuda.empty_cache()
            except Exception as ex:                # reported, not fatal
                extra[name] = {"error": f"{type(ex).__name__}: {ex}"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not args.profile:
        try:
            inputs = _oracle_inputs(cfg)
            cpu = cpu_oracle_run(cfg, 1, 0, budget_s=args.cpu_budget, inputs=inputs)
            cpu.pop("ms_per_step", None)
            one = cpu_oracle_run(cfg, 1, 0, budget_s=args.cpu_budget, threads=1, inputs=inputs)
            one.pop("ms_per_step", None)
            cpu["single_thread"] = one
            del inputs
        except Exception as ex:
            cpu = {"error": f"{type(ex).__name__}: {ex}"}

    out = {
        "metric": METRIC, "value": job_rate(ws, T, args.steps, ms), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Gaussian draws; chunk caches from fuse_pic_precompute, "
                "KIVI codes from fuse_kivi_quantize)",
        "config": config_json(cfg, layouts, ws), "roofline": roof, "kernels": kernels,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(round(per_step * args.steps * args.regions)),
        "launches_per_step": per_step, "timed_regions": args.regions, "regions_ms": regions,
        "counts": counts, "clocks": clocks, "graph": graph, "impl": "native",
    }
    if extra:
        out["workloads"] = extra
    out.update(aux)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def reference_run(args, ws, rank):
    if rank != 0:
        return
    from rag_kv_cache_rerotate_gb300 import synth
    cfg = synth.CONFIGS[args.workload]
    layouts = synth.draw_layouts(cfg)
    r = cpu_oracle_run(cfg, args.steps, args.warmup, budget_s=args.ref_budget)
    ms = r.pop("ms_per_step")
    out = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_json(cfg, layouts, ws), "impl": "reference", "cpu_baseline": r,
        "e2e": {"value": r["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "ran_on": "rank 0's host cores (the oracle; other ranks exit without work)",
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--regions", type=int, default=10, help="timed regions of K steps (median)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--profile", action="store_true",
                    help="headline workload only (no e2e, extra workloads or CPU baseline)")
    ap.add_argument("--profile-scorer", type=int, default=0,
                    help="with --profile: this many query-aware scorer calls after the steps")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scorer-calls", type=int, default=50)
    ap.add_argument("--key-deviation-calls", type=int, default=50)
    ap.add_argument("--streamed-layers", type=int, default=4)
    ap.add_argument("--streamed-reps", type=int, default=5)
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--ref-budget", type=float, default=120.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = _dist()
    if args.impl == "reference":
        reference_run(args, ws, rank)
    else:
        native_run(args, ws, rank, local)


if __name__ == "__main__":
    main()
