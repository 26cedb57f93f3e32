// The exported C ABI of libfusekv: argument validation, workspace carving,
// and the order of launches of one layer-step (QCFuse section 2.1, Eqs.
// 4-7; KVBoost Alg. 2: stitch, probe/deviation, select, patch).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "launch.h"
#include "trace.h"

namespace fusekv {

// Tensor-core paths (bf16), defined in their own translation units.
bool tc_gemm_supported(const fuse_layer_desc_t& desc);
cudaError_t launch_deviation_partials_tc(const fuse_layer_desc_t& desc, int64_t n_rows,
                                         const void* H, const void* Wv, const void* Vf,
                                         const int32_t* map, const fuse_request_t* d_req,
                                         int n_req, float* partial,
                                         const fuse_chunks_t* v_chunks, uint32_t* err,
                                         cudaStream_t s);
int deviation_tc_ctas(const fuse_layer_desc_t& d, int64_t n_rows);
cudaError_t launch_project_recompute_tc(const fuse_layer_desc_t& desc, int64_t n_rows,
                                        const WorkRow* rows, const float2* rope, const void* H,
                                        const void* Wq, const void* Wk, const void* Wv, void* Q,
                                        void* Kf, void* Vf, void* Hs, uint32_t* err, cudaStream_t s);
cudaError_t launch_project_query_tc(const fuse_layer_desc_t& d, int64_t n_rows, const float2* rope,
                                    const void* Wq, void* Q, const void* Hs, uint32_t* err,
                                    cudaStream_t s, float* split_ws = nullptr, int max_splits = 1);
bool tc_attention_supported(const fuse_layer_desc_t& desc);
cudaError_t launch_selftest_wait(uint32_t* err, cudaStream_t s);
// Query rows projected head by head with the rows on the MMA's short side
// (csrc/query_proj_tc.cu).
bool qproj_tc_supported(const fuse_layer_desc_t& d, int64_t n_rows);
cudaError_t launch_qproj_tc(const fuse_layer_desc_t& d, int64_t n_rows, const float2* rope,
                            const void* Wq, const void* X, void* Q, float* part, int max_splits,
                            uint32_t* err, cudaStream_t s);
// Query-aware attention mass on the tensor cores (csrc/attention_mass_tc.cu).
bool mass_tc_supported(const fuse_layer_desc_t& d);
int mass_tc_chunks(const fuse_layer_desc_t& d, const fuse_requests_t& reqs, int max_ctx,
                   int max_query);
cudaError_t launch_attention_mass_tc(const fuse_layer_desc_t& d, const fuse_requests_t& reqs,
                                     int max_ctx, int max_query, int64_t n_qrows, int64_t n_tok,
                                     const int32_t* qoff, const void* Q, const void* Kf,
                                     float2* stats, float* part, int n_chunks, float* score,
                                     int accumulate, uint32_t* err, cudaStream_t s);
// Key deviation (csrc/key_deviation.cu).
cudaError_t launch_key_rows(const fuse_requests_t& reqs, int max_tok, const RopeFreqs& freqs,
                            int head_dim, int64_t n_rows, WorkRow* rows, float2* rope,
                            cudaStream_t s);
cudaError_t launch_key_cosine(const fuse_layer_desc_t& d, const fuse_requests_t& reqs, int max_ctx,
                              const void* Kn, const void* Kf, float weight, int accumulate,
                              float* score, cudaStream_t s);
int attention_rtile(const fuse_layer_desc_t& d);
size_t attention_tiles_bytes(int64_t n_out, int n_req);
cudaError_t launch_attention_tc(const fuse_layer_desc_t& d, const fuse_requests_t& reqs,
                                int64_t n_out, int64_t n_tok, const WorkRow* rows,
                                const int32_t* idx, const void* Q, const void* Kf, const void* Vf,
                                void* O, void* tiles_ws, bool tiles_ready, uint32_t* err,
                                cudaStream_t s);

namespace {

constexpr int kMaxPosition = 1 << 24;   // positions stay exact in fp32
constexpr int kMaxRequests = 65535;      // launch grids give each request one y index

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_size(int dtype) { return dtype == FUSE_F32 ? 4 : (dtype == FUSE_BF16 ? 2 : 1); }

fuse_status_t check_desc(const fuse_layer_desc_t* d) {
  if (!d) return FUSE_ERR_INVALID_ARG;
  if (d->pos_encoding != FUSE_ROPE_ROTATE_HALF) return FUSE_ERR_UNSUPPORTED;
  if (d->dtype != FUSE_F32 && d->dtype != FUSE_BF16) return FUSE_ERR_UNSUPPORTED;
  if (d->hidden <= 0 || d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0)
    return FUSE_ERR_INVALID_ARG;
  if (d->n_q_heads % d->n_kv_heads != 0) return FUSE_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return FUSE_ERR_UNSUPPORTED;
  const int g = d->n_q_heads / d->n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return FUSE_ERR_UNSUPPORTED;
  if (d->hidden % 64 != 0) return FUSE_ERR_UNSUPPORTED;
  if (!(d->rope_base > 1.0) || !std::isfinite(d->rope_base)) return FUSE_ERR_INVALID_ARG;
  return FUSE_OK;
}

// theta_j / (2 pi) split into three floats (see rope_cos_sin).
RopeFreqs make_freqs(const fuse_layer_desc_t& d) {
  RopeFreqs f;
  std::memset(&f, 0, sizeof(f));
  const int h2 = d.head_dim / 2;
  const double two_pi = 6.283185307179586476925286766559;
  for (int j = 0; j < h2; ++j) {
    const double theta = std::pow(d.rope_base, -2.0 * j / (double)d.head_dim);
    const double turns = theta / two_pi;
    const float hi = (float)turns;
    const float mid = (float)(turns - (double)hi);
    const float lo = (float)(turns - (double)hi - (double)mid);
    f.hi[j] = hi;
    f.mid[j] = mid;
    f.lo[j] = lo;
  }
  return f;
}

struct ReqInfo {
  fuse_totals_t tot;   // extents implied by the offsets (max over requests)
  int n_req;
  bool sorted;         // row0 ascending, request row ranges disjoint
  int64_t n_qrows;     // sum of n_query: the packed query rows of the scorer
  int32_t max_query;   // max n_query
};

fuse_status_t check_reqs(const fuse_requests_t* r, ReqInfo* info, bool need_device = true) {
  if (!r || r->n_req < 0) return FUSE_ERR_INVALID_ARG;
  if (r->n_req > kMaxRequests) return FUSE_ERR_UNSUPPORTED;   // one grid row per request
  std::memset(info, 0, sizeof(*info));
  info->n_req = r->n_req;
  if (r->n_req == 0) return FUSE_OK;
  if (!r->h_req || (need_device && !r->d_req)) return FUSE_ERR_INVALID_ARG;
  fuse_totals_t& t = info->tot;
  info->sorted = true;
  for (int i = 0; i < r->n_req; ++i) {
    const fuse_request_t& q = r->h_req[i];
    if (i > 0 && q.row0 < r->h_req[i - 1].row0 + r->h_req[i - 1].n_ctx + r->h_req[i - 1].n_query)
      info->sorted = false;
    if (q.n_ctx < 0 || q.n_query < 0 || q.k < 0 || q.k > q.n_ctx || q.reserved != 0)
      return FUSE_ERR_INVALID_ARG;
    if (q.row0 < 0 || q.score0 < 0 || q.sel0 < 0 || q.out0 < 0) return FUSE_ERR_INVALID_ARG;
    const int64_t T = (int64_t)q.n_ctx + q.n_query;
    if (T > kMaxPosition) return FUSE_ERR_UNSUPPORTED;
    t.n_tok = std::max<int64_t>(t.n_tok, q.row0 + T);
    t.n_ctx = std::max<int64_t>(t.n_ctx, q.score0 + q.n_ctx);
    t.n_sel = std::max<int64_t>(t.n_sel, q.sel0 + q.k);
    t.n_out = std::max<int64_t>(t.n_out, q.out0 + q.k + q.n_query);
    t.max_ctx = std::max<int32_t>(t.max_ctx, q.n_ctx);
    t.max_tok = std::max<int32_t>(t.max_tok, (int32_t)T);
    info->n_qrows += q.n_query;
    info->max_query = std::max(info->max_query, q.n_query);
  }
  if (t.n_tok > INT32_MAX) return FUSE_ERR_UNSUPPORTED;
  return FUSE_OK;
}

fuse_status_t check_chunks(const fuse_layer_desc_t& d, const fuse_chunks_t* c, int64_t fused_rows,
                           int* max_len) {
  if (!c || c->n_chunks < 0) return FUSE_ERR_INVALID_ARG;
  *max_len = 0;
  if (c->kv_layout != FUSE_KV_CONTIGUOUS && c->kv_layout != FUSE_KV_PAGED)
    return FUSE_ERR_INVALID_ARG;
  if (c->kv_storage != FUSE_F32 && c->kv_storage != FUSE_BF16 && c->kv_storage != FUSE_U8_ASYM &&
      c->kv_storage != FUSE_U4_ASYM)
    return FUSE_ERR_INVALID_ARG;
  const bool paged = c->kv_layout == FUSE_KV_PAGED;
  const bool u8 = c->kv_storage == FUSE_U8_ASYM || c->kv_storage == FUSE_U4_ASYM;   // quantised
  if (paged && (c->block_size <= 0 || c->n_pool_blocks <= 0)) return FUSE_ERR_INVALID_ARG;
  if (c->n_chunks == 0) return FUSE_OK;
  if (!c->h_chunks || !c->d_chunks) return FUSE_ERR_INVALID_ARG;
  for (int i = 0; i < c->n_chunks; ++i) {
    const fuse_chunk_t& q = c->h_chunks[i];
    if (q.len < 0 || q.pos < 0 || q.dst_row < 0) return FUSE_ERR_INVALID_ARG;
    if ((int64_t)q.pos + q.len > kMaxPosition) return FUSE_ERR_UNSUPPORTED;
    if (q.dst_row + q.len > fused_rows) return FUSE_ERR_INVALID_ARG;
    *max_len = std::max(*max_len, q.len);
    if (q.len == 0) continue;
    if (!q.k || !q.v) return FUSE_ERR_INVALID_ARG;
    if (!aligned16(q.k) || !aligned16(q.v)) return FUSE_ERR_MISALIGNED;
    if (paged && !q.block_table) return FUSE_ERR_INVALID_ARG;
    if (u8) {
      if (!q.k_scale || !q.k_zero || !q.v_scale || !q.v_zero) return FUSE_ERR_INVALID_ARG;
      if (!aligned16(q.k_scale) || !aligned16(q.k_zero)) return FUSE_ERR_MISALIGNED;
      if ((reinterpret_cast<uintptr_t>(q.v_scale) | reinterpret_cast<uintptr_t>(q.v_zero)) & 1u)
        return FUSE_ERR_MISALIGNED;
    }
  }
  (void)d;
  return FUSE_OK;
}

// Workspace regions (each 256-byte aligned).
struct WsLayout {
  size_t partial, keys, map, rows, rope, q, hs, tiles;
  size_t mrows, mrope, mq, mhs, mstats, mnorm, qoff;   // query-aware scorer
  size_t krows, krope, kn;                             // key deviation
  size_t total;
};

WsLayout ws_layout(const fuse_layer_desc_t& d, const ReqInfo& info) {
  const fuse_totals_t& t = info.tot;
  const int n_req = info.n_req;
  const size_t nq = (size_t)info.n_qrows;
  WsLayout L;
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  const size_t es = elem_size(d.dtype);
  L.keys = take((size_t)t.n_ctx * sizeof(uint32_t));          // first: top-k needs only this
  L.partial = take((size_t)t.n_ctx * d.n_kv_heads * sizeof(float));
  L.map = take((size_t)t.n_tok * sizeof(int32_t));
  L.rows = take((size_t)t.n_out * sizeof(WorkRow));
  L.rope = take((size_t)t.n_out * (d.head_dim / 2) * sizeof(float2));
  L.q = take((size_t)t.n_out * d.n_q_heads * d.head_dim * es);
  L.hs = take((size_t)t.n_out * d.hidden * es);
  L.tiles = take(attention_tiles_bytes(t.n_out, n_req));
  L.mrows = take(nq * sizeof(WorkRow));
  L.mrope = take(nq * (d.head_dim / 2) * sizeof(float2));
  L.mq = take(nq * d.n_q_heads * d.head_dim * es);
  L.mhs = take(nq * d.hidden * es);
  L.mstats = take(nq * d.n_q_heads * (size_t)mass_key_tiles(t.max_ctx) * sizeof(float2));
  L.mnorm = take(nq * d.n_q_heads * sizeof(float2));
  L.qoff = take((size_t)n_req * sizeof(int32_t));
  L.krows = take((size_t)t.n_tok * sizeof(WorkRow));
  L.krope = take((size_t)t.n_tok * (d.head_dim / 2) * sizeof(float2));
  // the key deviation's fresh keys; the query-aware scorer uses the same
  // region for its split-K projection partials and, on the tensor-core path,
  // for its per-(token, KV head, 128-vector tile, half) mass
  const int g = d.n_q_heads / d.n_kv_heads;
  const size_t n_vt = ((size_t)info.max_query * g + 127) / 128;
  L.kn = take(std::max((size_t)t.n_tok * d.n_kv_heads * d.head_dim * es,
                       (size_t)t.n_ctx * d.n_kv_heads * n_vt * 2 * sizeof(float)));
  L.total = off;
  return L;
}

// Cosine partials per context token: one per pair of KV heads on the
// tensor-core path (the two heads of a tile are summed in its epilogue), one
// per KV head otherwise.
int score_parts(const fuse_layer_desc_t& d) {
  return tc_gemm_supported(d) ? d.n_kv_heads / 2 : d.n_kv_heads;
}

template <typename T> T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + off);
}

fuse_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? FUSE_OK : FUSE_ERR_CUDA; }

fuse_status_t check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return FUSE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return FUSE_ERR_MISALIGNED;
  if (ws_bytes < need) return FUSE_ERR_WORKSPACE;
  return FUSE_OK;
}

// ---- the steps (validated arguments) ------------------------------------

fuse_status_t do_stitch(const fuse_layer_desc_t& d, const fuse_chunks_t& c, int max_len, void* Kf,
                        void* Vf, void* ws, cudaStream_t s, int free_sms = -1) {
  if (c.n_chunks == 0 || max_len == 0) return FUSE_OK;
  const RopeFreqs f = make_freqs(d);
  return cuda_status(traced("stitch_rerotate", s, [&] {
    return launch_stitch(d, c, f, max_len, Kf, Vf, at<uint32_t>(ws, 0), s, free_sms);
  }));
}

// Chunks placed in ascending, non-overlapping fused rows (host table).
bool chunks_sorted(const fuse_chunks_t& c) {
  for (int i = 1; i < c.n_chunks; ++i)
    if (c.h_chunks[i].dst_row < c.h_chunks[i - 1].dst_row + c.h_chunks[i - 1].len) return false;
  return true;
}

fuse_status_t do_score(const fuse_layer_desc_t& d, const fuse_requests_t& r, const ReqInfo& info,
                       const void* H, const void* Wv, const void* Vf, float* score, void* ws,
                       cudaStream_t s, bool reduce = true, const fuse_chunks_t* v_chunks = nullptr) {
  const WsLayout L = ws_layout(d, info);
  if (info.tot.n_ctx == 0) return FUSE_OK;
  int32_t* map = at<int32_t>(ws, L.map);
  float* partial = at<float>(ws, L.partial);
  const bool tc = tc_gemm_supported(d);
  const bool need_map = !tc || !info.sorted;    // the tensor-core epilogue searches sorted tables
  cudaError_t e = cudaSuccess;
  if (need_map) {
    e = cudaMemsetAsync(map, 0xFF, (size_t)info.tot.n_tok * sizeof(int32_t), s);
    if (e == cudaSuccess)
      e = traced("score_map", s, [&] { return launch_build_score_map(r, info.tot.max_tok, map, s); });
  }
  if (e == cudaSuccess) {
    if (tc)
      e = traced("deviation_gemm_tc", s, [&] {
        return launch_deviation_partials_tc(d, info.tot.n_tok, H, Wv, Vf, need_map ? map : nullptr,
                                            r.d_req, r.n_req, partial, v_chunks,
                                            at<uint32_t>(ws, 0), s);
      });
    else
      e = traced("deviation_gemm_simt", s, [&] {
        return launch_deviation_partials_simt(d, info.tot.n_tok, H, Wv, Vf, map, partial,
                                              at<uint32_t>(ws, 0), s);
      });
  }
  if (e == cudaSuccess && reduce)
    e = traced("deviation_reduce", s, [&] {
      return launch_deviation_reduce(info.tot.n_ctx, score_parts(d), d.n_kv_heads, partial, score,
                                     s);
    });
  return cuda_status(e);
}

// score from the partials of do_score(..., reduce = false), then top-k, one launch
fuse_status_t do_reduce_topk(const fuse_layer_desc_t& d, const fuse_requests_t& r,
                             const ReqInfo& info, float* score, int32_t* idx, void* ws,
                             cudaStream_t s) {
  const WsLayout L = ws_layout(d, info);
  if (info.tot.n_ctx == 0) return FUSE_OK;
  return cuda_status(traced("reduce_topk", s, [&] {
    return launch_reduce_topk(r, info.tot.max_ctx, at<float>(ws, L.partial), score_parts(d),
                              d.n_kv_heads, score, idx, at<uint32_t>(ws, L.keys),
                              at<uint32_t>(ws, 0), s);
  }));
}

fuse_status_t do_recompute(const fuse_layer_desc_t& d, const fuse_requests_t& r,
                           const ReqInfo& info, const void* H, const void* Wq, const void* Wk,
                           const void* Wv, const int32_t* idx, void* Kf, void* Vf, void* O,
                           void* ws, cudaStream_t s) {
  const WsLayout L = ws_layout(d, info);
  const int64_t R = info.tot.n_out;
  if (R == 0) return FUSE_OK;
  int max_rows = 0;
  for (int i = 0; i < r.n_req; ++i)
    max_rows = std::max(max_rows, r.h_req[i].k + r.h_req[i].n_query);
  WorkRow* rows = at<WorkRow>(ws, L.rows);
  float2* rope = at<float2>(ws, L.rope);
  void* Q = at<void>(ws, L.q);
  uint32_t* err = at<uint32_t>(ws, 0);
  const RopeFreqs f = make_freqs(d);
  const bool tc_gemm = tc_gemm_supported(d);
  const bool tc_attn = tc_attention_supported(d);
  cudaError_t e;
  if (tc_gemm) {
    e = traced("prepare_rows", s, [&] {
      return launch_prepare_rows(r, max_rows, idx, f, d.head_dim, H, d.hidden, rows, rope, R,
                                 at<void>(ws, L.hs), tc_attn ? attention_rtile(d) : 128,
                                 tc_attn ? at<void>(ws, L.tiles) : nullptr, err, s);
    });
    if (e != cudaSuccess) return FUSE_ERR_CUDA;
    e = traced("qkv_gemm_tc", s, [&] {
      return launch_project_recompute_tc(d, R, rows, rope, H, Wq, Wk, Wv, Q, Kf, Vf,
                                         at<void>(ws, L.hs), err, s);
    });
  } else {
    e = traced("sel_rows", s, [&] {
      return launch_build_sel_rows(r, max_rows, idx, f, d.head_dim, rows, rope, R, err, s);
    });
    if (e != cudaSuccess) return FUSE_ERR_CUDA;
    e = traced("qkv_gemm_simt", s, [&] {
      return launch_project_recompute_simt(d, R, rows, rope, H, Wq, Wk, Wv, Q, Kf, Vf, err, s);
    });
  }
  if (e != cudaSuccess) return FUSE_ERR_CUDA;
  if (tc_attn)
    e = traced("attention_tc", s, [&] {
      return launch_attention_tc(d, r, R, info.tot.n_tok, rows, idx, Q, Kf, Vf, O,
                                 at<void>(ws, L.tiles), /*tiles_ready=*/tc_gemm, err, s);
    });
  else
    e = traced("attention_simt", s, [&] { return launch_attention_simt(d, R, rows, Q, Kf, Vf, O, s); });
  return cuda_status(e);
}

// Query-aware attention mass (QCFuse Eqs. 9-10, 20): the query rows packed,
// their Q projected (Q heads only), then the scoring launches.
fuse_status_t do_mass(const fuse_layer_desc_t& d, const fuse_requests_t& r, const ReqInfo& info,
                      const void* H, const void* Wq, const void* Kf, float* score, int accumulate,
                      void* ws, cudaStream_t s) {
  const WsLayout L = ws_layout(d, info);
  if (info.tot.n_ctx == 0 || info.tot.max_ctx == 0) return FUSE_OK;
  const int64_t nq = info.n_qrows;
  WorkRow* rows = at<WorkRow>(ws, L.mrows);
  float2* rope = at<float2>(ws, L.mrope);
  void* Q = at<void>(ws, L.mq);
  int32_t* qoff = at<int32_t>(ws, L.qoff);
  uint32_t* err = at<uint32_t>(ws, 0);
  const bool tc = tc_gemm_supported(d);
  const RopeFreqs f = make_freqs(d);
  cudaError_t e = traced("query_rows", s, [&] {
    return launch_query_rows(r, info.max_query, f, d.head_dim, H, d.hidden, rows, rope, nq,
                             tc ? at<void>(ws, L.mhs) : nullptr, qoff, err, s);
  });
  if (e == cudaSuccess && nq > 0) {
    if (tc)
      e = traced("query_gemm_tc", s, [&] {
        // the split-K partials use the key deviation's fresh-key region
        const size_t per_split = (size_t)nq * d.n_q_heads * d.head_dim * sizeof(float);
        const size_t room = L.total - L.kn;
        const int max_splits = (int)std::min<size_t>(8, room / std::max<size_t>(per_split, 1));
        if (max_splits >= 1 && qproj_tc_supported(d, nq))
          return launch_qproj_tc(d, nq, rope, Wq, at<void>(ws, L.mhs), Q, at<float>(ws, L.kn),
                                 max_splits, err, s);
        return launch_project_query_tc(d, nq, rope, Wq, Q, at<void>(ws, L.mhs), err, s,
                                       at<float>(ws, L.kn), max_splits);
      });
    else
      e = traced("query_gemm_simt", s, [&] {
        return launch_project_query_simt(d, nq, rows, rope, H, Wq, Q, err, s);
      });
  }
  if (e == cudaSuccess) {
    if (mass_tc_supported(d)) {
      const int n_chunks = mass_tc_chunks(d, r, info.tot.max_ctx, info.max_query);
      e = traced("attention_mass_tc", s, [&] {
        return launch_attention_mass_tc(d, r, info.tot.max_ctx, info.max_query, nq,
                                        info.tot.n_tok, qoff, Q, Kf, at<float2>(ws, L.mstats),
                                        at<float>(ws, L.kn), n_chunks, score, accumulate, err,
                                        s);
      });
    } else {
      e = traced("attention_mass", s, [&] {
        return launch_attention_mass(d, r, info.tot.max_ctx, nq, rows, qoff, Q, Kf,
                                     at<float2>(ws, L.mstats), at<float2>(ws, L.mnorm),
                                     at<float>(ws, L.partial), score, accumulate, s);
      });
    }
  }
  return cuda_status(e);
}

// Key deviation, one layer's term (KVBoost Alg. 2 step 2): fresh keys of
// every packed row at its request position through the query-state
// projection with the key heads in place of the query heads, then the
// per-token cosines against the stitched keys.
fuse_status_t do_key_deviation(const fuse_layer_desc_t& d, const fuse_requests_t& r,
                               const ReqInfo& info, const void* H, const void* Wk, const void* Kf,
                               float weight, int accumulate, float* score, void* ws,
                               cudaStream_t s) {
  const WsLayout L = ws_layout(d, info);
  if (info.tot.n_ctx == 0 || info.tot.max_ctx == 0) return FUSE_OK;
  const int64_t n = info.tot.n_tok;
  WorkRow* rows = at<WorkRow>(ws, L.krows);
  float2* rope = at<float2>(ws, L.krope);
  void* Kn = at<void>(ws, L.kn);
  uint32_t* err = at<uint32_t>(ws, 0);
  fuse_layer_desc_t dk = d;
  dk.n_q_heads = d.n_kv_heads;
  const RopeFreqs f = make_freqs(d);
  cudaError_t e = traced("key_rows", s, [&] {
    return launch_key_rows(r, info.tot.max_tok, f, d.head_dim, n, rows, rope, s);
  });
  if (e == cudaSuccess) {
    if (tc_gemm_supported(dk))
      e = traced("key_gemm_tc", s, [&] {
        return launch_project_query_tc(dk, n, rope, Wk, Kn, H, err, s);
      });
    else
      e = traced("key_gemm_simt", s, [&] {
        return launch_project_query_simt(dk, n, rows, rope, H, Wk, Kn, err, s);
      });
  }
  if (e == cudaSuccess)
    e = traced("key_cosine", s, [&] {
      return launch_key_cosine(d, r, info.tot.max_ctx, Kn, Kf, weight, accumulate, score, s);
    });
  return cuda_status(e);
}

struct LayerArgs {
  const fuse_chunks_t* chunks;
  const void* H;
  const void* Wq;
  const void* Wk;
  const void* Wv;
  void* Kf;
  void* Vf;
  void* O;
};

// Validation of one layer of fuse_layer_step / fuse_stack_step.
fuse_status_t check_layer(const fuse_layer_desc_t& d, const ReqInfo& info, const LayerArgs& a,
                          bool scoring, const int32_t* idx, const float* score, void* ws,
                          size_t ws_bytes, int* max_len) {
  fuse_status_t st = check_chunks(d, a.chunks, info.tot.n_tok, max_len);
  if (st != FUSE_OK) return st;
  if (info.tot.n_out > 0 && (!a.H || !a.Wq || !a.Wk || !a.Wv || !a.Kf || !a.Vf || !a.O))
    return FUSE_ERR_INVALID_ARG;
  if (info.tot.n_sel > 0 && !idx) return FUSE_ERR_INVALID_ARG;
  if (scoring && info.tot.n_ctx > 0 && !score) return FUSE_ERR_INVALID_ARG;
  if (!aligned16(a.H) || !aligned16(a.Wq) || !aligned16(a.Wk) || !aligned16(a.Wv) ||
      !aligned16(a.Kf) || !aligned16(a.Vf) || !aligned16(a.O) || !aligned16(score))
    return FUSE_ERR_MISALIGNED;
  return check_ws(ws, ws_bytes, ws_layout(d, info).total);
}

// Deviation scores and the top-k selection of one (scoring) layer.
fuse_status_t do_score_select(const fuse_layer_desc_t& d, const fuse_requests_t& r,
                              const ReqInfo& info, const void* H, const void* Wv, const void* Vf,
                              float* score, int32_t* idx, void* ws, cudaStream_t s) {
  fuse_status_t st = do_score(d, r, info, H, Wv, Vf, score, ws, s, /*reduce=*/false);
  if (st != FUSE_OK) return st;
  return do_reduce_topk(d, r, info, score, idx, ws, s);
}

// Stitch and score/select of one layer.  On the tensor-core path with chunk
// caches of the layer's type placed in order, the deviation GEMM reads the
// cached V rows from the chunks themselves and the stitch runs beside it (it
// waits for the GEMM only at its end); otherwise in sequence.
fuse_status_t do_stitch_score_select(const fuse_layer_desc_t& d, const fuse_chunks_t& c,
                                     int max_len, const fuse_requests_t& r, const ReqInfo& info,
                                     const void* H, const void* Wv, void* Kf, void* Vf,
                                     float* score, int32_t* idx, void* ws, cudaStream_t s) {
  const bool together = tc_gemm_supported(d) && info.tot.n_ctx > 0 && c.n_chunks > 0 &&
                        max_len > 0 && stitch_streamed(d, c) && chunks_sorted(c);
  if (!together) {
    fuse_status_t st = do_stitch(d, c, max_len, Kf, Vf, ws, s);
    if (st != FUSE_OK) return st;
    return do_score_select(d, r, info, H, Wv, Vf, score, idx, ws, s);
  }
  fuse_status_t st = do_score(d, r, info, H, Wv, Vf, score, ws, s, /*reduce=*/false, &c);
  if (st != FUSE_OK) return st;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int free_sms = std::max(0, sms - deviation_tc_ctas(d, info.tot.n_tok));
  st = do_stitch(d, c, max_len, Kf, Vf, ws, s, free_sms);
  if (st != FUSE_OK) return st;
  return do_reduce_topk(d, r, info, score, idx, ws, s);
}

// Schedule of a streamed stack (QCFuse Figure 9; PCR layer-wise overlapping).
// Layers run in the order score layer, then the others by index.  The
// copies are issued as early as the slots allow: a layer's copies follow the
// previous user of its slot (in that order) once that user's release has
// been issued, and copies stay in layer order.  Because a slot's next copy is
// issued only after its current user's release, every wait binds to the
// record it is meant for (a CUDA wait takes the event's latest record).
constexpr int kMaxSlots = 64;

fuse_status_t stack_plan(int n_layers, int score_layer, const int32_t* slot_of_layer, int n_slots,
                         std::vector<fuse_pipeline_op_t>& ops) {
  if (n_layers <= 0 || score_layer < 0 || score_layer >= n_layers || n_slots <= 0 ||
      n_slots > kMaxSlots || !slot_of_layer)
    return FUSE_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (slot_of_layer[l] < 0 || slot_of_layer[l] >= n_slots) return FUSE_ERR_INVALID_ARG;
  std::vector<int> order;
  order.push_back(score_layer);
  for (int l = 0; l < n_layers; ++l)
    if (l != score_layer) order.push_back(l);
  std::vector<int> last_user(n_slots, -1);     // order index of the slot's latest copy
  std::vector<char> released(n_layers, 0);     // order index -> release issued
  ops.clear();
  auto op = [&](int kind, int l) { ops.push_back(fuse_pipeline_op_t{kind, l, slot_of_layer[l]}); };
  int next_copy = 0;
  auto issue_copies = [&] {
    while (next_copy < n_layers) {
      const int l = order[next_copy];
      const int sl = slot_of_layer[l];
      const int prev = last_user[sl];
      if (prev >= 0 && !released[prev]) break;
      if (prev >= 0) op(FUSE_OP_WAIT_FREE, l);
      op(FUSE_OP_COPY, l);
      op(FUSE_OP_MARK_READY, l);
      last_user[sl] = next_copy;
      ++next_copy;
    }
  };
  issue_copies();
  for (int i = 0; i < n_layers; ++i) {
    const int l = order[i];
    op(FUSE_OP_WAIT_READY, l);
    op(FUSE_OP_COMPUTE, l);
    op(FUSE_OP_MARK_FREE, l);
    released[i] = 1;
    issue_copies();
  }
  return FUSE_OK;
}

}  // namespace
}  // namespace fusekv

using namespace fusekv;

extern "C" {

int64_t fuse_k_from_ratio(double ratio, int64_t n_ctx) {
  if (n_ctx <= 0 || !(ratio > 0.0)) return 0;
  const double v = std::floor(ratio * (double)n_ctx + 1e-9);
  if (v >= (double)n_ctx) return n_ctx;
  return (int64_t)v;
}

fuse_status_t fuse_plan_requests(int32_t n_req, const int32_t* n_ctx, const int32_t* n_query,
                                 double ratio, fuse_request_t* out, fuse_totals_t* totals) {
  if (n_req < 0 || (n_req > 0 && (!n_ctx || !n_query || !out))) return FUSE_ERR_INVALID_ARG;
  fuse_totals_t t;
  std::memset(&t, 0, sizeof(t));
  for (int i = 0; i < n_req; ++i) {
    if (n_ctx[i] < 0 || n_query[i] < 0) return FUSE_ERR_INVALID_ARG;
    fuse_request_t q;
    std::memset(&q, 0, sizeof(q));
    q.row0 = t.n_tok;
    q.score0 = t.n_ctx;
    q.sel0 = t.n_sel;
    q.out0 = t.n_out;
    q.n_ctx = n_ctx[i];
    q.n_query = n_query[i];
    q.k = (int32_t)fuse_k_from_ratio(ratio, n_ctx[i]);
    out[i] = q;
    t.n_tok += (int64_t)n_ctx[i] + n_query[i];
    t.n_ctx += n_ctx[i];
    t.n_sel += q.k;
    t.n_out += (int64_t)q.k + n_query[i];
    t.max_ctx = std::max(t.max_ctx, n_ctx[i]);
    t.max_tok = std::max<int32_t>(t.max_tok, n_ctx[i] + n_query[i]);
  }
  if (t.n_tok > INT32_MAX) return FUSE_ERR_INVALID_ARG;
  if (totals) *totals = t;
  return FUSE_OK;
}

fuse_status_t fuse_workspace_size(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                  size_t* bytes) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  if (!bytes) return FUSE_ERR_INVALID_ARG;
  ReqInfo info;
  st = check_reqs(reqs, &info, /*need_device=*/false);
  if (st != FUSE_OK) return st;
  *bytes = ws_layout(*desc, info).total;
  return FUSE_OK;
}

fuse_status_t fuse_workspace_reset(void* ws, size_t ws_bytes, fuse_stream_t stream) {
  if (!ws || ws_bytes < sizeof(WsHeader)) return FUSE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
}

fuse_status_t fuse_selftest_wait_timeout(void* ws, size_t ws_bytes, fuse_stream_t stream) {
  const fuse_status_t st = check_ws(ws, ws_bytes, sizeof(WsHeader));
  if (st != FUSE_OK) return st;
  return cuda_status(launch_selftest_wait(at<uint32_t>(ws, 0), (cudaStream_t)stream));
}

fuse_status_t fuse_stitch_rerotate(const fuse_layer_desc_t* desc, const fuse_chunks_t* chunks,
                                   void* Kf, void* Vf, int64_t fused_rows, void* ws,
                                   size_t ws_bytes, fuse_stream_t stream) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  int max_len;
  st = check_chunks(*desc, chunks, fused_rows, &max_len);
  if (st != FUSE_OK) return st;
  if (fused_rows < 0) return FUSE_ERR_INVALID_ARG;
  if (fused_rows > 0 && (!Kf || !Vf)) return FUSE_ERR_INVALID_ARG;
  if (!aligned16(Kf) || !aligned16(Vf)) return FUSE_ERR_MISALIGNED;
  st = check_ws(ws, ws_bytes, sizeof(WsHeader));
  if (st != FUSE_OK) return st;
  return do_stitch(*desc, *chunks, max_len, Kf, Vf, ws, (cudaStream_t)stream);
}

fuse_status_t fuse_score_deviation(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                   const void* H, const void* Wv, const void* Vf, float* score,
                                   void* ws, size_t ws_bytes, fuse_stream_t stream) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  ReqInfo info;
  st = check_reqs(reqs, &info);
  if (st != FUSE_OK) return st;
  if (info.tot.n_ctx > 0 && (!H || !Wv || !Vf || !score)) return FUSE_ERR_INVALID_ARG;
  if (!aligned16(H) || !aligned16(Wv) || !aligned16(Vf) || !aligned16(score))
    return FUSE_ERR_MISALIGNED;
  st = check_ws(ws, ws_bytes, ws_layout(*desc, info).total);
  if (st != FUSE_OK) return st;
  return do_score(*desc, *reqs, info, H, Wv, Vf, score, ws, (cudaStream_t)stream);
}

fuse_status_t fuse_score_attention_mass(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                        const void* H, const void* Wq, const void* Kf,
                                        int32_t accumulate, float* score, void* ws,
                                        size_t ws_bytes, fuse_stream_t stream) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  ReqInfo info;
  st = check_reqs(reqs, &info);
  if (st != FUSE_OK) return st;
  if (info.n_qrows > INT32_MAX) return FUSE_ERR_UNSUPPORTED;
  if (info.tot.n_ctx > 0 && (!H || !Wq || !Kf || !score)) return FUSE_ERR_INVALID_ARG;
  if (!aligned16(H) || !aligned16(Wq) || !aligned16(Kf) || !aligned16(score))
    return FUSE_ERR_MISALIGNED;
  st = check_ws(ws, ws_bytes, ws_layout(*desc, info).total);
  if (st != FUSE_OK) return st;
  return do_mass(*desc, *reqs, info, H, Wq, Kf, score, accumulate, ws, (cudaStream_t)stream);
}

fuse_status_t fuse_score_key_deviation(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                      const void* H, const void* Wk, const void* Kf, float weight,
                                      int32_t accumulate, float* score, void* ws, size_t ws_bytes,
                                      fuse_stream_t stream) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  ReqInfo info;
  st = check_reqs(reqs, &info);
  if (st != FUSE_OK) return st;
  if (!std::isfinite(weight)) return FUSE_ERR_INVALID_ARG;
  if (info.tot.n_ctx > 0 && (!H || !Wk || !Kf || !score)) return FUSE_ERR_INVALID_ARG;
  if (!aligned16(H) || !aligned16(Wk) || !aligned16(Kf) || !aligned16(score))
    return FUSE_ERR_MISALIGNED;
  st = check_ws(ws, ws_bytes, ws_layout(*desc, info).total);
  if (st != FUSE_OK) return st;
  return do_key_deviation(*desc, *reqs, info, H, Wk, Kf, weight, accumulate, score, ws,
                          (cudaStream_t)stream);
}

fuse_status_t fuse_select_topk(const fuse_requests_t* reqs, const float* score, int32_t* idx,
                               void* ws, size_t ws_bytes, fuse_stream_t stream) {
  ReqInfo info;
  fuse_status_t st = check_reqs(reqs, &info);
  if (st != FUSE_OK) return st;
  if (info.tot.n_sel > 0 && (!score || !idx)) return FUSE_ERR_INVALID_ARG;
  // the top-k needs only the header and the key buffer (N_total words), the
  // first region of every workspace layout
  const size_t keys_at = sizeof(WsHeader);
  st = check_ws(ws, ws_bytes, keys_at + (size_t)info.tot.n_ctx * sizeof(uint32_t));
  if (st != FUSE_OK) return st;
  if (info.tot.n_sel == 0) return FUSE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  return cuda_status(traced("topk", s, [&] {
    return launch_topk(*reqs, info.tot.max_ctx, score, idx, at<uint32_t>(ws, keys_at),
                       at<uint32_t>(ws, 0), s);
  }));
}

fuse_status_t fuse_recompute_selected(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                      const void* H, const void* Wq, const void* Wk,
                                      const void* Wv, const int32_t* idx, void* Kf, void* Vf,
                                      void* O, void* ws, size_t ws_bytes, fuse_stream_t stream) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  ReqInfo info;
  st = check_reqs(reqs, &info);
  if (st != FUSE_OK) return st;
  if (info.tot.n_out > 0 && (!H || !Wq || !Wk || !Wv || !Kf || !Vf || !O))
    return FUSE_ERR_INVALID_ARG;
  if (info.tot.n_sel > 0 && !idx) return FUSE_ERR_INVALID_ARG;
  if (!aligned16(H) || !aligned16(Wq) || !aligned16(Wk) || !aligned16(Wv) || !aligned16(Kf) ||
      !aligned16(Vf) || !aligned16(O))
    return FUSE_ERR_MISALIGNED;
  st = check_ws(ws, ws_bytes, ws_layout(*desc, info).total);
  if (st != FUSE_OK) return st;
  return do_recompute(*desc, *reqs, info, H, Wq, Wk, Wv, idx, Kf, Vf, O, ws, (cudaStream_t)stream);
}

fuse_status_t fuse_layer_step(const fuse_layer_desc_t* desc, const fuse_chunks_t* chunks,
                              const fuse_requests_t* reqs, const void* H, const void* Wq,
                              const void* Wk, const void* Wv, int32_t score_this_layer,
                              int32_t* idx, void* Kf, void* Vf, void* O, float* score, void* ws,
                              size_t ws_bytes, fuse_stream_t stream) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  ReqInfo info;
  st = check_reqs(reqs, &info);
  if (st != FUSE_OK) return st;
  LayerArgs la{chunks, H, Wq, Wk, Wv, Kf, Vf, O};
  int max_len;
  st = check_layer(*desc, info, la, score_this_layer != 0, idx, score, ws, ws_bytes, &max_len);
  if (st != FUSE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (score_this_layer)
    st = do_stitch_score_select(*desc, *chunks, max_len, *reqs, info, H, Wv, Kf, Vf, score, idx, ws, s);
  else
    st = do_stitch(*desc, *chunks, max_len, Kf, Vf, ws, s);
  if (st != FUSE_OK) return st;
  return do_recompute(*desc, *reqs, info, H, Wq, Wk, Wv, idx, Kf, Vf, O, ws, s);
}

fuse_status_t fuse_stack_step(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                              int32_t n_layers, int32_t score_layer, const fuse_layer_io_t* layers,
                              int32_t* idx, float* score, void* ws, size_t ws_bytes,
                              fuse_stream_t stream) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  ReqInfo info;
  st = check_reqs(reqs, &info);
  if (st != FUSE_OK) return st;
  if (n_layers <= 0 || !layers || score_layer < 0 || score_layer >= n_layers)
    return FUSE_ERR_INVALID_ARG;
  std::vector<int> max_len(n_layers);
  for (int l = 0; l < n_layers; ++l) {
    const fuse_layer_io_t& L = layers[l];
    LayerArgs la{L.chunks, L.H, L.Wq, L.Wk, L.Wv, L.Kf, L.Vf, L.O};
    st = check_layer(*desc, info, la, l == score_layer, idx, score, ws, ws_bytes, &max_len[l]);
    if (st != FUSE_OK) return st;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const fuse_layer_io_t& S = layers[score_layer];
  st = do_stitch_score_select(*desc, *S.chunks, max_len[score_layer], *reqs, info, S.H, S.Wv, S.Kf,
                              S.Vf, score, idx, ws, s);
  if (st != FUSE_OK) return st;
  for (int l = 0; l < n_layers; ++l) {
    const fuse_layer_io_t& L = layers[l];
    if (l != score_layer) {
      st = do_stitch(*desc, *L.chunks, max_len[l], L.Kf, L.Vf, ws, s);
      if (st != FUSE_OK) return st;
    }
    st = do_recompute(*desc, *reqs, info, L.H, L.Wq, L.Wk, L.Wv, idx, L.Kf, L.Vf, L.O, ws, s);
    if (st != FUSE_OK) return st;
  }
  return FUSE_OK;
}

struct fuse_graph_st {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

fuse_status_t fuse_stack_graph_create(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                      int32_t n_layers, int32_t score_layer,
                                      const fuse_layer_io_t* layers, int32_t* idx, float* score,
                                      void* ws, size_t ws_bytes, fuse_stream_t stream,
                                      fuse_graph_t* out) {
  if (!out) return FUSE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!stream) return FUSE_ERR_INVALID_ARG;     // the legacy stream cannot be captured
  cudaStream_t s = (cudaStream_t)stream;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return FUSE_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return FUSE_ERR_INVALID_ARG;
  // relaxed mode: the once-per-device set-up of a first call (shared-memory
  // limits, occupancy queries) is not a stream operation and may run inside
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) return FUSE_ERR_CUDA;
  const fuse_status_t st =
      fuse_stack_step(desc, reqs, n_layers, score_layer, layers, idx, score, ws, ws_bytes, stream);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(s, &g);
  if (st != FUSE_OK || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return st != FUSE_OK ? st : FUSE_ERR_CUDA;
  }
  cudaGraphExec_t x = nullptr;
  if (cudaGraphInstantiate(&x, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return FUSE_ERR_CUDA;
  }
  fuse_graph_st* h = new (std::nothrow) fuse_graph_st{g, x};
  if (!h) {
    cudaGraphExecDestroy(x);
    cudaGraphDestroy(g);
    return FUSE_ERR_INVALID_ARG;
  }
  *out = h;
  return FUSE_OK;
}

fuse_status_t fuse_graph_launch(fuse_graph_t graph, fuse_stream_t stream) {
  if (!graph) return FUSE_ERR_INVALID_ARG;
  return cuda_status(cudaGraphLaunch(graph->exec, (cudaStream_t)stream));
}

void fuse_graph_destroy(fuse_graph_t graph) {
  if (!graph) return;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
}

fuse_status_t fuse_stack_pipeline_plan(int32_t n_layers, int32_t score_layer,
                                       const int32_t* slot_of_layer, int32_t n_slots,
                                       fuse_pipeline_op_t* ops, int32_t max_ops, int32_t* n_ops) {
  if (!n_ops || max_ops < 0 || (max_ops > 0 && !ops)) return FUSE_ERR_INVALID_ARG;
  std::vector<fuse_pipeline_op_t> plan;
  const fuse_status_t st = stack_plan(n_layers, score_layer, slot_of_layer, n_slots, plan);
  if (st != FUSE_OK) return st;
  *n_ops = (int32_t)plan.size();
  if ((int64_t)plan.size() > max_ops) return FUSE_ERR_WORKSPACE;
  std::copy(plan.begin(), plan.end(), ops);
  return FUSE_OK;
}

fuse_status_t fuse_stack_step_streamed(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                       int32_t n_layers, int32_t score_layer,
                                       const fuse_layer_io_t* layers,
                                       const fuse_layer_upload_t* uploads, int32_t n_slots,
                                       fuse_stream_t copy_stream, int32_t* idx, float* score,
                                       void* ws, size_t ws_bytes, fuse_stream_t stream) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  ReqInfo info;
  st = check_reqs(reqs, &info);
  if (st != FUSE_OK) return st;
  if (n_layers <= 0 || !layers || !uploads || score_layer < 0 || score_layer >= n_layers)
    return FUSE_ERR_INVALID_ARG;
  std::vector<int> max_len(n_layers);
  std::vector<int32_t> slot_of(n_layers);
  for (int l = 0; l < n_layers; ++l) {
    const fuse_layer_io_t& L = layers[l];
    LayerArgs la{L.chunks, L.H, L.Wq, L.Wk, L.Wv, L.Kf, L.Vf, L.O};
    st = check_layer(*desc, info, la, l == score_layer, idx, score, ws, ws_bytes, &max_len[l]);
    if (st != FUSE_OK) return st;
    const fuse_layer_upload_t& U = uploads[l];
    if (U.n_copies < 0 || (U.n_copies > 0 && !U.copies)) return FUSE_ERR_INVALID_ARG;
    for (int c = 0; c < U.n_copies; ++c)
      if (U.copies[c].bytes > 0 && (!U.copies[c].dst || !U.copies[c].src))
        return FUSE_ERR_INVALID_ARG;
    slot_of[l] = U.slot;
  }
  std::vector<fuse_pipeline_op_t> plan;
  st = stack_plan(n_layers, score_layer, slot_of.data(), n_slots, plan);
  if (st != FUSE_OK) return st;

  cudaStream_t s = (cudaStream_t)stream, cs = (cudaStream_t)copy_stream;
  std::vector<cudaEvent_t> ready(n_slots, nullptr), freed(n_slots, nullptr);
  cudaEvent_t entry = nullptr;
  cudaError_t e = cudaEventCreateWithFlags(&entry, cudaEventDisableTiming);
  for (int i = 0; i < n_slots && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&ready[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&freed[i], cudaEventDisableTiming);
  }
  // every upload follows the work enqueued on `stream` before this call: a
  // slot's buffers may still be read by an earlier call's kernels
  if (e == cudaSuccess) e = cudaEventRecord(entry, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, entry, 0);
  st = cuda_status(e);
  for (size_t i = 0; i < plan.size() && st == FUSE_OK; ++i) {
    const fuse_pipeline_op_t& o = plan[i];
    const fuse_layer_io_t& L = layers[o.layer];
    switch (o.kind) {
      case FUSE_OP_WAIT_FREE:
        st = cuda_status(cudaStreamWaitEvent(cs, freed[o.slot], 0));
        break;
      case FUSE_OP_COPY: {
        const fuse_layer_upload_t& U = uploads[o.layer];
        for (int c = 0; c < U.n_copies && st == FUSE_OK; ++c)
          if (U.copies[c].bytes > 0)
            st = cuda_status(cudaMemcpyAsync(U.copies[c].dst, U.copies[c].src, U.copies[c].bytes,
                                             cudaMemcpyDefault, cs));
        break;
      }
      case FUSE_OP_MARK_READY:
        st = cuda_status(cudaEventRecord(ready[o.slot], cs));
        break;
      case FUSE_OP_WAIT_READY:
        st = cuda_status(cudaStreamWaitEvent(s, ready[o.slot], 0));
        break;
      case FUSE_OP_COMPUTE:
        if (o.layer == score_layer)
          st = do_stitch_score_select(*desc, *L.chunks, max_len[o.layer], *reqs, info, L.H, L.Wv,
                                      L.Kf, L.Vf, score, idx, ws, s);
        else
          st = do_stitch(*desc, *L.chunks, max_len[o.layer], L.Kf, L.Vf, ws, s);
        if (st == FUSE_OK)
          st = do_recompute(*desc, *reqs, info, L.H, L.Wq, L.Wk, L.Wv, idx, L.Kf, L.Vf, L.O, ws, s);
        break;
      case FUSE_OP_MARK_FREE:
        st = cuda_status(cudaEventRecord(freed[o.slot], s));
        break;
      default:
        st = FUSE_ERR_INVALID_ARG;
    }
  }
  // destroying an event with work still pending is allowed: it is released
  // once that work completes
  if (entry) cudaEventDestroy(entry);
  for (int i = 0; i < n_slots; ++i) {
    if (ready[i]) cudaEventDestroy(ready[i]);
    if (freed[i]) cudaEventDestroy(freed[i]);
  }
  return st;
}

fuse_status_t fuse_pic_precompute(const fuse_layer_desc_t* desc, const fuse_chunks_t* chunks,
                                  const void* H_clean, const void* Wk, const void* Wv, void* ws,
                                  size_t ws_bytes, fuse_stream_t stream) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  if (!chunks) return FUSE_ERR_INVALID_ARG;
  if (chunks->kv_layout != FUSE_KV_CONTIGUOUS || chunks->kv_storage != desc->dtype)
    return FUSE_ERR_UNSUPPORTED;
  int max_len;
  st = check_chunks(*desc, chunks, INT64_MAX / 2, &max_len);
  if (st != FUSE_OK) return st;
  if (chunks->n_chunks > 0 && (!H_clean || !Wk || !Wv)) return FUSE_ERR_INVALID_ARG;
  if (!aligned16(H_clean) || !aligned16(Wk) || !aligned16(Wv)) return FUSE_ERR_MISALIGNED;
  st = check_ws(ws, ws_bytes, sizeof(WsHeader));
  if (st != FUSE_OK) return st;
  if (chunks->n_chunks == 0 || max_len == 0) return FUSE_OK;
  const RopeFreqs f = make_freqs(*desc);
  cudaStream_t s = (cudaStream_t)stream;
  return cuda_status(traced("pic_precompute", s, [&] {
    return launch_project_pic(*desc, chunks->n_chunks, max_len, f, H_clean, Wk, Wv,
                              chunks->d_chunks, at<uint32_t>(ws, 0), s);
  }));
}

fuse_status_t fuse_kivi_quantize(const fuse_layer_desc_t* desc, const fuse_chunks_t* src,
                                 const fuse_chunks_t* dst, fuse_stream_t stream) {
  fuse_status_t st = check_desc(desc);
  if (st != FUSE_OK) return st;
  if (!src || !dst) return FUSE_ERR_INVALID_ARG;
  if (src->kv_layout != FUSE_KV_CONTIGUOUS || dst->kv_layout != FUSE_KV_CONTIGUOUS ||
      src->kv_storage != desc->dtype ||
      (dst->kv_storage != FUSE_U8_ASYM && dst->kv_storage != FUSE_U4_ASYM))
    return FUSE_ERR_UNSUPPORTED;
  if (src->n_chunks != dst->n_chunks) return FUSE_ERR_INVALID_ARG;
  int max_len = 0, max_len_dst = 0;
  st = check_chunks(*desc, src, INT64_MAX / 2, &max_len);
  if (st != FUSE_OK) return st;
  st = check_chunks(*desc, dst, INT64_MAX / 2, &max_len_dst);
  if (st != FUSE_OK) return st;
  for (int i = 0; i < src->n_chunks; ++i)
    if (src->h_chunks[i].len != dst->h_chunks[i].len) return FUSE_ERR_INVALID_ARG;
  if (src->n_chunks == 0 || max_len == 0) return FUSE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  return cuda_status(traced("kivi_quantize", s, [&] {
    return launch_kivi_quantize(*desc, *src, *dst, max_len, s);
  }));
}

fuse_status_t fuse_check_errors(void* ws, fuse_stream_t stream, uint32_t* detail) {
  if (!ws) return FUSE_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return FUSE_ERR_CUDA;
  uint32_t h[2] = {0, 0};
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FUSE_ERR_CUDA;
  if (detail) *detail = h[1];
  if (h[0] != 0 && cudaMemset(ws, 0, sizeof(h)) != cudaSuccess) return FUSE_ERR_CUDA;
  return (fuse_status_t)h[0];
}

const char* fuse_status_string(fuse_status_t s) {
  switch (s) {
    case FUSE_OK: return "ok";
    case FUSE_ERR_INVALID_ARG: return "invalid argument";
    case FUSE_ERR_MISALIGNED: return "pointer or stride not aligned";
    case FUSE_ERR_UNSUPPORTED: return "unsupported configuration";
    case FUSE_ERR_WORKSPACE: return "workspace missing or too small";
    case FUSE_ERR_CUDA: return "CUDA error";
    case FUSE_ERR_TIMEOUT: return "device wait timed out";
    case FUSE_ERR_DEVICE_BOUNDS: return "device-detected index out of range or order";
  }
  return "unknown status";
}

int32_t fuse_version(void) { return 100; }

}  // extern "C"
