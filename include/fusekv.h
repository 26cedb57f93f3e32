/*
 * fusekv.h -- C ABI of the cache-fusion layer-step library (libfusekv.so).
 *
 * One layer-step of RAG KV-cache fusion with selective recomputation, as
 * stated on two pages:
 *   [QCFuse]  "QCFuse: Query-Aware Cache Fusion via Compressed View for
 *             Efficient RAG Serving", section 2.1 (Eqs. 1-7), Eq. 11,
 *             section 3.2.1 (Eqs. 9-10), section 3.4.2 (Eq. 20).
 *   [KVBoost] "KVBoost: Chunk-Level KV Cache Reuse with Deviation-Guided
 *             Recomputation", sections 3.1-3.2 (Eqs. 1-3), 4.5 (Eq. 7),
 *             4.6.2 (Alg. 2, CacheBlendRecompute).
 *   [PCR]     "PCR: A Prefetch-Enhanced Cache Reuse System for Low-Latency
 *             RAG Serving", layer-wise overlapping (Figure 8).
 *
 * Conventions shared by every call
 * --------------------------------
 * Ownership.  The caller allocates and owns every buffer, the workspace
 *   included.  The library allocates no device memory and keeps no pointer
 *   after a call returns.  All work is enqueued on the caller's stream; the
 *   buffers must stay valid until the stream has passed that point.
 * Pointers.  Every tensor pointer is a device pointer aligned to 16 bytes,
 *   unless the field says "host".
 * Errors.  Argument errors are detected on the host and returned before any
 *   launch; every call that takes a request table rejects one of more
 *   than 65535 requests with FUSE_ERR_UNSUPPORTED.  Launch failures return
 *   FUSE_ERR_CUDA.  Errors that only the GPU can see (an out-of-range block
 *   id or selected index, an unsorted index list, a wait that timed out)
 *   are recorded in the workspace's error word
 *   and reported by fuse_check_errors().  Nothing aborts or exits.
 * Layouts (row-major, innermost last).
 *   H        [T_total, hidden]            current hidden states; request r owns
 *                                         rows [row0, row0 + N_r + Qn_r): its N_r
 *                                         context tokens, then its Qn_r query tokens.
 *   Wq       [Hq * d, hidden]             projection weights (nn.Linear layout:
 *   Wk, Wv   [Hkv * d, hidden]             out x in, both GEMM operands K-major).
 *   Kf, Vf   [T_total, Hkv, d]            the fused cache, rows aligned with H.
 *   score    [N_total]                    request r's scores at [score0, score0 + N_r).
 *   idx      [K_total] int32              request r's k_r selected context
 *                                         positions (request-local, ascending) at
 *                                         [sel0, sel0 + k_r).
 *   O        [R_total, Hq, d]             attention rows of S_r = idx_r U {N_r .. T_r-1}
 *                                         in ascending position, at [out0, out0 + R_r),
 *                                         R_r = k_r + Qn_r.
 *   Query head h reads KV head h / (Hq / Hkv).  Positions are request-local:
 *   context token t sits at position t, query token j at N_r + j.
 * RoPE.  Rotate-half pairing (j, j + d/2) with theta_j = base^(-2j/d); the
 *   rotation R^p turns pair j by the angle p * theta_j ([KVBoost] Eq. 3).
 */
#ifndef FUSEKV_H
#define FUSEKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st* fuse_stream_t;

typedef enum {
  FUSE_OK = 0,
  FUSE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent tables      */
  FUSE_ERR_MISALIGNED = 2,    /* a pointer or row stride not aligned to 16 bytes   */
  FUSE_ERR_UNSUPPORTED = 3,   /* a valid request the library does not handle       */
  FUSE_ERR_WORKSPACE = 4,     /* workspace null or smaller than fuse_workspace_size */
  FUSE_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed              */
  FUSE_ERR_TIMEOUT = 6,       /* (device) a bounded wait gave up                   */
  FUSE_ERR_DEVICE_BOUNDS = 7  /* (device) an index read from device memory was out
                                 of range or out of order; the access was skipped  */
} fuse_status_t;

typedef enum { FUSE_F32 = 0, FUSE_BF16 = 1, FUSE_U8_ASYM = 2, FUSE_U4_ASYM = 3 } fuse_dtype_t;
typedef enum { FUSE_KV_CONTIGUOUS = 0, FUSE_KV_PAGED = 1 } fuse_kv_layout_t;
typedef enum { FUSE_ROPE_ROTATE_HALF = 0 } fuse_pos_encoding_t;

/* Shape of one attention layer.  head_dim must be 64 or 128 and n_q_heads a
 * multiple of n_kv_heads.  dtype (FUSE_F32 or FUSE_BF16) is the storage type
 * of H, the weights, the fused cache, Q and O; arithmetic accumulates in fp32.
 * Only rotary position encoding is accepted ([KVBoost] section 5 limits reuse
 * to RoPE models): any other pos_encoding returns FUSE_ERR_UNSUPPORTED. */
typedef struct {
  int32_t hidden;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  double rope_base;
  int32_t pos_encoding;
  int32_t dtype;
} fuse_layer_desc_t;

/* One cached chunk c_i of a request ([QCFuse] Eqs. 1, 3): its keys were
 * computed alone at chunk-local positions 0 .. len-1.
 *   dst_row  first row of the chunk in the packed fused cache / H.
 *   pos      request-local position o_i of the chunk's first token (the
 *            re-rotation angle offset, [QCFuse] Eq. 4).
 *   len      number of tokens.
 * Storage, selected by fuse_chunks_t.kv_layout / kv_storage:
 *   CONTIGUOUS  k, v point at this chunk's own [len, Hkv, d] arrays.
 *   PAGED       k, v point at the shared pool [n_blocks, block_size, Hkv, d];
 *               block_table (device, [ceil(len / block_size)] int32) lists the
 *               pool blocks holding tokens 0.., block_size per block.
 *   U8_ASYM     KIVI asymmetric int8 ([KVBoost] Eq. 7), codes uint8 0..255,
 *               x = zero + q * scale with fp16 scale and zero:
 *               k_scale, k_zero  [Hkv, d]  per channel over the chunk's tokens;
 *               v_scale, v_zero  [len, Hkv] per token (CONTIGUOUS) or
 *                                [n_blocks, block_size, Hkv] (PAGED pool).
 *   U4_ASYM     the same with 4-bit codes 0..15 (KIVI's b = 4), two per byte:
 *               element 2m of a row in the low nibble of byte m, 2m + 1 in
 *               the high nibble, so k and v arrays (and the pool) hold d / 2
 *               bytes per (token, head); scale and zero as for U8_ASYM.
 *   For fuse_pic_precompute, k and v are outputs (CONTIGUOUS F32/BF16 only). */
typedef struct {
  const void* k;
  const void* v;
  const int32_t* block_table;
  const void* k_scale;
  const void* k_zero;
  const void* v_scale;
  const void* v_zero;
  int64_t dst_row;
  int32_t pos;
  int32_t len;
} fuse_chunk_t;

/* The chunk table of a call: the same n_chunks entries twice, once in host
 * memory (validated and used to size the grid) and once in device memory
 * (read by the kernels).  The two copies must be identical. */
typedef struct {
  int32_t n_chunks;
  int32_t kv_layout;        /* fuse_kv_layout_t */
  int32_t kv_storage;       /* fuse_dtype_t of the chunk caches */
  int32_t block_size;       /* PAGED: tokens per pool block (> 0) */
  int64_t n_pool_blocks;    /* PAGED: pool size in blocks, for bounds checks */
  const fuse_chunk_t* h_chunks;   /* host   [n_chunks] */
  const fuse_chunk_t* d_chunks;   /* device [n_chunks] */
} fuse_chunks_t;

/* One request of a batch.  fuse_plan_requests() fills these offsets for the
 * packed layouts described at the top of this file. */
typedef struct {
  int64_t row0;     /* first row of the request in H, Kf, Vf            */
  int64_t score0;   /* first entry of its N_r scores in score[]          */
  int64_t sel0;     /* first entry of its k_r selected indices in idx[]  */
  int64_t out0;     /* first row of its R_r = k_r + Qn_r rows in O       */
  int32_t n_ctx;    /* N_r context tokens                                 */
  int32_t n_query;  /* Qn_r query tokens (always recomputed, never scored) */
  int32_t k;        /* k_r selected context tokens, 0 <= k_r <= N_r        */
  int32_t reserved; /* must be 0 */
} fuse_request_t;

/* The request table of a call, host and device copies (identical). */
typedef struct {
  int32_t n_req;
  const fuse_request_t* h_req;   /* host   [n_req] */
  const fuse_request_t* d_req;   /* device [n_req] */
} fuse_requests_t;

/* Totals of a request table (filled by fuse_plan_requests). */
typedef struct {
  int64_t n_tok;    /* T_total = sum (N_r + Qn_r): rows of H, Kf, Vf */
  int64_t n_ctx;    /* N_total: entries of score[] */
  int64_t n_sel;    /* K_total = sum k_r: entries of idx[] */
  int64_t n_out;    /* R_total = sum (k_r + Qn_r): rows of O */
  int32_t max_ctx;  /* max N_r */
  int32_t max_tok;  /* max N_r + Qn_r */
} fuse_totals_t;

/* ---------------------------------------------------------------------- */

/* Number of recomputed context tokens for ratio rho = |P| / N ([QCFuse]
 * Eq. 6): floor(rho * n_ctx + 1e-9), clamped to [0, n_ctx].  The epsilon
 * keeps products such as 0.29 * 100 = 28.999999999999996 from losing a
 * token.  Host function. */
int64_t fuse_k_from_ratio(double ratio, int64_t n_ctx);

/* Host helper: lay requests out back to back.  n_ctx, n_query: host arrays
 * [n_req].  Writes out[n_req] (k_r = fuse_k_from_ratio(ratio, N_r)) and, if
 * totals is not NULL, the totals.  Returns FUSE_ERR_INVALID_ARG on a
 * negative size or a total beyond 2^31 - 1 rows. */
fuse_status_t fuse_plan_requests(int32_t n_req, const int32_t* n_ctx, const int32_t* n_query,
                                 double ratio, fuse_request_t* out, fuse_totals_t* totals);

/* Workspace bytes needed by every call below for the given request table
 * (host copy read) and layer shape.  The workspace is caller-owned device
 * memory, 256-byte aligned, zero-filled before its first use (for example by
 * fuse_workspace_reset) and reusable across calls on one stream; calls on
 * different streams need their own.  It begins with the error word that
 * fuse_check_errors() reads; the rest is scratch that every call writes
 * before it reads. */
fuse_status_t fuse_workspace_size(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                  size_t* bytes);

/* Zero-fill the whole workspace (enqueued on the stream): before its first
 * use, and after a call that recorded a device error. */
fuse_status_t fuse_workspace_reset(void* ws, size_t ws_bytes, fuse_stream_t stream);

/* Position remapping and stitching, [QCFuse] Eq. 4 with the RoPE correction
 * of [KVBoost] section 3.2: for every chunk i and local row r < len_i,
 *   Kf[dst_row_i + r] = R^{pos_i} K_i[r]     (keys re-rotated by the offset)
 *   Vf[dst_row_i + r] = V_i[r]               (values copied in token order)
 * after dequantisation when kv_storage is FUSE_U8_ASYM or FUSE_U4_ASYM
 * ([KVBoost] Eq. 7).
 * A chunk with pos 0 whose storage type equals desc->dtype is copied bit for
 * bit.  Kf, Vf: [fused_rows, Hkv, d] in desc->dtype; every chunk must satisfy
 * dst_row + len <= fused_rows.  Query rows are not touched. */
fuse_status_t fuse_stitch_rerotate(const fuse_layer_desc_t* desc, const fuse_chunks_t* chunks,
                                   void* Kf, void* Vf, int64_t fused_rows,
                                   void* ws, size_t ws_bytes, fuse_stream_t stream);

/* Deviation score of every context token ([KVBoost] Alg. 2 step 2, taken on
 * the values of one layer): with Vn = H_t W_V^T split into Hkv heads,
 *   score_t = 1 - (1/Hkv) sum_h cos(Vn[t,h], Vf[t,h]),
 * the cosine's denominator clamped at 1e-30.  Reads H and Vf at the context
 * rows of each request (Vf holds the stitched cached values); writes
 * score[score0 + t] in fp32.  Deterministic: no floating-point atomics. */
fuse_status_t fuse_score_deviation(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                   const void* H, const void* Wv, const void* Vf, float* score,
                                   void* ws, size_t ws_bytes, fuse_stream_t stream);

/* Key deviation, one layer's term of [KVBoost] Alg. 2 step 2 as printed,
 *   delta_t = 1 - (1/(L Hkv)) sum_{l,h} cos(K~_t^(l,h), K_t^(l,h)),
 * which is the mean over the L layers of 1 - (1/Hkv) sum_h cos.  For every
 * context token t of every request, with the fresh key at the token's
 * request position (where the probe pass puts it),
 *   K~_t = R^t W_K x_t  (x_t = H[row0 + t]),   K_t = Kf[row0 + t] (stitched),
 *   v_t  = weight * (1 - (1/Hkv) sum_h cos(K~_t[h], K_t[h])),
 * each cosine's denominator clamped at 1e-30; accumulate == 0 writes v_t to
 * score[score0 + t], accumulate != 0 adds it.  One call per layer with
 * weight = 1/L (the first with accumulate == 0) leaves delta_t in score.
 * The fresh keys are materialised in desc->dtype (a bf16 layer rounds them
 * to bf16); cosines and sums are fp32, heads summed in order, no atomics.
 * Kf and H are only read.  Needs the workspace of fuse_workspace_size.
 * FUSE_ERR_INVALID_ARG for a weight that is not finite. */
fuse_status_t fuse_score_key_deviation(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                       const void* H, const void* Wk, const void* Kf, float weight,
                                       int32_t accumulate, float* score, void* ws,
                                       size_t ws_bytes, fuse_stream_t stream);

/* Query-aware importance of every context token ([QCFuse] section 3.2.1,
 * Eqs. 9-10, the full-view attention mass; section 3.4.2, Eq. 20, its sum
 * over the critical layers).  For request r with N = N_r context and
 * Qn = Qn_r query tokens, query token u (row row0 + N + u of H) has the state
 *   q_{u,h} = R^{N+u} W_Q x_u        (head h, the recomputation's projection)
 * and the score of context token t is the attention weight it receives,
 *   I(t) = sum_{u < Qn} sum_h softmax_{t' < N}(q_{u,h} . Kf[row0 + t', h/g] / sqrt(d))[t],
 * the softmax over the N context keys of the layer's fused cache (Kf after
 * fuse_stitch_rerotate: the PIC keys of [QCFuse] Eq. 4).  Every (u, h)
 * spreads a total of 1, so the scores of a request sum to Qn * Hq.
 * accumulate == 0 writes I to score[score0 + t]; accumulate != 0 adds it
 * (call once per critical layer for Eq. 20's sum).  Kf and H are only read.
 * Query states are materialised in desc->dtype (bf16 layers round q to
 * bf16); logits, weights and sums are fp32.  Deterministic: no
 * floating-point atomics.  Needs the workspace of fuse_workspace_size. */
fuse_status_t fuse_score_attention_mass(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                        const void* H, const void* Wq, const void* Kf,
                                        int32_t accumulate, float* score, void* ws,
                                        size_t ws_bytes, fuse_stream_t stream);

/* TopK(score, k_r) per request ([QCFuse] Eq. 11; [KVBoost] Alg. 2 step 3):
 * the k_r largest scores, ties broken toward the lower token index, -0 equal
 * to +0, written as ascending request-local indices to idx[sel0 ..].  A NaN
 * score is recorded as FUSE_ERR_DEVICE_BOUNDS (it ranks below every number). */
fuse_status_t fuse_select_topk(const fuse_requests_t* reqs, const float* score, int32_t* idx,
                               void* ws, size_t ws_bytes, fuse_stream_t stream);

/* Selective recomputation, [QCFuse] Eqs. 6-7 with [KVBoost] Eqs. 1-3.  For
 * every request and every row s of S_r = idx_r U {N_r .. T_r - 1}:
 *   q = R^s W_Q x_s,  k = R^s W_K x_s,  v = W_V x_s     (x_s = H[row0 + s])
 *   Kf[row0 + s] = k,  Vf[row0 + s] = v                 (scatter, Eq. 7)
 * and, after all scatters, the causal attention row
 *   O[s, h] = softmax_j(q_h . Kf[j, h/g] / sqrt(d)) Vf[j, h/g],  j <= s,
 * over the fused cache (unselected j hold reused entries, selected j the
 * refreshed ones).  idx must be ascending and < N_r (checked on the device). */
fuse_status_t fuse_recompute_selected(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                      const void* H, const void* Wq, const void* Wk,
                                      const void* Wv, const int32_t* idx, void* Kf, void* Vf,
                                      void* O, void* ws, size_t ws_bytes, fuse_stream_t stream);

/* One whole layer-step: fuse_stitch_rerotate, then (if score_this_layer)
 * fuse_score_deviation and fuse_select_topk writing idx, then
 * fuse_recompute_selected reading idx -- the order of [KVBoost] Alg. 2
 * (probe, deviation, select, patch) on the cache of [QCFuse] Eq. 4.  With
 * score_this_layer == 0, idx is an input (a selection made at another layer)
 * and score is not touched (may be NULL).  Kf, Vf have reqs' T_total rows. */
fuse_status_t fuse_layer_step(const fuse_layer_desc_t* desc, const fuse_chunks_t* chunks,
                              const fuse_requests_t* reqs, const void* H, const void* Wq,
                              const void* Wk, const void* Wv, int32_t score_this_layer,
                              int32_t* idx, void* Kf, void* Vf, void* O, float* score,
                              void* ws, size_t ws_bytes, fuse_stream_t stream);

/* The buffers of one layer of a stack (every pointer as in fuse_layer_step;
 * chunks points at this layer's chunk table, in host memory). */
typedef struct {
  const fuse_chunks_t* chunks;
  const void* H;
  const void* Wq;
  const void* Wk;
  const void* Wv;
  void* Kf;
  void* Vf;
  void* O;
} fuse_layer_io_t;

/* A stack of n_layers attention layers sharing one selection ([QCFuse]
 * section 3.4 scores critical layers only; the selection is made at one
 * layer and reused by every layer): the scoring layer is stitched, scored
 * and its top-k written to idx first; then every layer l = 0 .. n_layers-1
 * is stitched (the scoring layer only once) and recomputed with that idx.
 * layers: host array [n_layers]; all layers share desc and reqs; score
 * receives the scoring layer's scores.  One workspace serves every layer
 * (the calls run in stream order). */
fuse_status_t fuse_stack_step(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                              int32_t n_layers, int32_t score_layer, const fuse_layer_io_t* layers,
                              int32_t* idx, float* score, void* ws, size_t ws_bytes,
                              fuse_stream_t stream);

/* The same stack as one CUDA graph ([QCFuse] section 3.5: the layers of a
 * fusion step run back to back; a graph replays their launches without the
 * host issuing each one).  fuse_stack_graph_create captures fuse_stack_step
 * with these arguments on `stream` (not the legacy NULL stream, and not a
 * stream already being captured) and instantiates it; fuse_graph_launch
 * replays it on any stream, with every pointer, table and size as captured
 * (the buffers' contents may change between replays; their addresses and
 * the request and chunk tables may not).  A replay computes what the eager
 * call computes, bit for bit.  Argument errors of the captured call are
 * returned by create; no kernel runs during create.  Keep no kernel trace
 * open while creating.  fuse_graph_destroy releases the graph (host-side
 * state; call it after the last replay has been enqueued). */
typedef struct fuse_graph_st* fuse_graph_t;
fuse_status_t fuse_stack_graph_create(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                      int32_t n_layers, int32_t score_layer,
                                      const fuse_layer_io_t* layers, int32_t* idx, float* score,
                                      void* ws, size_t ws_bytes, fuse_stream_t stream,
                                      fuse_graph_t* out);
fuse_status_t fuse_graph_launch(fuse_graph_t graph, fuse_stream_t stream);
void fuse_graph_destroy(fuse_graph_t graph);

/* ---------------------------------------------------------------------- */
/* Layer-wise loading overlapped with the layers' fusion ([QCFuse] Figure 9,
 * pipeline cache fusion: each layer starts from its loaded PIC entries while
 * later layers' caches are still loading; [PCR] layer-wise overlapping,
 * Figure 8: computation starts once the first layer's cache is loaded).     */

/* One host-to-device copy: `bytes` from host memory `src` to device memory
 * `dst`.  The copy overlaps kernels only when `src` is page-locked. */
typedef struct {
  void* dst;
  const void* src;
  size_t bytes;
} fuse_copy_t;

/* The uploads of one layer of a streamed stack: the copies that fill its
 * staging slot (the device buffers its chunk table points into, and any
 * other input the caller streams through the slot). */
typedef struct {
  int32_t slot;                /* 0 .. n_slots - 1 */
  int32_t n_copies;
  const fuse_copy_t* copies;   /* host [n_copies] */
} fuse_layer_upload_t;

/* fuse_stack_step with every layer's inputs uploaded into a ring of n_slots
 * staging slots on copy_stream while earlier layers compute on stream.
 * Layers run in the order: score_layer (stitch, score, select, recompute),
 * then every other layer in index order (stitch, recompute).  The layers
 * share only the selection, so every output equals fuse_stack_step's on the
 * uploaded data.  Layer l's copies start after every earlier layer that
 * used the same slot has finished on stream; layer l's kernels start after
 * its copies.  Every copy also follows all work enqueued on stream before
 * the call (an earlier call's kernels may still read the slots), and the
 * call's last kernel on stream follows every copy, so back-to-back calls on
 * one stream need no ordering by the caller.  With n_slots >= 2 one layer's
 * upload overlaps the previous layer's kernels.  The schedule is the one
 * fuse_stack_pipeline_plan returns.  The call creates and destroys its own
 * CUDA events (2 * n_slots + 1, n_slots <= 64); everything else is as for
 * fuse_stack_step.  copy_stream
 * and stream must differ for any overlap (the same stream runs everything
 * in order).  Argument errors are returned before any copy or launch. */
fuse_status_t fuse_stack_step_streamed(const fuse_layer_desc_t* desc, const fuse_requests_t* reqs,
                                       int32_t n_layers, int32_t score_layer,
                                       const fuse_layer_io_t* layers,
                                       const fuse_layer_upload_t* uploads, int32_t n_slots,
                                       fuse_stream_t copy_stream, int32_t* idx, float* score,
                                       void* ws, size_t ws_bytes, fuse_stream_t stream);

/* The operations of a streamed stack, in issue order. */
typedef enum {
  FUSE_OP_WAIT_FREE = 0,    /* copy stream waits until the slot's last user finished  */
  FUSE_OP_COPY = 1,         /* copy stream: the layer's uploads                        */
  FUSE_OP_MARK_READY = 2,   /* copy stream: the slot's data is in place               */
  FUSE_OP_WAIT_READY = 3,   /* compute stream waits for the slot's data               */
  FUSE_OP_COMPUTE = 4,      /* compute stream: the layer's kernels                      */
  FUSE_OP_MARK_FREE = 5     /* compute stream: the layer is done with the slot          */
} fuse_pipeline_op_kind_t;

typedef struct {
  int32_t kind;    /* fuse_pipeline_op_kind_t */
  int32_t layer;
  int32_t slot;
} fuse_pipeline_op_t;

/* The schedule of fuse_stack_step_streamed (host only, no CUDA call):
 * slot_of_layer[l] in 0 .. n_slots-1 for every layer.  Writes at most
 * max_ops operations to ops and their count to *n_ops (5 per layer, plus a
 * FUSE_OP_WAIT_FREE before every reuse of a slot); FUSE_ERR_WORKSPACE when
 * max_ops is too small (*n_ops then holds the count needed). */
fuse_status_t fuse_stack_pipeline_plan(int32_t n_layers, int32_t score_layer,
                                       const int32_t* slot_of_layer, int32_t n_slots,
                                       fuse_pipeline_op_t* ops, int32_t max_ops, int32_t* n_ops);

/* Position-independent chunk caches, [QCFuse] Eq. 3 with one projection layer
 * standing in for the model: for every chunk i and local row r,
 *   K_i[r] = R^r W_K x,  V_i[r] = W_V x,   x = H_clean[dst_row_i + r].
 * This prepares inputs for the calls above (it is not part of a layer-step).
 * Chunk storage must be CONTIGUOUS and equal to desc->dtype. */
fuse_status_t fuse_pic_precompute(const fuse_layer_desc_t* desc, const fuse_chunks_t* chunks,
                                  const void* H_clean, const void* Wk, const void* Wv,
                                  void* ws, size_t ws_bytes, fuse_stream_t stream);

/* KIVI asymmetric quantisation of chunk caches ([KVBoost] section 4.5,
 * Eq. 7, b = 8 for FUSE_U8_ASYM, b = 4 for FUSE_U4_ASYM), the inverse of the
 * stitch's dequantisation; it prepares int8 / int4 inputs (it is not part of
 * a layer-step).  src: CONTIGUOUS caches in desc->dtype; dst: CONTIGUOUS
 * with the same n_chunks and lengths, kv_storage FUSE_U8_ASYM or
 * FUSE_U4_ASYM, its k, v, k_scale, k_zero, v_scale, v_zero are outputs
 * (layouts as in fuse_chunk_t).  With L = 2^b - 1, a group with minimum mn
 * and maximum mx is stored as q = rint((x - mn) / (mx - mn) * L) (round half
 * to even, in fp64), scale = fp16((mx - mn) / L), zero = fp16(mn); a constant
 * group gets q = 0 and scale 0.  Key groups: (chunk, head, channel) over the
 * chunk's tokens; value groups: (token, head) over d.  Argument errors
 * (mismatched tables, other layouts or storage) are returned before any
 * launch. */
fuse_status_t fuse_kivi_quantize(const fuse_layer_desc_t* desc, const fuse_chunks_t* src,
                                 const fuse_chunks_t* dst, fuse_stream_t stream);

/* Synchronise the stream, read the workspace's error word, clear it, and
 * return it (FUSE_OK if no device-side error was recorded).  If detail is
 * not NULL it receives a code locating the failed check. */
fuse_status_t fuse_check_errors(void* ws, fuse_stream_t stream, uint32_t* detail);

/* Top-k without a workspace (no counterpart on the pages).  Same selection
 * as fuse_select_topk, for callers that cannot allocate device memory when
 * they select: a serving loop that has given all free HBM to its KV-cache
 * pool, or code running where the allocator must not be touched.  The key
 * scratch is a fixed device array inside the library (4 *
 * FUSE_TOPK_NOALLOC_MAX_KEYS + 256 bytes, 2 MiB), held on every GPU that
 * loads the library until the process exits; this call allocates nothing.
 *   - N_total (the largest score0 + N_r) above FUSE_TOPK_NOALLOC_MAX_KEYS is
 *     rejected with FUSE_ERR_WORKSPACE before any launch.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture.
 *   - All calls share the one array: calls whose work overlaps on the GPU
 *     (different streams, no ordering between them) race and give wrong
 *     indices.  Order them on one stream or with events.
 *   - NaN scores still rank below every number, but this variant does not
 *     report them (fuse_select_topk with a workspace does). */
#define FUSE_TOPK_NOALLOC_MAX_KEYS (1 << 19)
fuse_status_t fuse_select_topk_noalloc(const fuse_requests_t* reqs, const float* score,
                                       int32_t* idx, fuse_stream_t stream);

/* Static selectors: indices generated from the chunk layout alone, no
 * scores (the query-agnostic selectors of the "Token Selection" related-work
 * section of the QCFuse page, and SelectiveRecompute, "Seam Repair" section
 * of the KVBoost page).  A request's context is the concatenation of the
 * chunks whose fused rows lie in [row0, row0 + N_r); a chunk starts at
 * position s = dst_row - row0 of its request.
 *   FUSE_SEL_CHUNK_HEAD: the first n tokens of every chunk, [s, s + min(n, len))
 *     (EPIC's LegoLink rule: the first tokens of a stitched chunk act as
 *     attention sinks; the page gives no count, so n is a parameter).
 *   FUSE_SEL_SEAM_TAIL: the n tokens before every seam, [max(0, p - n), p)
 *     for each p = s of a chunk that is not the request's first (a seam is
 *     where two chunks join; the page's default is n = 16).
 * The selection of a request is the union of its ranges, ascending.
 * Requirements (else FUSE_ERR_INVALID_ARG): host mirrors of both tables;
 * chunks sorted by dst_row and non-overlapping; every chunk with len > 0
 * inside exactly one request's context rows; n >= 0. */
typedef enum { FUSE_SEL_CHUNK_HEAD = 0, FUSE_SEL_SEAM_TAIL = 1 } fuse_static_sel_t;

/* Host only, no launch: k_out[r] = size of request r's selection (host array
 * of n_req entries), to be written into the request table's k before
 * fuse_static_select. */
fuse_status_t fuse_static_select_count(const fuse_requests_t* reqs, const fuse_chunks_t* chunks,
                                       int32_t kind, int32_t n, int32_t* k_out);

/* Enqueues one kernel that writes each request's selection, ascending, to
 * idx[sel0 .. sel0 + k_r) (device array).  reqs->h_req[r].k must equal the
 * count of fuse_static_select_count (else FUSE_ERR_INVALID_ARG).  The
 * indices feed fuse_recompute_selected like those of fuse_select_topk. */
fuse_status_t fuse_static_select(const fuse_requests_t* reqs, const fuse_chunks_t* chunks,
                                 int32_t kind, int32_t n, int32_t* idx, fuse_stream_t stream);

/* Kernel timing trace (no counterpart on the pages; a measurement aid).
 * fuse_trace_begin(n) creates n pairs of CUDA events and, until
 * fuse_trace_end, records one pair around each kernel the library launches,
 * on that launch's stream; launches past n are not recorded.  fuse_trace_end
 * waits for the recorded events and writes up to max_out entries
 * {kernel name (static string), elapsed ms} in launch order, *n_out their
 * count.  Host-side state: one trace at a time per process.  Do not open a
 * trace while a stream is being captured into a CUDA graph. */
typedef struct {
  const char* kernel;
  float ms;
} fuse_trace_entry_t;

fuse_status_t fuse_trace_begin(int32_t max_records);
fuse_status_t fuse_trace_end(fuse_trace_entry_t* out, int32_t max_out, int32_t* n_out);

/* Self-test of the device-side failure detection (no counterpart on the
 * pages; a diagnostic).  Launches one CTA on `stream` whose thread waits,
 * through the same bounded mbarrier wait every pipeline of the library uses,
 * on a barrier that nothing arrives on.  When the wait gives up (after its
 * one-second limit) the kernel records FUSE_ERR_TIMEOUT in the workspace's
 * error word and returns, so the context stays usable: fuse_check_errors then
 * returns FUSE_ERR_TIMEOUT.  ws: a workspace of at least 256 bytes (only its
 * header is used), 256-byte aligned.  No fault, trap or endless wait is
 * involved. */
fuse_status_t fuse_selftest_wait_timeout(void* ws, size_t ws_bytes, fuse_stream_t stream);

/* A static, human-readable name of a status code. */
const char* fuse_status_string(fuse_status_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t fuse_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FUSEKV_H */
