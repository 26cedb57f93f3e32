// Launchers of the kernels of libfusekv (host side, called by api.cu).
#pragma once

#include <cuda_runtime.h>

#include <mutex>
#include <set>
#include <tuple>
#include <utility>

#include "common.cuh"

namespace fusekv {

// Raise a kernel's dynamic shared-memory limit to `bytes`, once per device
// (the call costs host time on every launch otherwise).
inline cudaError_t set_dyn_smem_once(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::tuple<int, const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_tuple(dev, kernel, bytes);
  std::lock_guard<std::mutex> g(mu);
  if (done.count(key)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert(key);
  return e;
}

// Launch with programmatic stream serialisation (see pdl_trigger/pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same, in clusters of two CTAs (2-SM MMA pairs).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_pairs(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Stitch + re-rotate (+ dequantise, + paged gather) every chunk.  free_sms
// < 0: after the previous kernel; otherwise alongside it (the previous kernel
// reads no output of the stitch and leaves free_sms SMs free), which needs
// stitch_streamed(): chunk caches of the layer's type.
cudaError_t launch_stitch(const fuse_layer_desc_t& desc, const fuse_chunks_t& chunks,
                          const RopeFreqs& freqs, int max_len, void* Kf, void* Vf, uint32_t* err,
                          cudaStream_t s, int free_sms = -1);
bool stitch_streamed(const fuse_layer_desc_t& desc, const fuse_chunks_t& chunks);

// Score slot of every packed row: score0 + t for context rows, -1 for query rows.
cudaError_t launch_build_score_map(const fuse_requests_t& reqs, int max_tok, int32_t* map,
                                   cudaStream_t s);

// Work rows (and their RoPE table) of S_r = idx_r U query rows, per request.
cudaError_t launch_build_sel_rows(const fuse_requests_t& reqs, int max_rows, const int32_t* idx,
                                  const RopeFreqs& freqs, int head_dim, WorkRow* rows,
                                  float2* rope, int64_t n_rows, uint32_t* err, cudaStream_t s);

// Deviation: partial[slot, h] = cos(H_t W_V^T [h], Vf[t, h]) over all packed rows.
cudaError_t launch_deviation_partials_simt(const fuse_layer_desc_t& desc, int64_t n_rows, const void* H,
                                      const void* Wv, const void* Vf, const int32_t* map,
                                      float* partial, uint32_t* err, cudaStream_t s);

// score[i] = 1 - (sum_p partial[i, p]) / n_kv_heads over n_parts partials.
cudaError_t launch_deviation_reduce(int64_t n_ctx, int n_parts, int n_kv_heads,
                                    const float* partial, float* score, cudaStream_t s);

// Work rows, RoPE table, gathered Hs and attention tiles of the recomputed rows
// (tensor-core path), one launch.
cudaError_t launch_prepare_rows(const fuse_requests_t& reqs, int max_rows, const int32_t* idx,
                                const RopeFreqs& freqs, int head_dim, const void* H, int hidden,
                                WorkRow* rows, float2* rope, int64_t n_rows, void* Hs, int rtile,
                                void* tiles, uint32_t* err, cudaStream_t s);

// score = 1 - (sum_p partial[p]) / n_kv_heads, written to score[], then
// top-k per request.
cudaError_t launch_reduce_topk(const fuse_requests_t& reqs, int max_ctx, const float* partial,
                               int n_parts, int n_kv_heads, float* score, int32_t* idx,
                               uint32_t* keys_ws, uint32_t* err, cudaStream_t s);

// Top-k per request, ascending indices.
cudaError_t launch_topk(const fuse_requests_t& reqs, int max_ctx, const float* score, int32_t* idx,
                        uint32_t* keys_ws, uint32_t* err, cudaStream_t s);

// Gathered projection of work rows with RoPE and scatter (recompute: Q | K | V).
cudaError_t launch_project_recompute_simt(const fuse_layer_desc_t& desc, int64_t n_rows,
                                          const WorkRow* rows, const float2* rope, const void* H,
                                          const void* Wq, const void* Wk, const void* Wv, void* Q,
                                          void* Kf, void* Vf, uint32_t* err, cudaStream_t s);

// Projection of chunk tokens into the chunk caches (PIC: K | V), RoPE at the
// chunk-local position.
cudaError_t launch_project_pic(const fuse_layer_desc_t& desc, int n_chunks, int max_len,
                               const RopeFreqs& freqs, const void* H, const void* Wk, const void* Wv,
                               const fuse_chunk_t* d_chunks, uint32_t* err, cudaStream_t s);

// KIVI quantisation of layer-type chunk caches into codes with fp16 scale / zero
// (input preparation).
cudaError_t launch_kivi_quantize(const fuse_layer_desc_t& d, const fuse_chunks_t& src,
                                 const fuse_chunks_t& dst, int max_len, cudaStream_t s);

// Query projection of packed work rows (Q heads only, RoPE at each row's position).
cudaError_t launch_project_query_simt(const fuse_layer_desc_t& desc, int64_t n_rows,
                                      const WorkRow* rows, const float2* rope, const void* H,
                                      const void* Wq, void* Q, uint32_t* err, cudaStream_t s);

// Query-aware attention mass: key tiles per request, the packed query rows
// (offsets, work rows, RoPE table, gathered inputs), and the scoring launches.
int mass_key_tiles(int max_ctx);
cudaError_t launch_query_rows(const fuse_requests_t& reqs, int max_query, const RopeFreqs& freqs,
                              int head_dim, const void* H, int hidden, WorkRow* rows, float2* rope,
                              int64_t n_rows, void* Hs, int32_t* qoff, uint32_t* err,
                              cudaStream_t s);
cudaError_t launch_attention_mass(const fuse_layer_desc_t& d, const fuse_requests_t& reqs,
                                  int max_ctx, int64_t n_qrows, const WorkRow* rows,
                                  const int32_t* qoff, const void* Q, const void* Kf,
                                  float2* stats, float2* norm, float* partial, float* score,
                                  int accumulate, cudaStream_t s);

// Causal GQA attention of the work rows over the fused cache.
cudaError_t launch_attention_simt(const fuse_layer_desc_t& desc, int64_t n_rows, const WorkRow* rows,
                                  const void* Q, const void* Kf, const void* Vf, void* O,
                                  cudaStream_t s);

}  // namespace fusekv
