// Static selectors: recomputed positions from the chunk layout alone.
//
// QCFuse ("Related Work on Token Selection", query-agnostic selection): EPIC
// recomputes a fixed number of boundary tokens of every stitched chunk, the
// first tokens of a chunk behaving like attention sinks after linking.
// KVBoost ("Seam Repair", SelectiveRecompute): for each seam at position p the
// tokens [max(0, p - R), p) are recomputed with their full preceding context.
//
// Every chunk contributes one range of positions of its request (the first n
// of the chunk, or the n before the chunk's start when it is not the
// request's first).  With chunks in position order, both the starts and the
// ends of these ranges never decrease, so the union is each range clipped at
// the previous range's end, and a chunk's first output slot is the running
// sum of the clipped sizes before it.
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "launch.h"

namespace fusekv {

namespace {

struct Range {
  int64_t a, b;   // [a, b) in request positions; b of a range that selects nothing marks its end
};

__host__ __device__ inline Range chunk_range(int kind, int n, int64_t s, int64_t len, bool first) {
  if (kind == FUSE_SEL_CHUNK_HEAD) return {s, s + (len < n ? len : n)};
  if (first) return {0, 0};
  return {s - n > 0 ? s - n : 0, s};
}

// One block per request.  Threads find the request's chunks (those whose
// fused rows lie in its context), then take them blockDim at a time: each
// thread clips its chunk's range at the previous chunk's end, a block scan
// gives the output slots, and the thread writes its positions.
__global__ void __launch_bounds__(256) static_select_kernel(const fuse_request_t* reqs,
                                                            const fuse_chunk_t* chunks, int n_chunks,
                                                            int kind, int n, int32_t* idx) {
  __shared__ int s_lo, s_hi;
  __shared__ int s_warp[8];
  const fuse_request_t R = reqs[blockIdx.x];
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_lo = n_chunks;
    s_hi = -1;
  }
  __syncthreads();
  for (int c = tid; c < n_chunks; c += blockDim.x) {
    const int64_t r = chunks[c].dst_row - R.row0;
    if (r >= 0 && r < R.n_ctx) {
      atomicMin(&s_lo, c);
      atomicMax(&s_hi, c);
    }
  }
  __syncthreads();
  const int lo = s_lo, hi = s_hi;                 // chunks lo..hi (sorted, consecutive)
  int32_t* out = idx + R.sel0;
  int64_t carry = 0;
  for (int c0 = lo; c0 <= hi; c0 += blockDim.x) {
    const int c = c0 + tid;
    int64_t a = 0, b = 0;
    if (c <= hi) {
      const fuse_chunk_t ch = chunks[c];
      const Range cur = chunk_range(kind, n, ch.dst_row - R.row0, ch.len, c == lo);
      int64_t prev_end = 0;
      if (c > lo) {
        const fuse_chunk_t pc = chunks[c - 1];
        prev_end = chunk_range(kind, n, pc.dst_row - R.row0, pc.len, c - 1 == lo).b;
      }
      a = cur.a > prev_end ? cur.a : prev_end;
      b = cur.b > a ? cur.b : a;
    }
    // exclusive scan of the clipped sizes over the block (8 warps)
    const int cnt = (int)(b - a);
    int x = cnt;
    const int lane = tid % 32, warp = tid / 32;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < (int)(blockDim.x / 32); ++w) {
      if (w < warp) before += s_warp[w];
      total += s_warp[w];
    }
    before += x - cnt;
    const int64_t slot = carry + before;
    for (int64_t t = a; t < b; ++t) {
      const int64_t o = slot + (t - a);
      if (o < R.k) out[o] = (int32_t)t;
    }
    carry += total;
    __syncthreads();                              // s_warp is rewritten by the next pass
  }
}

// The counts on the host, with the same ranges; also validates the tables.
fuse_status_t static_counts(const fuse_requests_t& reqs, const fuse_chunks_t& chunks, int kind,
                            int n, std::vector<int32_t>& k) {
  if (kind != FUSE_SEL_CHUNK_HEAD && kind != FUSE_SEL_SEAM_TAIL) return FUSE_ERR_INVALID_ARG;
  if (n < 0 || reqs.n_req < 0 || chunks.n_chunks < 0) return FUSE_ERR_INVALID_ARG;
  if (reqs.n_req > 65535) return FUSE_ERR_UNSUPPORTED;
  if ((reqs.n_req > 0 && !reqs.h_req) || (chunks.n_chunks > 0 && !chunks.h_chunks))
    return FUSE_ERR_INVALID_ARG;
  const fuse_chunk_t* ch = chunks.h_chunks;
  for (int c = 0; c < chunks.n_chunks; ++c) {
    if (ch[c].len < 0 || ch[c].dst_row < 0) return FUSE_ERR_INVALID_ARG;
    if (c > 0 && ch[c].dst_row < ch[c - 1].dst_row + ch[c - 1].len) return FUSE_ERR_INVALID_ARG;
  }
  k.assign(reqs.n_req, 0);
  std::vector<int> owner(chunks.n_chunks, -1);
  for (int r = 0; r < reqs.n_req; ++r) {
    const fuse_request_t& R = reqs.h_req[r];
    if (R.n_ctx < 0) return FUSE_ERR_INVALID_ARG;
    int64_t prev_end = 0;
    bool first = true;
    for (int c = 0; c < chunks.n_chunks; ++c) {
      const int64_t s = ch[c].dst_row - R.row0;
      if (s < 0 || s >= R.n_ctx) continue;
      if (owner[c] >= 0 || s + ch[c].len > R.n_ctx) return FUSE_ERR_INVALID_ARG;
      owner[c] = r;
      const Range cur = chunk_range(kind, n, s, ch[c].len, first);
      const int64_t a = std::max(cur.a, prev_end), b = std::max(cur.b, a);
      k[r] += (int32_t)(b - a);
      prev_end = cur.b;
      first = false;
    }
  }
  for (int c = 0; c < chunks.n_chunks; ++c)
    if (owner[c] < 0 && ch[c].len > 0) return FUSE_ERR_INVALID_ARG;
  return FUSE_OK;
}

}  // namespace

}  // namespace fusekv

using namespace fusekv;

extern "C" fuse_status_t fuse_static_select_count(const fuse_requests_t* reqs,
                                                  const fuse_chunks_t* chunks, int32_t kind,
                                                  int32_t n, int32_t* k_out) {
  if (!reqs || !chunks || (reqs->n_req > 0 && !k_out)) return FUSE_ERR_INVALID_ARG;
  std::vector<int32_t> k;
  const fuse_status_t st = static_counts(*reqs, *chunks, kind, n, k);
  if (st != FUSE_OK) return st;
  std::copy(k.begin(), k.end(), k_out);
  return FUSE_OK;
}

extern "C" fuse_status_t fuse_static_select(const fuse_requests_t* reqs, const fuse_chunks_t* chunks,
                                            int32_t kind, int32_t n, int32_t* idx,
                                            fuse_stream_t stream) {
  if (!reqs || !chunks) return FUSE_ERR_INVALID_ARG;
  std::vector<int32_t> k;
  const fuse_status_t st = static_counts(*reqs, *chunks, kind, n, k);
  if (st != FUSE_OK) return st;
  int64_t n_sel = 0;
  for (int r = 0; r < reqs->n_req; ++r) {
    const fuse_request_t& R = reqs->h_req[r];
    if (R.k != k[r] || R.sel0 < 0) return FUSE_ERR_INVALID_ARG;
    n_sel = std::max<int64_t>(n_sel, R.sel0 + R.k);
  }
  if (n_sel == 0) return FUSE_OK;
  if (!idx || !reqs->d_req || !chunks->d_chunks) return FUSE_ERR_INVALID_ARG;
  static_select_kernel<<<reqs->n_req, 256, 0, (cudaStream_t)stream>>>(
      reqs->d_req, chunks->d_chunks, chunks->n_chunks, kind, n, idx);
  return cudaGetLastError() == cudaSuccess ? FUSE_OK : FUSE_ERR_CUDA;
}
