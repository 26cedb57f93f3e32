// Shared device helpers of libfusekv: error word, element loads/stores,
// RoPE angles, the workspace header.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fusekv.h"

namespace fusekv {

// ----------------------------------------------------------------------------
// Workspace header: the first 256 bytes of every workspace.
// ----------------------------------------------------------------------------
struct WsHeader {
  uint32_t err_code;     // first device-detected fuse_status_t, 0 if none
  uint32_t err_detail;   // where it was detected (see ErrSite)
  uint32_t pad[62];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Sites that record a device error (err_detail = site << 24 | low bits of an index).
enum ErrSite : uint32_t {
  SITE_STITCH_BLOCK = 1,     // paged block id outside the pool
  SITE_STITCH_ROWS = 2,      // chunk rows outside the fused cache
  SITE_SEL_RANGE = 3,        // selected index >= N_r or < 0
  SITE_SEL_ORDER = 4,        // selected indices not strictly ascending
  SITE_TOPK_NAN = 5,         // NaN score
  SITE_GEMM_TIMEOUT = 6,     // tensor-core pipeline wait gave up
  SITE_ATTN_TIMEOUT = 7,     // attention pipeline wait gave up
  SITE_STITCH_TIMEOUT = 8,   // stitch bulk-copy wait gave up
  SITE_MASS_ROWS = 9,        // query rows past the host's count (device table differs)
  SITE_MASS_TIMEOUT = 10,    // tensor-core attention-mass pipeline wait gave up
};

__device__ __forceinline__ void report_error(uint32_t* err, fuse_status_t code, uint32_t site,
                                             uint32_t info) {
  if (atomicCAS(err, 0u, (uint32_t)code) == 0u) {
    err[1] = (site << 24) | (info & 0xFFFFFFu);
  }
}

// ----------------------------------------------------------------------------
// Programmatic dependent launch: every kernel of a call sequence is launched so
// that it may start while the previous one drains (launch_pdl).  A kernel lets
// the next one start once all of its own CTAs are running (pdl_trigger) and
// waits for the previous kernel to complete, with its writes visible, before
// it touches global memory (pdl_wait); only on-chip set-up, and reads of the
// caller's request table (which no kernel writes), run before that.
// Both are no-ops for a kernel launched without the attribute.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------------------
// Element types
// ----------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 8 consecutive elements -> fp32.
template <typename T> struct Vec8;

template <> struct Vec8<float> {
  static __device__ __forceinline__ void load_shared(const float* p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  static __device__ __forceinline__ void load(const float* p, float (&x)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&x)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
};

template <> struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load_shared(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
    x[4] = bf16_lo(a.z); x[5] = bf16_hi(a.z); x[6] = bf16_lo(a.w); x[7] = bf16_hi(a.w);
  }
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[8]) {
    uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
    x[4] = bf16_lo(a.z); x[5] = bf16_hi(a.z); x[6] = bf16_lo(a.w); x[7] = bf16_hi(a.w);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&x)[8]) {
    uint4 a;
    a.x = pack_bf16x2(x[0], x[1]); a.y = pack_bf16x2(x[2], x[3]);
    a.z = pack_bf16x2(x[4], x[5]); a.w = pack_bf16x2(x[6], x[7]);
    *reinterpret_cast<uint4*>(p) = a;
  }
};

// ----------------------------------------------------------------------------
// RoPE angles in fp32 without losing the large-position accuracy.
//
// The rotation angle of pair j at position p is p * theta_j radians, i.e.
// p * f_j turns with f_j = theta_j / (2 pi).  f_j is split on the host (in
// fp64) into three floats hi + mid + lo.  The fractional part of p * f_j is
// then formed with Cody and Waite's additive reduction against a multi-word
// constant, using the FMA-exact product error (Dekker's two-product) for the
// leading term:
//   a = p * hi,  e = fma(p, hi, -a)   (a + e == p * hi exactly)
//   t = (a - rint(a)) + (e + p * mid + p * lo),  t -= rint(t)
// so |t| <= 1/2 turn with an absolute error near 2^-25 turn for p < 2^24.
// sincospif(2 t) then gives cos and sin of the angle.
// ----------------------------------------------------------------------------
constexpr int kMaxHalfDim = 64;   // head_dim <= 128

struct RopeFreqs {
  float hi[kMaxHalfDim];
  float mid[kMaxHalfDim];
  float lo[kMaxHalfDim];
};

__device__ __forceinline__ void rope_cos_sin(int p, float hi, float mid, float lo, float& c,
                                             float& s) {
  const float fp = (float)p;
  const float a = fp * hi;
  const float e = fmaf(fp, hi, -a);
  float t = (a - rintf(a)) + (e + fmaf(fp, mid, fp * lo));
  t -= rintf(t);
  sincospif(2.0f * t, &s, &c);
}

// ----------------------------------------------------------------------------
// Deviation score of one token from its cosine partials.
// ----------------------------------------------------------------------------
// The partials of a token are n_parts sums of its per-KV-head cosines (one
// per head, or one per pair of heads); the score is
// The same for n_parts == 4, from the four partials already loaded (the
// same additions in the same order).
__device__ __forceinline__ float head_mean_score4(float4 v, int n_heads) {
  const float acc = (((0.f + v.x) + v.y) + v.z) + v.w;
  return 1.0f - acc / (float)n_heads;
}

// 1 - (sum_p partial[p]) / n_heads, the sum taken in partial order; 16-byte
// loads when n_parts % 4 == 0.
__device__ __forceinline__ float head_mean_score(const float* pr, int n_parts, int n_heads) {
  float acc = 0.f;
  if ((n_parts & 3) == 0) {
    float4 v[4];
    for (int h0 = 0; h0 < n_parts; h0 += 16) {
      const int nq = min(4, (n_parts - h0) / 4);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < nq) v[q] = __ldg(reinterpret_cast<const float4*>(pr + h0) + q);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < nq) acc = (((acc + v[q].x) + v[q].y) + v[q].z) + v[q].w;
    }
  } else {
    for (int h = 0; h < n_parts; ++h) acc += pr[h];
  }
  return 1.0f - acc / (float)n_heads;
}

// ----------------------------------------------------------------------------
// Per-row work item of the gathered GEMMs and the attention kernel.
// ----------------------------------------------------------------------------
struct WorkRow {
  int64_t a_row;     // row of H (or H_clean) feeding the projection
  int64_t dst_row;   // fused-cache row (recompute) or chunk-local row (PIC)
  int32_t pos;       // RoPE position p
  int32_t aux;       // request (recompute) or chunk (PIC) index
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// RoPE table of the work rows: (cos, sin) of frequency pair j of work row m
// sits at this float2 index.  Pairs of pairs are stored pair-major, so the
// four floats of pairs 2i, 2i + 1 of row m are one float4 at i * n_rows + m
// and threads holding consecutive rows read consecutive 16-byte entries.
__host__ __device__ inline int64_t rope_index(int j, int64_t m, int64_t n_rows) {
  return (((int64_t)(j >> 1) * n_rows + m) << 1) | (j & 1);
}

#ifdef __CUDACC__
// Tile records of the tensor-core attention: the recomputed rows of each
// request cut into tiles of rtile rows, in request order, each recorded as
// (first output row, the request's first fused row, rows, key blocks), the
// key blocks being those up to the position of the tile's last row (selected
// index, clamped to the request like the row tables, or n_ctx + query row).
// Run by every thread of one block of a multiple of 32 threads, at most 1024
// (the caller's branch must be block-uniform); requests past kTileReqsSmem
// are enumerated by one thread (slower, same result).  Up to kTileSortMax
// tiles are ordered by key blocks, ascending and stable, so that the
// attention kernel (which takes the last tiles first) starts the heaviest
// tiles of every request of a batch first; more stay in request order.
constexpr int kTileReqsSmem = 1024;
constexpr int kTileSortMax = 1024;
__device__ inline void build_attn_tiles(const fuse_request_t* reqs, int n_req, const int32_t* idx,
                                        int rtile, int4* tiles) {
  __shared__ int s_first[kTileReqsSmem + 1];     // first tile of each request, then the total
  __shared__ int s_warp[32];
  const int tid = threadIdx.x, nth = blockDim.x;
  if (n_req > kTileReqsSmem) {
    if (tid == 0) {
      int nt = 0;
      for (int q = 0; q < n_req; ++q) {
        const int n = reqs[q].k + reqs[q].n_query;
        for (int r0 = 0; r0 < n; r0 += rtile) tiles[nt++] = make_int4(q, r0, min(rtile, n - r0), 0);
      }
      s_first[0] = nt;
    }
    __syncthreads();
    const int nt = s_first[0];
    for (int t = tid; t < nt; t += nth) {
      const int4 x = tiles[t];
      const fuse_request_t R = reqs[x.x];
      const int o = x.y + x.z - 1;
      const int pos = o < R.k ? min(max(idx[R.sel0 + o], 0), max(R.n_ctx - 1, 0)) : R.n_ctx + (o - R.k);
      tiles[t] = make_int4((int)R.out0 + x.y, (int)R.row0, x.z, pos / 128 + 1);
    }
    return;
  }
  // tiles per request, and their running sum, blockDim requests at a time
  const int lane = tid % 32, warp = tid / 32, nw = nth / 32;
  int carry = 0;                                 // block-uniform
  for (int q0 = 0; q0 < n_req; q0 += nth) {
    const int q = q0 + tid;
    const int cnt = q < n_req ? (reqs[q].k + reqs[q].n_query + rtile - 1) / rtile : 0;
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    if (q < n_req) s_first[q] = carry + (warp > 0 ? s_warp[warp - 1] : 0) + x - cnt;
    carry += s_warp[nw - 1];
    __syncthreads();                             // s_warp is rewritten by the next chunk
  }
  if (tid == 0) s_first[n_req] = carry;
  __syncthreads();
  const int nt = s_first[n_req];
  __shared__ int4 s_rec[kTileSortMax];
  const bool sort = nt <= kTileSortMax;          // block-uniform
  for (int t = tid; t < nt; t += nth) {
    int lo = 0, hi = n_req - 1;                  // the request: last q with s_first[q] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_first[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const fuse_request_t R = reqs[lo];
    const int r0 = (t - s_first[lo]) * rtile;
    const int rows = min(rtile, R.k + R.n_query - r0);
    const int o = r0 + rows - 1;
    const int pos = o < R.k ? min(max(idx[R.sel0 + o], 0), max(R.n_ctx - 1, 0)) : R.n_ctx + (o - R.k);
    const int4 rec = make_int4((int)R.out0 + r0, (int)R.row0, rows, pos / 128 + 1);
    if (sort)
      s_rec[t] = rec;
    else
      tiles[t] = rec;
  }
  if (!sort) return;
  __syncthreads();
  // stable rank by key blocks: the tiles with fewer blocks, and those with as
  // many that come earlier
  for (int t = tid; t < nt; t += nth) {
    const int w = s_rec[t].w;
    int rank = 0;
    for (int q = 0; q < nt; ++q) {
      const int wq = s_rec[q].w;
      rank += (wq < w) || (wq == w && q < t);
    }
    tiles[rank] = s_rec[t];
  }
}
#endif

}  // namespace fusekv
