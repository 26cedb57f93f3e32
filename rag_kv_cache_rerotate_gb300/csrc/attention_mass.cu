// Query-aware attention mass of the context tokens.
//
// QCFuse (section 3.2.1, Eqs. 9-10; section 3.4.2, Eq. 20): a full-view
// selector scores context token t by the attention weight the user query
// puts on it, over the query's tokens and heads, summed over the critical
// layers.  One layer's term, for a request with N context and Qn query
// tokens:
//   I(t) = sum_{u < Qn} sum_h softmax_{t' < N}(q_{u,h} . Kf[t', h/g] / sqrt(d))[t],
//   q_{u,h} = R^{N+u} W_Q x_u,
// the softmax over the stitched context keys.
//
// The query rows of all requests are packed (request r's at qoff[r] = the
// query rows of the requests before it); their Q comes from the
// recomputation's projection, restricted to the Q heads.  Then, per (key
// tile of 64 tokens, KV head, request), a block forms the logits of the tile
// against every query vector (query token x the g query heads that read the
// KV head), 64 vectors at a time:
//   * statistics pass: each vector's maximum and sum of exp over the tile;
//   * a per-vector combination over the tiles (maximum, 1 / sum);
//   * mass pass: the logits again, each turned into its softmax weight and
//     summed over the vectors, per key -> partial[token, KV head];
// and a last launch adds the KV heads in a fixed order into the score.
// Exponentials are base 2 on logits scaled by log2(e) / sqrt(d).
#include <cmath>

#include "common.cuh"
#include "launch.h"

namespace fusekv {

namespace {

constexpr int kKT = 64;           // keys per tile
constexpr int kQC = 64;           // query vectors per chunk
constexpr int kLd = 68;           // row pitch (floats) of the transposed tiles
constexpr int kThreads = 256;     // 16 x 16 threads, 4 x 4 logits each

struct MassArgs {
  const fuse_request_t* reqs;
  const int32_t* qoff;      // [n_req] first packed query row of each request
  const void* Q;            // [Rq, Hq, d] rotated query states
  const void* Kf;           // [T_total, Hkv, d] fused cache
  float2* stats;            // [Rq * Hq, max_tiles] (max, sum) of each key tile
  const float2* norm;       // [Rq * Hq] (max, 1 / sum) over all tiles
  float* partial;           // [N_total, Hkv] mass per token and KV head
  int64_t n_qrows;          // packed query rows the host counted
  int Hq, Hkv, g, d;
  int max_tiles;
  float scale_log2;         // log2(e) / sqrt(d)
};

template <typename T> struct Vec4;
template <> struct Vec4<float> {
  static __device__ __forceinline__ float4 load(const void* base, int64_t elem) {
    return __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + elem));
  }
};
template <> struct Vec4<__nv_bfloat16> {
  static __device__ __forceinline__ float4 load(const void* base, int64_t elem) {
    const uint2 v =
        __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(base) + elem));
    return make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
  }
};

// Keys t0 .. t0 + nk - 1 of KV head g, transposed: Ks[c * kLd + key]; keys
// past nk are zero.
template <typename T>
__device__ __forceinline__ void load_keys(const MassArgs& a, const fuse_request_t& R, int g,
                                          int t0, int nk, float* Ks) {
  const int q4 = a.d / 4;
  for (int e = threadIdx.x; e < kKT * q4; e += kThreads) {
    const int kk = e / q4;
    const int c = (e % q4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (kk < nk) v = Vec4<T>::load(a.Kf, ((R.row0 + t0 + kk) * a.Hkv + g) * (int64_t)a.d + c);
    Ks[(c + 0) * kLd + kk] = v.x;
    Ks[(c + 1) * kLd + kk] = v.y;
    Ks[(c + 2) * kLd + kk] = v.z;
    Ks[(c + 3) * kLd + kk] = v.w;
  }
}

// Packed index (query row * Hq + head) of query vector v of KV head g:
// vector v is query token v / g_ratio and head g * g_ratio + v % g_ratio.
__device__ __forceinline__ int64_t vec_index(const MassArgs& a, int qoff, int g, int v) {
  return ((int64_t)qoff + v / a.g) * a.Hq + g * a.g + v % a.g;
}

// Query vectors v0 .. v0 + 63 (those below nv), transposed: Qs[c * kLd + vv].
template <typename T>
__device__ __forceinline__ void load_queries(const MassArgs& a, int qoff, int g, int v0, int nv,
                                             float* Qs) {
  const int q4 = a.d / 4;
  for (int e = threadIdx.x; e < kQC * q4; e += kThreads) {
    const int vv = e / q4;
    const int c = (e % q4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (v0 + vv < nv) v = Vec4<T>::load(a.Q, vec_index(a, qoff, g, v0 + vv) * a.d + c);
    Qs[(c + 0) * kLd + vv] = v.x;
    Qs[(c + 1) * kLd + vv] = v.y;
    Qs[(c + 2) * kLd + vv] = v.z;
    Qs[(c + 3) * kLd + vv] = v.w;
  }
}

// acc[i][j] = q(vector ty * 4 + i) . k(key tx * 4 + j), scaled to log2 units.
__device__ __forceinline__ void tile_logits(const float* Qs, const float* Ks, int d, int ty, int tx,
                                            float scale_log2, float (&acc)[4][4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 8
  for (int c = 0; c < d; ++c) {
    const float4 q = *reinterpret_cast<const float4*>(Qs + c * kLd + ty * 4);
    const float4 k = *reinterpret_cast<const float4*>(Ks + c * kLd + tx * 4);
    const float qa[4] = {q.x, q.y, q.z, q.w};
    const float ka[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(qa[i], ka[j], acc[i][j]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] *= scale_log2;
}

// The 16 threads of a row (same ty) are 16 consecutive lanes of one warp.
__device__ __forceinline__ float row_max16(float x) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float row_sum16(float x) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Statistics pass: grid (key tiles, Hkv, requests).
template <typename T>
__global__ void __launch_bounds__(kThreads) mass_stats_kernel(const MassArgs a) {
  extern __shared__ __align__(16) float smem[];
  float* Ks = smem;
  float* Qs = smem + a.d * kLd;
  const fuse_request_t R = a.reqs[blockIdx.z];
  const int g = blockIdx.y;
  const int tile = blockIdx.x;
  const int t0 = tile * kKT;
  if (t0 >= R.n_ctx) return;
  const int nk = min(kKT, R.n_ctx - t0);
  const int qoff = a.qoff[blockIdx.z];
  // query vectors of the request (its packed rows stay below the host's count)
  const int64_t avail = qoff < 0 ? 0 : a.n_qrows - qoff;
  const int nv = (int)(avail <= 0 ? 0 : (R.n_query < avail ? R.n_query : avail)) * a.g;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  load_keys<T>(a, R, g, t0, nk, Ks);
  for (int v0 = 0; v0 < nv; v0 += kQC) {
    __syncthreads();                          // Ks written / Qs of the last chunk read
    load_queries<T>(a, qoff, g, v0, nv, Qs);
    __syncthreads();
    float acc[4][4];
    tile_logits(Qs, Ks, a.d, ty, tx, a.scale_log2, acc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (tx * 4 + j < nk) m = fmaxf(m, acc[i][j]);
      m = row_max16(m);                       // finite: key 0 of the tile is valid
      float l = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (tx * 4 + j < nk) l += exp2f(acc[i][j] - m);
      l = row_sum16(l);
      const int v = v0 + ty * 4 + i;
      if (tx == 0 && v < nv)
        a.stats[vec_index(a, qoff, g, v) * a.max_tiles + tile] = make_float2(m, l);
    }
  }
}

// One thread per (packed query row, query head): the maximum over the tiles
// and 1 / the sum of exp relative to it.
__global__ void mass_norm_kernel(const fuse_request_t* reqs, int n_req, const WorkRow* rows,
                                 int64_t n_vec, int Hq, int max_tiles, const float2* stats,
                                 float2* norm) {
  const int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (id >= n_vec) return;
  const int r = rows[id / Hq].aux;
  if (r < 0 || r >= n_req) return;             // a row no request packed (tables differ)
  const int n = reqs[r].n_ctx;
  const int nt = (n + kKT - 1) / kKT;
  const float2* st = stats + id * max_tiles;
  float m = -INFINITY;
  for (int i = 0; i < nt; ++i) m = fmaxf(m, st[i].x);
  float l = 0.f;
  for (int i = 0; i < nt; ++i) l += st[i].y * exp2f(st[i].x - m);
  norm[id] = make_float2(m, l > 0.f ? 1.0f / l : 0.f);
}

// Mass pass: grid (key tiles, Hkv, requests).
template <typename T>
__global__ void __launch_bounds__(kThreads) mass_columns_kernel(const MassArgs a) {
  extern __shared__ __align__(16) float smem[];
  float* Ks = smem;
  float* Qs = smem + a.d * kLd;
  float2* Ns = reinterpret_cast<float2*>(Qs + a.d * kLd);
  const fuse_request_t R = a.reqs[blockIdx.z];
  const int g = blockIdx.y;
  const int t0 = blockIdx.x * kKT;
  if (t0 >= R.n_ctx) return;
  const int nk = min(kKT, R.n_ctx - t0);
  const int qoff = a.qoff[blockIdx.z];
  // query vectors of the request (its packed rows stay below the host's count)
  const int64_t avail = qoff < 0 ? 0 : a.n_qrows - qoff;
  const int nv = (int)(avail <= 0 ? 0 : (R.n_query < avail ? R.n_query : avail)) * a.g;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  load_keys<T>(a, R, g, t0, nk, Ks);
  float col[4] = {0.f, 0.f, 0.f, 0.f};
  for (int v0 = 0; v0 < nv; v0 += kQC) {
    __syncthreads();
    load_queries<T>(a, qoff, g, v0, nv, Qs);
    if (threadIdx.x < kQC) {
      const int v = v0 + threadIdx.x;
      Ns[threadIdx.x] = v < nv ? a.norm[vec_index(a, qoff, g, v)] : make_float2(0.f, 0.f);
    }
    __syncthreads();
    float acc[4][4];
    tile_logits(Qs, Ks, a.d, ty, tx, a.scale_log2, acc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 nm = Ns[ty * 4 + i];       // (0, 0) past nv: weight 0
#pragma unroll
      for (int j = 0; j < 4; ++j) col[j] = fmaf(exp2f(acc[i][j] - nm.x), nm.y, col[j]);
    }
  }
  // sum over the 16 rows of threads, in row order
  __syncthreads();
  float* red = Qs;                            // 16 x 64 floats
#pragma unroll
  for (int j = 0; j < 4; ++j) red[ty * kKT + tx * 4 + j] = col[j];
  __syncthreads();
  if (threadIdx.x < nk) {
    float s = 0.f;
    for (int y = 0; y < 16; ++y) s += red[y * kKT + threadIdx.x];
    a.partial[(R.score0 + t0 + threadIdx.x) * a.Hkv + g] = s;
  }
}

// score[score0 + t] (+)= sum over KV heads of partial[score0 + t, h].
__global__ void mass_reduce_kernel(const fuse_request_t* reqs, const float* partial, int Hkv,
                                   float* score, int accumulate) {
  const fuse_request_t R = reqs[blockIdx.y];
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= R.n_ctx) return;
  const float* p = partial + (R.score0 + t) * Hkv;
  float s = 0.f;
  for (int h = 0; h < Hkv; ++h) s += p[h];
  float* o = score + R.score0 + t;
  *o = accumulate ? *o + s : s;
}

// qoff[r] = sum of n_query over the requests before r (one block, chunks of
// 1024 requests with a running carry).
__global__ void __launch_bounds__(1024) query_offsets_kernel(const fuse_request_t* reqs, int n_req,
                                                             int32_t* qoff) {
  __shared__ int s_warp[32];
  __shared__ int s_carry;
  pdl_trigger();
  pdl_wait();
  const int t = threadIdx.x, lane = t % 32, warp = t / 32;
  if (t == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < n_req; base += 1024) {
    const int r = base + t;
    const int v = r < n_req ? reqs[r].n_query : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_warp[lane] = w;                       // inclusive sums of the warp totals
    }
    __syncthreads();
    if (r < n_req) qoff[r] = s_carry + (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
    __syncthreads();
    if (t == 0) s_carry += s_warp[31];
    __syncthreads();
  }
}

// One block per (query token, request): its packed work row, RoPE table at
// position N + u, and (tensor-core projection) its gathered input row.  With
// own_offsets (few requests) each block sums the query counts of the
// requests before its own, and the first block of a request writes qoff;
// otherwise query_offsets_kernel wrote qoff before.
__global__ void __launch_bounds__(256) prepare_query_rows_kernel(
    const fuse_request_t* reqs, int32_t* qoff, RopeFreqs f, int half_dim,
    const __nv_bfloat16* H, int hidden, WorkRow* rows, float2* rope, int64_t n_rows,
    __nv_bfloat16* Hs, uint32_t* err, int own_offsets) {
  __shared__ int s_off[8];
  const int r = blockIdx.y;
  const fuse_request_t R = reqs[r];   // the caller's table: no kernel writes it
  const int u = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  if (u >= R.n_query) return;         // block-uniform
  int off;
  if (own_offsets) {
    int acc = 0;
    for (int i = threadIdx.x; i < r; i += 256) acc += reqs[i].n_query;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) s_off[threadIdx.x >> 5] = acc;
    __syncthreads();
    off = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) off += s_off[w];
    if (u == 0 && threadIdx.x == 0) qoff[r] = off;
  } else {
    off = qoff[r];
  }
  const int64_t m = (int64_t)off + u;
  if (m < 0 || m >= n_rows) {                 // the device table differs from the host's
    if (threadIdx.x == 0) report_error(err, FUSE_ERR_DEVICE_BOUNDS, SITE_MASS_ROWS, r);
    return;
  }
  const int s = R.n_ctx + u;
  const int t = threadIdx.x;
  if (t == 0) {
    WorkRow w;
    w.a_row = R.row0 + s;
    w.dst_row = R.row0 + s;
    w.pos = s;
    w.aux = r;
    rows[m] = w;
  }
  if (t < half_dim) {
    float c, sn;
    rope_cos_sin(s, f.hi[t], f.mid[t], f.lo[t], c, sn);
    rope[rope_index(t, m, n_rows)] = make_float2(c, sn);
  }
  if (Hs) {
    const uint4* src = reinterpret_cast<const uint4*>(H + (R.row0 + s) * (int64_t)hidden);
    uint4* dst = reinterpret_cast<uint4*>(Hs + m * (int64_t)hidden);
    for (int c = t; c < hidden / 8; c += 256) dst[c] = __ldg(src + c);
  }
}

template <typename T>
cudaError_t run_mass(const MassArgs& a, int n_req, int max_ctx, const fuse_request_t* reqs,
                     const WorkRow* rows, int64_t n_qrows, float* score, int accumulate,
                     cudaStream_t s) {
  const int smem_stats = 2 * a.d * kLd * (int)sizeof(float);
  const int smem_cols = smem_stats + kQC * (int)sizeof(float2);
  cudaError_t e = set_dyn_smem_once(reinterpret_cast<const void*>(mass_stats_kernel<T>), smem_stats);
  if (e == cudaSuccess)
    e = set_dyn_smem_once(reinterpret_cast<const void*>(mass_columns_kernel<T>), smem_cols);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.max_tiles, a.Hkv, n_req);
  if (n_qrows > 0) {
    mass_stats_kernel<T><<<grid, kThreads, smem_stats, s>>>(a);
    const int64_t n_vec = n_qrows * a.Hq;
    mass_norm_kernel<<<(unsigned)((n_vec + 255) / 256), 256, 0, s>>>(
        reqs, n_req, rows, n_vec, a.Hq, a.max_tiles, a.stats, const_cast<float2*>(a.norm));
  }
  mass_columns_kernel<T><<<grid, kThreads, smem_cols, s>>>(a);
  mass_reduce_kernel<<<dim3((unsigned)((max_ctx + 255) / 256), n_req), 256, 0, s>>>(
      reqs, a.partial, a.Hkv, score, accumulate);
  return cudaGetLastError();
}

}  // namespace

int mass_key_tiles(int max_ctx) { return (max_ctx + kKT - 1) / kKT; }

cudaError_t launch_query_rows(const fuse_requests_t& reqs, int max_query, const RopeFreqs& freqs,
                              int head_dim, const void* H, int hidden, WorkRow* rows, float2* rope,
                              int64_t n_rows, void* Hs, int32_t* qoff, uint32_t* err,
                              cudaStream_t s) {
  if (reqs.n_req == 0) return cudaSuccess;
  // few requests: the row kernel forms the offsets itself (one launch); else
  // a block scan first
  const int own = reqs.n_req <= 1024 && max_query > 0 && n_rows > 0;
  cudaError_t e = cudaSuccess;
  if (!own) e = launch_pdl(query_offsets_kernel, dim3(1), dim3(1024), 0, s, reqs.d_req,
                           reqs.n_req, qoff);
  if (e == cudaSuccess && max_query > 0 && n_rows > 0)
    e = launch_pdl(prepare_query_rows_kernel, dim3(max_query, reqs.n_req), dim3(256), 0, s,
                   reqs.d_req, qoff, freqs, head_dim / 2, reinterpret_cast<const __nv_bfloat16*>(H),
                   hidden, rows, rope, n_rows, reinterpret_cast<__nv_bfloat16*>(Hs), err, own);
  return e;
}

cudaError_t launch_attention_mass(const fuse_layer_desc_t& d, const fuse_requests_t& reqs,
                                  int max_ctx, int64_t n_qrows, const WorkRow* rows,
                                  const int32_t* qoff, const void* Q, const void* Kf,
                                  float2* stats, float2* norm, float* partial, float* score,
                                  int accumulate, cudaStream_t s) {
  if (reqs.n_req == 0 || max_ctx == 0) return cudaSuccess;
  MassArgs a;
  a.reqs = reqs.d_req;
  a.qoff = qoff;
  a.Q = Q;
  a.Kf = Kf;
  a.stats = stats;
  a.norm = norm;
  a.partial = partial;
  a.n_qrows = n_qrows;
  a.Hq = d.n_q_heads;
  a.Hkv = d.n_kv_heads;
  a.g = d.n_q_heads / d.n_kv_heads;
  a.d = d.head_dim;
  a.max_tiles = mass_key_tiles(max_ctx);
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d.head_dim));
  if (d.dtype == FUSE_BF16)
    return run_mass<__nv_bfloat16>(a, reqs.n_req, max_ctx, reqs.d_req, rows, n_qrows, score,
                                   accumulate, s);
  return run_mass<float>(a, reqs.n_req, max_ctx, reqs.d_req, rows, n_qrows, score, accumulate, s);
}

}  // namespace fusekv
