// Key deviation of the context tokens, one layer's term.
//
// KVBoost (section 4.6.2, Alg. 2 step 2) averages, over the layers and key
// heads, the cosine between a token's key from the probe pass and its
// assembled (stitched) key:
//   delta_t = 1 - (1/(L Hkv)) sum_{l,h} cos(K~_t^(l,h), K_t^(l,h)),
//   K~_t = R^t W_K x_t   (the token at its request position t).
// delta_t is the mean over layers of 1 - (1/Hkv) sum_h cos, so one call per
// layer adds weight * (1 - (1/Hkv) sum_h cos) into the score, weight = 1/L.
//
// Launches: the work rows and RoPE table of every packed row (identity rows
// at position 0 first, then each request's rows at their positions), the
// fresh keys of all packed rows through the projection used for the query
// states (key heads in place of query heads), and one warp per context token
// for the cosines.
#include "common.cuh"
#include "launch.h"

namespace fusekv {

namespace {

// Every packed row: identity work row, RoPE at position 0 (rows outside all
// requests are projected too; their keys are never read).
__global__ void key_rows_init_kernel(int64_t n_rows, int half_dim, WorkRow* rows, float2* rope) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_rows * half_dim) return;
  const int64_t m = i / half_dim;
  const int j = (int)(i % half_dim);
  if (j == 0) {
    WorkRow w;
    w.a_row = m;
    w.dst_row = m;
    w.pos = 0;
    w.aux = -1;
    rows[m] = w;
  }
  rope[rope_index(j, m, n_rows)] = make_float2(1.f, 0.f);
}

// The rows of request blockIdx.y at their request positions.
__global__ void key_rows_kernel(const fuse_request_t* reqs, RopeFreqs f, int half_dim,
                                WorkRow* rows, float2* rope, int64_t n_rows) {
  const fuse_request_t R = reqs[blockIdx.y];
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int T = R.n_ctx + R.n_query;
  if (i >= (int64_t)T * half_dim) return;
  const int p = (int)(i / half_dim);
  const int j = (int)(i % half_dim);
  const int64_t m = R.row0 + p;
  if (m >= n_rows) return;
  if (j == 0) {
    WorkRow w;
    w.a_row = m;
    w.dst_row = m;
    w.pos = p;
    w.aux = (int)blockIdx.y;
    rows[m] = w;
  }
  float c, s;
  rope_cos_sin(p, f.hi[j], f.mid[j], f.lo[j], c, s);
  rope[rope_index(j, m, n_rows)] = make_float2(c, s);
}

template <typename T> __device__ __forceinline__ float ld(const T* p);
template <> __device__ __forceinline__ float ld<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// One warp per context token: score (+)= weight * (1 - (1/Hkv) sum_h cos),
// heads in order, each cosine's denominator clamped at 1e-30.
template <typename T>
__global__ void key_cosine_kernel(const fuse_request_t* reqs, const T* Kn, const T* Kf, int Hkv,
                                  int d, float weight, int accumulate, float* score) {
  const fuse_request_t R = reqs[blockIdx.y];
  const int lane = threadIdx.x % 32;
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= R.n_ctx) return;
  const int64_t row = (R.row0 + t) * (int64_t)Hkv;
  float sum = 0.f;
  for (int h = 0; h < Hkv; ++h) {
    const T* a = Kn + (row + h) * d;
    const T* b = Kf + (row + h) * d;
    float dot = 0.f, na = 0.f, nb = 0.f;
    for (int c = lane; c < d; c += 32) {
      const float x = ld<T>(a + c), y = ld<T>(b + c);
      dot = fmaf(x, y, dot);
      na = fmaf(x, x, na);
      nb = fmaf(y, y, nb);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      dot += __shfl_xor_sync(0xffffffffu, dot, o);
      na += __shfl_xor_sync(0xffffffffu, na, o);
      nb += __shfl_xor_sync(0xffffffffu, nb, o);
    }
    sum += dot / fmaxf(sqrtf(na) * sqrtf(nb), 1e-30f);
  }
  if (lane == 0) {
    float* o = score + R.score0 + t;
    const float v = weight * (1.0f - sum / (float)Hkv);
    *o = accumulate ? *o + v : v;
  }
}

}  // namespace

cudaError_t launch_key_rows(const fuse_requests_t& reqs, int max_tok, const RopeFreqs& freqs,
                            int head_dim, int64_t n_rows, WorkRow* rows, float2* rope,
                            cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int h2 = head_dim / 2;
  const int64_t items = n_rows * h2;
  key_rows_init_kernel<<<(unsigned)((items + 255) / 256), 256, 0, s>>>(n_rows, h2, rows, rope);
  if (reqs.n_req > 0 && max_tok > 0) {
    const int64_t per = (int64_t)max_tok * h2;
    key_rows_kernel<<<dim3((unsigned)((per + 255) / 256), reqs.n_req), 256, 0, s>>>(
        reqs.d_req, freqs, h2, rows, rope, n_rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_key_cosine(const fuse_layer_desc_t& d, const fuse_requests_t& reqs, int max_ctx,
                              const void* Kn, const void* Kf, float weight, int accumulate,
                              float* score, cudaStream_t s) {
  if (reqs.n_req == 0 || max_ctx == 0) return cudaSuccess;
  const dim3 grid((unsigned)((max_ctx + 7) / 8), reqs.n_req);
  if (d.dtype == FUSE_BF16)
    key_cosine_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        reqs.d_req, reinterpret_cast<const __nv_bfloat16*>(Kn),
        reinterpret_cast<const __nv_bfloat16*>(Kf), d.n_kv_heads, d.head_dim, weight, accumulate,
        score);
  else
    key_cosine_kernel<float><<<grid, 256, 0, s>>>(
        reqs.d_req, reinterpret_cast<const float*>(Kn), reinterpret_cast<const float*>(Kf),
        d.n_kv_heads, d.head_dim, weight, accumulate, score);
  return cudaGetLastError();
}

}  // namespace fusekv
