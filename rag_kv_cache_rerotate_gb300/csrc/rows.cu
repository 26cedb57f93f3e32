// Row tables: which packed row feeds each GEMM row, where its result goes,
// and the (cos, sin) of its RoPE position.
//
// QCFuse (section 2.1.3, Eqs. 6-7): the rows recomputed for one request are
// S = P U U -- the selected context positions and every user-query token --
// each at its own request position; results are written back to the same
// positions.  QCFuse (Eq. 3): a chunk cache is built at chunk-local
// positions 0 .. len-1.
#include "common.cuh"
#include "launch.h"

namespace fusekv {

namespace {

__global__ void score_map_kernel(const fuse_request_t* reqs, int32_t* map) {
  const fuse_request_t R = reqs[blockIdx.y];
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int T = R.n_ctx + R.n_query;
  if (t >= T) return;
  map[R.row0 + t] = t < R.n_ctx ? (int32_t)(R.score0 + t) : -1;
}

// One thread per (work row, frequency pair).
__global__ void sel_rows_kernel(const fuse_request_t* reqs, const int32_t* idx, RopeFreqs f,
                                int half_dim, WorkRow* rows, float2* rope, int64_t total_rows,
                                uint32_t* err) {
  const int r = blockIdx.y;
  const fuse_request_t R = reqs[r];
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int n_rows = R.k + R.n_query;
  const int o = (int)(i / half_dim);
  const int j = (int)(i % half_dim);
  if (o >= n_rows) return;
  int s;
  if (o < R.k) {
    s = idx[R.sel0 + o];
    if (j == 0) {
      if (s < 0 || s >= R.n_ctx) {
        report_error(err, FUSE_ERR_DEVICE_BOUNDS, SITE_SEL_RANGE, r);
      } else if (o > 0 && idx[R.sel0 + o - 1] >= s) {
        report_error(err, FUSE_ERR_DEVICE_BOUNDS, SITE_SEL_ORDER, r);
      }
    }
    s = min(max(s, 0), max(R.n_ctx - 1, 0));
  } else {
    s = R.n_ctx + (o - R.k);
  }
  const int64_t out = R.out0 + o;
  if (j == 0) {
    WorkRow w;
    w.a_row = R.row0 + s;
    w.dst_row = R.row0 + s;
    w.pos = s;
    w.aux = r;
    rows[out] = w;
  }
  float c, sn;
  rope_cos_sin(s, f.hi[j], f.mid[j], f.lo[j], c, sn);
  rope[rope_index(j, out, total_rows)] = make_float2(c, sn);
}

// One block per recomputed row (blockIdx.y = request): the work row, its RoPE
// table and the gathered copy Hs[out] = H[row0 + s]; block (0, 0) also writes
// the attention tile records (build_attn_tiles).
__global__ void __launch_bounds__(256) prepare_rows_kernel(const fuse_request_t* reqs, int n_req,
                                                           const int32_t* idx, RopeFreqs f,
                                                           int half_dim, const __nv_bfloat16* H,
                                                           int hidden, WorkRow* rows, float2* rope,
                                                           int64_t n_rows,
                                                           __nv_bfloat16* Hs, int rtile,
                                                           int4* tiles, uint32_t* err) {
  const int r = blockIdx.y;
  const fuse_request_t R = reqs[r];     // the caller's table: no kernel writes it
  pdl_trigger();
  pdl_wait();
  const int o = blockIdx.x;
  const int t = threadIdx.x;
  if (tiles && o == 0 && r == 0) build_attn_tiles(reqs, n_req, idx, rtile, tiles);
  if (o >= R.k + R.n_query) return;
  int s;
  if (o < R.k) {
    s = idx[R.sel0 + o];
    if (t == 0) {
      if (s < 0 || s >= R.n_ctx)
        report_error(err, FUSE_ERR_DEVICE_BOUNDS, SITE_SEL_RANGE, r);
      else if (o > 0 && idx[R.sel0 + o - 1] >= s)
        report_error(err, FUSE_ERR_DEVICE_BOUNDS, SITE_SEL_ORDER, r);
    }
    s = min(max(s, 0), max(R.n_ctx - 1, 0));
  } else {
    s = R.n_ctx + (o - R.k);
  }
  const int64_t out = R.out0 + o;
  if (t == 0) {
    WorkRow w;
    w.a_row = R.row0 + s;
    w.dst_row = R.row0 + s;
    w.pos = s;
    w.aux = r;
    rows[out] = w;
  }
  if (t < half_dim) {
    float c, sn;
    rope_cos_sin(s, f.hi[t], f.mid[t], f.lo[t], c, sn);
    rope[rope_index(t, out, n_rows)] = make_float2(c, sn);
  }
  const uint4* src = reinterpret_cast<const uint4*>(H + (R.row0 + s) * (int64_t)hidden);
  uint4* dst = reinterpret_cast<uint4*>(Hs + out * (int64_t)hidden);
  for (int c = t; c < hidden / 8; c += 256) dst[c] = __ldg(src + c);
}

}  // namespace

cudaError_t launch_prepare_rows(const fuse_requests_t& reqs, int max_rows, const int32_t* idx,
                                const RopeFreqs& freqs, int head_dim, const void* H, int hidden,
                                WorkRow* rows, float2* rope, int64_t n_rows, void* Hs, int rtile,
                                void* tiles, uint32_t* err, cudaStream_t s) {
  if (reqs.n_req == 0 || max_rows == 0) return cudaSuccess;
  dim3 grid(max_rows, reqs.n_req);
  return launch_pdl(prepare_rows_kernel, grid, dim3(256), 0, s, reqs.d_req, reqs.n_req, idx, freqs,
                    head_dim / 2, reinterpret_cast<const __nv_bfloat16*>(H), hidden, rows, rope, n_rows,
                    reinterpret_cast<__nv_bfloat16*>(Hs), rtile, reinterpret_cast<int4*>(tiles),
                    err);
}

cudaError_t launch_build_score_map(const fuse_requests_t& reqs, int max_tok, int32_t* map,
                                   cudaStream_t s) {
  if (reqs.n_req == 0 || max_tok == 0) return cudaSuccess;
  dim3 grid((max_tok + 255) / 256, reqs.n_req);
  score_map_kernel<<<grid, 256, 0, s>>>(reqs.d_req, map);
  return cudaGetLastError();
}

cudaError_t launch_build_sel_rows(const fuse_requests_t& reqs, int max_rows, const int32_t* idx,
                                  const RopeFreqs& freqs, int head_dim, WorkRow* rows,
                                  float2* rope, int64_t n_rows, uint32_t* err, cudaStream_t s) {
  if (reqs.n_req == 0 || max_rows == 0) return cudaSuccess;
  const int h2 = head_dim / 2;
  const int64_t items = (int64_t)max_rows * h2;
  dim3 grid((unsigned)((items + 255) / 256), reqs.n_req);
  sel_rows_kernel<<<grid, 256, 0, s>>>(reqs.d_req, idx, freqs, h2, rows, rope, n_rows, err);
  return cudaGetLastError();
}

}  // namespace fusekv
