// Projection of a few rows onto the query heads on tcgen05 tensor cores: the
// query rows of the query-aware scorer, q_{u,h} = R^{N+u} W_Q x_u (QCFuse
// section 3.2.1, Eq. 9).
//
// The rows are the short side, so the product is formed transposed, Q^T =
// W_Q X^T head by head: a head's 128 weight rows are the M = 128 side of the
// MMA and up to 64 rows the N = 64 side, and the tile is full however few
// rows there are (a 256-row pair tile of the layer GEMM would be mostly
// empty).  One CTA per (head, group of 64 rows, split of the hidden
// dimension): lane 0 of warp 0 loads 64-deep W and X tiles through a
// 4-stage TMA ring, lane 0 of warp 1 issues four 128 x 64 x 16 MMAs per tile
// into a 64-column fp32 accumulator in TMEM; then the four warps read the
// accumulator (thread = feature = TMEM lane) and store the split's partial
// transposed back to [split][row][head * 128 + feature].  A second kernel
// adds the splits in order, rotates each pair (j, j + 64) by the row's RoPE
// factors and rounds to bf16.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace fusekv {

bool tma_encode_available();
bool make_map_3d(CUtensorMap* m, const void* base, const uint64_t dims[3], const uint64_t strides[2],
                 const uint32_t box[3]);

namespace {

constexpr int kQpM = 128;                            // features of one head
constexpr int kQpN = 64;                             // rows per CTA
constexpr int kQpK = 64;                             // depth of a stage (128 bytes of bf16)
constexpr int kQpStages = 4;
constexpr int kQpThreads = 128;
constexpr int kQpWBytes = kQpM * kQpK * 2;           // 16 KB
constexpr int kQpXBytes = kQpN * kQpK * 2;           // 8 KB
constexpr int kQpStageBytes = kQpWBytes + kQpXBytes;
constexpr int kQpTmemCols = kQpN;
constexpr int kQpMaxSplits = 8;
constexpr int64_t kQpMaxRows = 128;   // two groups of 64 rows; more rows fill the layer GEMM's pair tiles better

struct QpCtl {
  uint64_t full[kQpStages], empty[kQpStages];
  uint64_t acc_full;
  uint32_t tmem_base;
  volatile int abort_flag;
};
constexpr int kQpSmemBytes = kQpStages * kQpStageBytes + 1024 + (int)sizeof(QpCtl);

struct QpArgs {
  int n_rows;
  int n_heads;
  int k_steps;           // hidden / kQpK
  int steps_per_split;
  float* part;           // [split][row][n_heads * 128]
  uint32_t* err;
};

__device__ __forceinline__ void qp_abort(QpCtl* ctl, uint32_t* err) {
  ctl->abort_flag = 1;
  report_error(err, FUSE_ERR_TIMEOUT, SITE_GEMM_TIMEOUT, blockIdx.x);
}

__global__ void __launch_bounds__(kQpThreads, 1)
    qproj_tc_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX,
                    const QpArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  QpCtl* ctl = reinterpret_cast<QpCtl*>(smem + kQpStages * kQpStageBytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int head = blockIdx.x, row0 = blockIdx.y * kQpN, split = blockIdx.z;
  const int kb0 = split * a.steps_per_split;
  const int kb1 = min(a.k_steps, kb0 + a.steps_per_split);   // the host keeps every split non-empty
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kQpStages; ++s) {
      tc::mbar_init(&ctl->full[s], 1);
      tc::mbar_init(&ctl->empty[s], 1);
    }
    tc::mbar_init(&ctl->acc_full, 1);
    ctl->abort_flag = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&mapW);
    tc::tma_prefetch_desc(&mapX);
  }
  if (warp == 1) tc::tmem_alloc(&ctl->tmem_base, kQpTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_wait();                  // X is written by the previous kernel

  if (warp == 0 && lane == 0) {
    // ------------------------------ TMA loads ------------------------------
    int i = 0;
    for (int kb = kb0; kb < kb1; ++kb, ++i) {
      const int st = i % kQpStages;
      if (!tc::mbar_wait(&ctl->empty[st], ((i / kQpStages) & 1) ^ 1, &ctl->abort_flag)) {
        qp_abort(ctl, a.err);
        break;
      }
      uint8_t* w = smem + st * kQpStageBytes;
      tc::mbar_arrive_expect_tx(&ctl->full[st], kQpStageBytes);
      tc::tma_load_3d(w, &mapW, &ctl->full[st], kb * kQpK, head * kQpM, 0);
      tc::tma_load_3d(w + kQpWBytes, &mapX, &ctl->full[st], kb * kQpK, row0, 0);
    }
    // let copies in flight land before the CTA may exit
    for (int c = (i > kQpStages ? i - kQpStages : 0); c < i; ++c)
      tc::mbar_wait(&ctl->full[c % kQpStages], (c / kQpStages) & 1);
  } else if (warp == 1 && lane == 0) {
    // -------------------------------- MMAs ---------------------------------
    const uint32_t idesc = tc::idesc_bf16_f32(kQpM, kQpN);
    int i = 0;
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb, ++i) {
      const int st = i % kQpStages;
      if (!tc::mbar_wait(&ctl->full[st], (i / kQpStages) & 1, &ctl->abort_flag)) {
        qp_abort(ctl, a.err);
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const uint32_t w = tc::smem_u32(smem + st * kQpStageBytes);
#pragma unroll
      for (int kk = 0; kk < kQpK / 16; ++kk)
        tc::mma_bf16(tmem, tc::smem_desc_k128(w + kk * 32),
                     tc::smem_desc_k128(w + kQpWBytes + kk * 32), idesc, (i | kk) != 0);
      tc::mma_commit(&ctl->empty[st]);
    }
    if (ok) tc::mma_commit(&ctl->acc_full);
  }
  __syncwarp();

  // ------------------------------ epilogue ------------------------------
  // thread f (TMEM lane f) holds feature f of the head for the 64 rows
  if (tc::mbar_wait_warp(&ctl->acc_full, 0, &ctl->abort_flag)) {
    tc::tc_fence_after();
    const int f = warp * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    const int64_t cols = (int64_t)a.n_heads * kQpM;
#pragma unroll 1
    for (int c0 = 0; c0 < kQpN; c0 += 32) {
      uint32_t r[32];
      tc::tmem_ld_32x32b_x32(t_lane + c0, r);
      tc::tmem_ld_wait();
      float* dst = a.part + ((int64_t)split * a.n_rows + row0 + c0) * cols + head * kQpM + f;
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (row0 + c0 + c < a.n_rows) dst[c * cols] = __uint_as_float(r[c]);
    }
  } else if (threadIdx.x == 0) {
    qp_abort(ctl, a.err);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kQpTmemCols);
}

// Q[m, head] = RoPE(sum over splits of part[split][m][head]) in bf16: one
// block per (row, four heads), one thread per (head, rotation pair j); the
// splits' loads are all issued before the sum, which runs in split order.
__global__ void __launch_bounds__(256) qproj_sum_rope_kernel(const float* part, int k_splits,
                                                             int n_rows, int n_heads,
                                                             const float2* rope,
                                                             __nv_bfloat16* Q) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x;
  const int head = blockIdx.y * 4 + threadIdx.x / (kQpM / 2), j = threadIdx.x % (kQpM / 2);
  if (head >= n_heads) return;
  const int64_t cols = (int64_t)n_heads * kQpM;
  float xs[kQpMaxSplits], ys[kQpMaxSplits];
#pragma unroll
  for (int s = 0; s < kQpMaxSplits; ++s) {
    if (s < k_splits) {
      const float* p = part + ((int64_t)s * n_rows + m) * cols + head * kQpM;
      xs[s] = __ldg(p + j);
      ys[s] = __ldg(p + j + kQpM / 2);
    }
  }
  float x = 0.f, y = 0.f;
#pragma unroll
  for (int s = 0; s < kQpMaxSplits; ++s) {
    if (s < k_splits) {
      x += xs[s];
      y += ys[s];
    }
  }
  const float2 c = rope[rope_index(j, m, n_rows)];
  __nv_bfloat16* o = Q + ((int64_t)m * n_heads + head) * kQpM;
  o[j] = __float2bfloat16_rn(fmaf(x, c.x, -y * c.y));
  o[j + kQpM / 2] = __float2bfloat16_rn(fmaf(y, c.x, x * c.y));
}

int qp_sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

bool qproj_tc_supported(const fuse_layer_desc_t& d, int64_t n_rows) {
  return d.dtype == FUSE_BF16 && d.head_dim == kQpM && d.hidden % kQpK == 0 && n_rows > 0 &&
         n_rows <= kQpMaxRows && tma_encode_available();
}

// Q[m] = R^{pos_m} W_Q X[m] for the n_rows rows of X (bf16, hidden wide,
// gathered by the query-row preparation); part: room for max_splits *
// n_rows * Hq * 128 floats.
cudaError_t launch_qproj_tc(const fuse_layer_desc_t& d, int64_t n_rows, const float2* rope,
                            const void* Wq, const void* X, void* Q, float* part, int max_splits,
                            uint32_t* err, cudaStream_t s) {
  const int k_steps = d.hidden / kQpK;
  const int row_groups = (int)((n_rows + kQpN - 1) / kQpN);
  // splits: enough CTAs to cover the SMs, at least four stages each
  int ks = (qp_sm_count() + d.n_q_heads * row_groups - 1) / (d.n_q_heads * row_groups);
  ks = std::max(1, std::min({ks, kQpMaxSplits, max_splits, std::max(1, k_steps / 4)}));
  const int per = (k_steps + ks - 1) / ks;
  ks = (k_steps + per - 1) / per;                    // every split non-empty
  CUtensorMap mW, mX;
  const uint64_t dw[3] = {(uint64_t)d.hidden, (uint64_t)d.n_q_heads * kQpM, 1};
  const uint64_t sw[2] = {(uint64_t)d.hidden * 2, (uint64_t)d.hidden * 2 * d.n_q_heads * kQpM};
  const uint32_t bw[3] = {(uint32_t)kQpK, (uint32_t)kQpM, 1};
  const uint64_t dx[3] = {(uint64_t)d.hidden, (uint64_t)n_rows, 1};
  const uint64_t sx[2] = {(uint64_t)d.hidden * 2, (uint64_t)d.hidden * 2 * n_rows};
  const uint32_t bx[3] = {(uint32_t)kQpK, (uint32_t)kQpN, 1};
  if (!make_map_3d(&mW, Wq, dw, sw, bw) || !make_map_3d(&mX, X, dx, sx, bx))
    return cudaErrorInvalidValue;
  QpArgs a;
  a.n_rows = (int)n_rows;
  a.n_heads = d.n_q_heads;
  a.k_steps = k_steps;
  a.steps_per_split = per;
  a.part = part;
  a.err = err;
  cudaError_t e = set_dyn_smem_once(reinterpret_cast<const void*>(qproj_tc_kernel), kQpSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(qproj_tc_kernel, dim3(d.n_q_heads, row_groups, ks), dim3(kQpThreads),
                 kQpSmemBytes, s, mW, mX, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(qproj_sum_rope_kernel, dim3((unsigned)n_rows, (d.n_q_heads + 3) / 4),
                    dim3(256), 0, s, (const float*)part, ks, (int)n_rows, d.n_q_heads, rope,
                    reinterpret_cast<__nv_bfloat16*>(Q));
}

}  // namespace fusekv
