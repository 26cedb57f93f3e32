// Query-aware attention mass on tcgen05 tensor cores (bf16 layers, head_dim
// 128).
//
// QCFuse (section 3.2.1, Eqs. 9-10): context token t of a request scores the
// attention weight the user query puts on it,
//   I(t) = sum_{u < Qn} sum_h softmax_{t' < N}(q_{u,h} . Kf[t', h/g] / sqrt(d))[t].
// Per KV head, the query vectors that read it -- query token u and head
// h = kvh * g + hh, vector v = u * g + hh -- are cut into tiles of 128
// (128 / g tokens x g heads, the attention kernel's Q tile), the context keys
// into tiles of 128.  Each (vector tile, key tile) is one 128 x 128 x 128
// tcgen05.mma into TMEM, formed twice:
//   statistics pass  S = Q K^T (rows = vectors): each vector's running
//                    maximum and sum of 2^(S scale - max) over the CTA's key
//                    tiles -> stats[vector, chunk]
//   mass pass        first, per vector of the tile, over the chunks:
//                    c_v = max + log2(sum); then
//                    S^T = K Q^T (rows = keys): each key's sum over the tile's
//                    vectors of 2^(S scale - c_v), per 64-vector half ->
//                    part[key, kvh, vector tile, half]
//   reduce           score[t] (+)= sum over KV heads, vector tiles and halves,
//                    in order
// so no floating-point atomics.  A CTA takes one (request, KV head, vector
// tile) and a contiguous chunk of key tiles: warp 0 loads the Q tile once and
// the key tiles through a 2-stage ring (TMA, 128-byte swizzle), warp 1 issues
// the MMAs into two TMEM buffers, warps 2-9 read them (two warps per TMEM
// lane quarter, 64 columns each) while the next tile is formed.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace fusekv {

bool make_map_3d(CUtensorMap* m, const void* base, const uint64_t dims[3], const uint64_t strides[2],
                 const uint32_t box[3]);
bool tma_encode_available();

namespace {

constexpr int kD = 128;
constexpr int kT = 128;                        // keys per tile, vectors per tile
constexpr int kHalf = 128 * 64 * 2;            // one 64-column half of a tile (16 KB)
constexpr int kTile = 2 * kHalf;               // 32 KB
constexpr int kStages = 2;
constexpr int kThreads = 10 * 32;
constexpr int kEpi = 256;                      // epilogue threads (warps 2..9)
constexpr int kTmemCols = 256;                 // two S buffers
constexpr float kNegBig = -1.0e30f;

struct MassTcArgs {
  const fuse_request_t* reqs;
  const int32_t* qoff;     // first packed query row of each request
  int64_t n_qrows;         // packed query rows the host counted
  float2* stats;           // [n_qrows * Hq, n_chunks] (max, sum) per chunk
  float* part;             // [N_total, Hkv, n_vt, 2] mass per key, KV head, vector tile, half
  int Hq, Hkv, g, rtile;
  int n_vt;                // vector tiles per (request, KV head), maximum over requests
  int n_chunks;            // key-tile chunks per request
  float scale_log2;        // log2(e) / sqrt(d)
  uint32_t* err;
};

struct Ctl {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t s_full[2], s_empty[2];
  uint32_t tmem_base;
  volatile int abort_flag;
  float xa[128], xb[128];    // statistics: the second column half's (max, sum) per row
  float cv[128];             // mass pass: c_v of the tile's vectors
};
constexpr int kSmemBytes = (1 + kStages) * kTile + 1024 + (int)sizeof(Ctl);

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint64_t kmajor_step(uint32_t tile, int kk) {
  return tc::smem_desc_k128(tile + (kk >> 2) * kHalf + (kk & 3) * 32);
}

__device__ __forceinline__ void abort_mass(Ctl* ctl, uint32_t* err) {
  if (ctl->abort_flag == 0) report_error(err, FUSE_ERR_TIMEOUT, SITE_MASS_TIMEOUT, blockIdx.x);
  ctl->abort_flag = 1;
}

// The CTA's unit: request z, KV head y, vector tile and chunk of key tiles
// from x.  Returns false for a unit past the request's extent.
struct Unit {
  fuse_request_t R;
  int qoff, nv, vt, kvh, kt0, kt1;
};
__device__ __forceinline__ bool unit_of(const MassTcArgs& a, Unit& u) {
  u.R = a.reqs[blockIdx.z];
  u.kvh = blockIdx.y;
  u.vt = blockIdx.x / a.n_chunks;
  const int ch = blockIdx.x % a.n_chunks;
  u.qoff = a.qoff[blockIdx.z];
  // query vectors of the request (its packed rows stay below the host's count)
  const int64_t avail = u.qoff < 0 ? 0 : a.n_qrows - u.qoff;
  const int nq = (int)(avail <= 0 ? 0 : (u.R.n_query < avail ? u.R.n_query : avail));
  u.nv = nq * a.g;
  const int n_kt = (u.R.n_ctx + kT - 1) / kT;
  const int per = (n_kt + a.n_chunks - 1) / a.n_chunks;
  u.kt0 = ch * per;
  u.kt1 = min(n_kt, u.kt0 + per);
  return u.vt * kT < u.nv && u.kt0 < u.kt1;
}

template <bool MASS>
__global__ void __launch_bounds__(kThreads, 2)
    mass_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                   const MassTcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kTile;                   // stage s at sK + s * kTile
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (1 + kStages) * kTile);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  pdl_trigger();
  pdl_wait();                                   // Q, the offsets, the fused cache and c_v are complete
  Unit u;
  if (!unit_of(a, u)) return;                   // CTA-uniform, before any barrier
  const int n_tiles = u.kt1 - u.kt0;

  if (threadIdx.x == 0) {
    tc::mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&ctl->k_full[s], 1);
      tc::mbar_init(&ctl->k_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl->s_full[b], 1);
      tc::mbar_init(&ctl->s_empty[b], kEpi);
    }
    ctl->abort_flag = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&mapQ);
    tc::tma_prefetch_desc(&mapK);
  }
  if (warp == 1) tc::tmem_alloc(&ctl->tmem_base, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------ loads ------------------------------
    if (lane == 0) {
      const int qrow = u.qoff + u.vt * a.rtile;
      tc::mbar_arrive_expect_tx(&ctl->q_full, kTile);
      tc::tma_load_3d(sQ, &mapQ, &ctl->q_full, 0, u.kvh * a.g, qrow);
      tc::tma_load_3d(sQ + kHalf, &mapQ, &ctl->q_full, 64, u.kvh * a.g, qrow);
      int i = 0;
      for (; i < n_tiles; ++i) {
        const int st = i % kStages;
        if (!tc::mbar_wait(&ctl->k_empty[st], ((i / kStages) & 1) ^ 1, &ctl->abort_flag)) {
          abort_mass(ctl, a.err);
          break;
        }
        uint8_t* k = sK + st * kTile;
        const int z = (int)u.R.row0 + (u.kt0 + i) * kT;
        tc::mbar_arrive_expect_tx(&ctl->k_full[st], kTile);
        tc::tma_load_3d(k, &mapK, &ctl->k_full[st], 0, u.kvh, z);
        tc::tma_load_3d(k + kHalf, &mapK, &ctl->k_full[st], 64, u.kvh, z);
      }
      // copies in flight land before the CTA may exit
      tc::mbar_wait(&ctl->q_full, 0);
      for (int c = (i > kStages ? i - kStages : 0); c < i; ++c)
        tc::mbar_wait(&ctl->k_full[c % kStages], (c / kStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------ MMAs ------------------------------
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(128, kT);
      if (!tc::mbar_wait(&ctl->q_full, 0, &ctl->abort_flag)) {
        abort_mass(ctl, a.err);
      } else {
        const uint32_t qa = tc::smem_u32(sQ);
        for (int i = 0; i < n_tiles; ++i) {
          const int st = i % kStages, sb = i & 1;
          if (!tc::mbar_wait(&ctl->k_full[st], (i / kStages) & 1, &ctl->abort_flag) ||
              !tc::mbar_wait(&ctl->s_empty[sb], ((i >> 1) & 1) ^ 1, &ctl->abort_flag)) {
            abort_mass(ctl, a.err);
            break;
          }
          tc::tc_fence_after();
          const uint32_t ka = tc::smem_u32(sK + st * kTile);
          const uint32_t d = tmem + sb * kT;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            if (MASS)   // rows = keys, columns = vectors
              tc::mma_bf16(d, kmajor_step(ka, kk), kmajor_step(qa, kk), idesc, kk != 0);
            else        // rows = vectors, columns = keys
              tc::mma_bf16(d, kmajor_step(qa, kk), kmajor_step(ka, kk), idesc, kk != 0);
          }
          tc::mma_commit(&ctl->s_full[sb]);
          tc::mma_commit(&ctl->k_empty[st]);
        }
      }
    }
  } else {
    // ---------------------------- epilogue ----------------------------
    const int quarter = warp & 3;
    const int hf = (warp - 2) >> 2;               // column half
    const int row = quarter * 32 + lane;          // TMEM lane: vector (stats) or key (mass)
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sc = a.scale_log2;
    const int nvt = min(kT, u.nv - u.vt * kT);     // valid vectors of the tile
    if (MASS) {
      // c_v = m + log2(l) of the tile's vectors from their chunks' (max, sum)
      // (+inf past the request's vectors, or without context: weight 0)
      if (threadIdx.x - 64 < 128) {
        const int v = threadIdx.x - 64;
        float c = INFINITY;
        if (v < nvt) {
          const int vv = u.vt * kT + v;
          const int64_t vec = ((int64_t)u.qoff + vv / a.g) * a.Hq + u.kvh * a.g + vv % a.g;
          const int n_kt = (u.R.n_ctx + kT - 1) / kT;
          const int per = (n_kt + a.n_chunks - 1) / a.n_chunks;
          const int nc = (n_kt + per - 1) / per;
          const float2* st = a.stats + vec * a.n_chunks;
          float m = kNegBig;
          for (int i = 0; i < nc; ++i) m = fmaxf(m, st[i].x);
          float l = 0.f;
          for (int i = 0; i < nc; ++i) l += st[i].y * ex2(st[i].x - m);
          c = l > 0.f ? m + log2f(l) : INFINITY;
        }
        ctl->cv[v] = c;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kEpi) : "memory");
    }
    float m_run = kNegBig, l_run = 0.f;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int sb = i & 1;
      if (!tc::mbar_wait_warp(&ctl->s_full[sb], (i >> 1) & 1, &ctl->abort_flag)) {
        abort_mass(ctl, a.err);
        ok = false;
        break;
      }
      tc::tc_fence_after();
      uint32_t r[64];
      const uint32_t ts = tmem + lane_off + sb * kT + hf * 64;
      tc::tmem_ld_32x32b_x32(ts, *reinterpret_cast<uint32_t(*)[32]>(r));
      tc::tmem_ld_32x32b_x32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
      tc::tmem_ld_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(&ctl->s_empty[sb]);
      const int kt = u.kt0 + i;
      if (!MASS) {
        // columns are keys: those past the context are masked
        const int nk = min(kT, u.R.n_ctx - kt * kT) - hf * 64;
        float mx = kNegBig;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < nk) mx = fmaxf(mx, __uint_as_float(r[c]));
        const float mn = fmaxf(m_run, mx * sc);
        float l = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < nk) l += ex2(fmaf(__uint_as_float(r[c]), sc, -mn));
        l_run = l_run * ex2(m_run - mn) + l;
        m_run = mn;
      } else {
        // columns are vectors: weight 2^(s scale - c_v), summed per key over
        // this thread's 64 vectors (the two halves are added by the reduce)
        float l = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          l += ex2(fmaf(__uint_as_float(r[c]), sc, -ctl->cv[hf * 64 + c]));
        const int key = kt * kT + row;
        if (key < u.R.n_ctx)
          a.part[(((u.R.score0 + key) * a.Hkv + u.kvh) * a.n_vt + u.vt) * 2 + hf] = l;
      }
    }
    if (!MASS) {
      // the vector's (max, sum) over this chunk: the two halves combined (every
      // epilogue warp reaches this barrier, also after a failed wait)
      if (hf == 1) {
        ctl->xa[row] = m_run;
        ctl->xb[row] = l_run;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kEpi) : "memory");
      if (ok && hf == 0 && row < nvt) {
        const float m1 = ctl->xa[row], l1 = ctl->xb[row];
        const float m = fmaxf(m_run, m1);
        const float l = l_run * ex2(m_run - m) + l1 * ex2(m1 - m);
        const int vv = u.vt * kT + row;
        const int64_t vec = ((int64_t)u.qoff + vv / a.g) * a.Hq + u.kvh * a.g + vv % a.g;
        a.stats[vec * a.n_chunks + blockIdx.x % a.n_chunks] = make_float2(m, l);
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// score[score0 + t] (+)= sum over KV heads, then vector tiles, of part.
__global__ void mass_tc_reduce_kernel(const fuse_request_t* reqs, const int32_t* qoff,
                                      int64_t n_qrows, const float* part, int Hkv, int g,
                                      int n_vt, float* score, int accumulate) {
  pdl_trigger();
  pdl_wait();
  const fuse_request_t R = reqs[blockIdx.y];
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= R.n_ctx) return;
  const int64_t avail = qoff[blockIdx.y] < 0 ? 0 : n_qrows - qoff[blockIdx.y];
  const int nq = (int)(avail <= 0 ? 0 : (R.n_query < avail ? R.n_query : avail));
  const int nvt = (nq * g + kT - 1) / kT;
  const float* p = part + (R.score0 + t) * (int64_t)Hkv * n_vt * 2;
  float s = 0.f;
  if ((n_vt & 1) == 0) {
    // a token's 2 * Hkv * n_vt values, four to a 16-byte load, sixteen loads
    // issued before their sums (the same additions in the same order)
    const int nq = Hkv * n_vt / 2;
    const int per = n_vt / 2;               // float4 per KV head
    for (int i0 = 0; i0 < nq; i0 += 16) {
      float4 q[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i0 + i < nq) q[i] = __ldg(reinterpret_cast<const float4*>(p) + i0 + i);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i0 + i >= nq) break;
        const int v4 = (i0 + i) % per;      // values 4 v4 .. 4 v4 + 3 of head (i0 + i) / per
        if (4 * v4 < 2 * nvt) s += q[i].x;
        if (4 * v4 + 1 < 2 * nvt) s += q[i].y;
        if (4 * v4 + 2 < 2 * nvt) s += q[i].z;
        if (4 * v4 + 3 < 2 * nvt) s += q[i].w;
      }
    }
  } else {
    for (int h = 0; h < Hkv; ++h)
      for (int v = 0; v < 2 * nvt; ++v) s += p[h * n_vt * 2 + v];
  }
  float* o = score + R.score0 + t;
  *o = accumulate ? *o + s : s;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

bool mass_tc_supported(const fuse_layer_desc_t& d) {
  const int g = d.n_q_heads / d.n_kv_heads;
  return d.dtype == FUSE_BF16 && d.head_dim == kD && (g == 1 || g == 2 || g == 4 || g == 8) &&
         tma_encode_available();
}

// Chunks of key tiles per (request, KV head, vector tile): the count whose
// units fill the device's CTA slots (two per SM) in the fewest tile-steps.
int mass_tc_chunks(const fuse_layer_desc_t& d, const fuse_requests_t& reqs, int max_ctx,
                   int max_query) {
  const int g = d.n_q_heads / d.n_kv_heads;
  const int n_kt = (max_ctx + kT - 1) / kT;
  if (n_kt == 0) return 1;
  int64_t vt_total = 0;
  for (int r = 0; r < reqs.n_req; ++r)
    vt_total += ((int64_t)reqs.h_req[r].n_query * g + kT - 1) / kT;
  (void)max_query;
  const int64_t slots = 2 * (int64_t)sm_count();
  int best = 1;
  int64_t best_cost = INT64_MAX;
  for (int nc = 1; nc <= n_kt; ++nc) {
    const int per = (n_kt + nc - 1) / nc;
    const int used = (n_kt + per - 1) / per;
    const int64_t units = vt_total * d.n_kv_heads * used;
    const int64_t cost = ((units + slots - 1) / slots) * per + 1;   // + a unit's set-up
    if (cost < best_cost) {
      best_cost = cost;
      best = used;
    }
  }
  return best;
}

cudaError_t launch_attention_mass_tc(const fuse_layer_desc_t& d, const fuse_requests_t& reqs,
                                     int max_ctx, int max_query, int64_t n_qrows, int64_t n_tok,
                                     const int32_t* qoff, const void* Q, const void* Kf,
                                     float2* stats, float* part, int n_chunks, float* score,
                                     int accumulate, uint32_t* err, cudaStream_t s) {
  if (reqs.n_req == 0 || max_ctx == 0) return cudaSuccess;
  const int g = d.n_q_heads / d.n_kv_heads;
  MassTcArgs a;
  a.reqs = reqs.d_req;
  a.qoff = qoff;
  a.n_qrows = n_qrows;
  a.stats = stats;
  a.part = part;
  a.Hq = d.n_q_heads;
  a.Hkv = d.n_kv_heads;
  a.g = g;
  a.rtile = kT / g;
  a.n_vt = (int)std::max<int64_t>(1, ((int64_t)max_query * g + kT - 1) / kT);
  a.n_chunks = n_chunks;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)kD));
  a.err = err;
  cudaError_t e;
  if (n_qrows > 0) {
    CUtensorMap mQ, mK;
    const uint64_t dq[3] = {(uint64_t)kD, (uint64_t)d.n_q_heads, (uint64_t)n_qrows};
    const uint64_t sq[2] = {(uint64_t)kD * 2, (uint64_t)d.n_q_heads * kD * 2};
    const uint32_t bq[3] = {64, (uint32_t)g, (uint32_t)(kT / g)};
    const uint64_t dk[3] = {(uint64_t)kD, (uint64_t)d.n_kv_heads, (uint64_t)n_tok};
    const uint64_t sk[2] = {(uint64_t)kD * 2, (uint64_t)d.n_kv_heads * kD * 2};
    const uint32_t bk[3] = {64, 1, (uint32_t)kT};
    if (!make_map_3d(&mQ, Q, dq, sq, bq) || !make_map_3d(&mK, Kf, dk, sk, bk))
      return cudaErrorInvalidValue;
    e = set_dyn_smem_once(reinterpret_cast<const void*>(mass_tc_kernel<false>), kSmemBytes);
    if (e == cudaSuccess)
      e = set_dyn_smem_once(reinterpret_cast<const void*>(mass_tc_kernel<true>), kSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid(a.n_vt * n_chunks, d.n_kv_heads, reqs.n_req);
    e = launch_pdl(mass_tc_kernel<false>, grid, dim3(kThreads), kSmemBytes, s, mQ, mK, a);
    if (e != cudaSuccess) return e;
    e = launch_pdl(mass_tc_kernel<true>, grid, dim3(kThreads), kSmemBytes, s, mQ, mK, a);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(mass_tc_reduce_kernel, dim3((unsigned)((max_ctx + 255) / 256), reqs.n_req),
                    dim3(256), 0, s, reqs.d_req, qoff, n_qrows, (const float*)part, d.n_kv_heads,
                    g, a.n_vt, score, accumulate);
}

}  // namespace fusekv
