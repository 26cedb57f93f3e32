// Sparse-query causal GQA attention on tcgen05 tensor cores (bf16 layers,
// head_dim 128).
//
// QCFuse (section 2.1.3, Eq. 6): every recomputed row at position p reads the
// fused cache at positions j <= p.  KVBoost (section 3.1, Eq. 2):
// softmax(q K^T / sqrt(d)) V.
//
// Work unit: one KV head and a tile of 128 / g consecutive recomputed rows of
// one request, whose g query heads share that KV head, packed as the M = 128
// rows of the MMA (row r, head hh -> M row r * g + hh).  Keys stream in
// blocks of 128 up to the tile's last position.  Per block b of unit i:
//   S = Q K_b^T          tcgen05.mma into TMEM buffer b & 1 (columns
//                        [128 (b & 1), 128 (b & 1) + 128)), so the next
//                        block's scores are formed during this block's softmax
//   P = 2^(S - m)        one warpgroup, each thread one M row and all 128 keys:
//                        a pass for the row maximum, a pass for the
//                        probabilities, written back as bf16 over S
//   O_i += P V_b         tcgen05.mma with A = P in TMEM, V read from shared
//                        memory as an MN-major operand, O in TMEM buffer i & 1
//                        (columns [256 + 128 (i & 1), ...))
// The running maximum m is raised only when a block exceeds it by more than
// 2^8 (then O and the running sum l are rescaled).  A second warpgroup writes
// O / l of unit i while the first works on unit i + 1.
// Roles, each behind its own mbarriers: warp 0 loads Q and K blocks (3-stage
// ring), warp 2 V blocks (2-stage ring), warp 1 issues the S MMAs, warp 3 the
// P.V MMAs, warps 4-7 the softmax, warps 8-11 the output.  Every role reads
// the unit's tile record (first output row, first fused row, rows, key
// blocks) one unit ahead.  The kernel is persistent; units are taken heaviest
// first, snake-ordered over the CTAs (round r visits the CTAs upwards when r
// is even and downwards when r is odd).
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace fusekv {

bool tma_encode_available();
bool make_map_3d(CUtensorMap* m, const void* base, const uint64_t dims[3], const uint64_t strides[2],
                 const uint32_t box[3]);

namespace {

constexpr int kD = 128;
constexpr int kKB = 128;                      // keys per block
constexpr int kHalf = 128 * 64 * 2;           // one 64-column half of a 128-row tile (16 KB)
constexpr int kTile = 2 * kHalf;              // 32 KB
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kWarpQK = 0, kWarpS = 1, kWarpV = 2, kWarpPV = 3, kWarpSoft = 4, kWarpOut = 8;
constexpr int kThreads = 12 * 32;             // 3 warps per SM sub-partition: up to 168 registers
constexpr int kTmemCols = 512;                // S0 | S1 | O0 | O1
constexpr int kColO = 256;
constexpr float kRescaleThreshold = 8.0f;     // log2 units
// Reference maximum of a row none of whose keys so far was visible (log2
// units): above every masked score (-1e30 * scale) and below every real one,
// so masked probabilities are exactly 0 and the first visible block rescales
// by 2^(floor - m) = 0.
constexpr float kFloor = -1.0e29f;


struct AttnArgs {
  const int4* tiles;      // (first output row, request's first fused row, rows, key blocks)
  int n_tiles;
  int n_units;
  const fuse_request_t* reqs;
  const WorkRow* rows;
  __nv_bfloat16* O;
  int Hq, Hkv, g, rtile;
  float scale_log2;       // log2(e) / sqrt(d)
  uint32_t* err;
};

struct Ctl {
  uint64_t q_full, q_empty;
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], p_full[2], pv_done[2];   // [block parity]
  uint64_t o_full[2], o_empty[2], l_full[2];   // [unit parity]
  uint32_t tmem_base;
  volatile int abort_flag;
  float xl[2][128];       // [unit parity][row] softmax row sum
};
constexpr int kSmemBytes = (1 + kKStages + kVStages) * kTile + 1024 + (int)sizeof(Ctl);
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Ctl* ctl) {
  return tc::mbar_wait(bar, parity, &ctl->abort_flag);
}

// Waits of warps that go on to warp-collective instructions.
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t* bar, uint32_t parity, Ctl* ctl) {
  return tc::mbar_wait_warp(bar, parity, &ctl->abort_flag);
}

// Which wait gave up: info = wait id (4 bits) << 20 | CTA (8 bits) << 12 | key block (12 bits).
enum AttnWait : uint32_t {
  W_Q_EMPTY = 1, W_K_EMPTY, W_V_EMPTY, W_Q_FULL, W_K_FULL, W_S_FREE, W_P_FULL, W_O_EMPTY,
  W_V_FULL, W_S_FULL, W_PV_DONE, W_O_FULL, W_L_FULL, W_L_FREE
};

__device__ __forceinline__ void abort_kernel(Ctl* ctl, uint32_t* err, uint32_t which = 0,
                                             int j = 0) {
  const bool first = ctl->abort_flag == 0;
  ctl->abort_flag = 1;
  if (first)
    report_error(err, FUSE_ERR_TIMEOUT, SITE_ATTN_TIMEOUT,
                 (which << 20) | ((blockIdx.x & 0xFFu) << 12) | ((uint32_t)j & 0xFFFu));
}

// The i-th unit of this CTA: round i visits CTAs upwards when i is even and
// downwards when i is odd.  Units past the end stay past it in later rounds.
__device__ __forceinline__ int unit_at(int i) {
  const int G = gridDim.x;
  return i * G + ((i & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

// Tile record of unit u (heaviest tiles, the last ones, first).
__device__ __forceinline__ int4 tile_of(const AttnArgs& a, int u) {
  return a.tiles[a.n_tiles - 1 - u / a.Hkv];
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// descriptor of K-step kk (16 columns) of a 128-row K-major tile stored as two
// 64-column halves
__device__ __forceinline__ uint64_t kmajor_step(uint32_t tile, int kk) {
  return tc::smem_desc_k128(tile + (kk >> 2) * kHalf + (kk & 3) * 32);
}

// Maximum of 32 scores, masked (-1e30) past position p when `mask`.
__device__ __forceinline__ float masked_max32(const uint32_t (&r)[32], bool mask, int key0, int p) {
  float v[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const float x = __uint_as_float(r[c]);
    v[c] = (mask && key0 + c > p) ? -1e30f : x;
  }
  float t[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) t[i] = max3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  t[10] = fmaxf(v[30], v[31]);
  const float u0 = max3(t[0], t[1], t[2]), u1 = max3(t[3], t[4], t[5]);
  const float u2 = max3(t[6], t[7], t[8]), u3 = fmaxf(t[9], t[10]);
  return fmaxf(max3(u0, u1, u2), u3);
}

// 32 probabilities 2^(s * scale - m) (0 past position p when `mask`) packed as
// bf16 pairs; returns their sum.
__device__ __forceinline__ float probs32(const uint32_t (&r)[32], bool mask, int key0, int p,
                                         float scale, float neg_m, uint32_t (&pk)[16]) {
  float e[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const float x = (mask && key0 + c > p) ? -1e30f : __uint_as_float(r[c]);
    e[c] = ex2(fmaf(x, scale, neg_m));
  }
#pragma unroll
  for (int c = 0; c < 32; c += 2) pk[c / 2] = pack_bf16x2(e[c], e[c + 1]);
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) e[i] += e[i + w];
  return e[0];
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                   const __grid_constant__ CUtensorMap mapV, const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kTile;                       // K stage s at sK + s * kTile
  uint8_t* sV = sK + kKStages * kTile;              // V stage s at sV + s * kTile
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (1 + kKStages + kVStages) * kTile);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    tc::mbar_init(&ctl->q_full, 1);
    tc::mbar_init(&ctl->q_empty, 1);
    for (int s = 0; s < kKStages; ++s) {
      tc::mbar_init(&ctl->k_full[s], 1);
      tc::mbar_init(&ctl->k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      tc::mbar_init(&ctl->v_full[s], 1);
      tc::mbar_init(&ctl->v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&ctl->s_full[s], 1);
      tc::mbar_init(&ctl->p_full[s], 128);
      tc::mbar_init(&ctl->pv_done[s], 1);
      tc::mbar_init(&ctl->o_full[s], 1);
      tc::mbar_init(&ctl->o_empty[s], 128);
      tc::mbar_init(&ctl->l_full[s], 128);
    }
    ctl->abort_flag = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&mapQ);
    tc::tma_prefetch_desc(&mapK);
    tc::tma_prefetch_desc(&mapV);
  }
  if (warp == kWarpS) tc::tmem_alloc(&ctl->tmem_base, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int n_units = a.n_units;

  if (warp == kWarpQK) {
    // --------------------------- Q and K loads ---------------------------
    if (lane == 0) {
      uint32_t kc = 0;
      int i = 0;
      bool ok = true;
      int4 T = unit_at(0) < n_units ? tile_of(a, unit_at(0)) : make_int4(0, 0, 0, 0);
      for (; unit_at(i) < n_units && ok; ++i) {
        const int u = unit_at(i);
        const int4 cur = T;
        if (unit_at(i + 1) < n_units) T = tile_of(a, unit_at(i + 1));   // next unit's record
        const int kvh = u % a.Hkv;
        if (!wait_or_abort(&ctl->q_empty, (i & 1) ^ 1, ctl)) {
          abort_kernel(ctl, a.err, W_Q_EMPTY, 0);
          break;
        }
        tc::mbar_arrive_expect_tx(&ctl->q_full, kTile);
        tc::tma_load_3d(sQ, &mapQ, &ctl->q_full, 0, kvh * a.g, cur.x);
        tc::tma_load_3d(sQ + kHalf, &mapQ, &ctl->q_full, 64, kvh * a.g, cur.x);
        for (int j = 0; j < cur.w; ++j, ++kc) {
          const int st = kc % kKStages;
          if (!wait_or_abort(&ctl->k_empty[st], ((kc / kKStages) & 1) ^ 1, ctl)) {
            abort_kernel(ctl, a.err, W_K_EMPTY, j);
            ok = false;
            break;
          }
          uint8_t* k = sK + st * kTile;
          const int z = cur.y + j * kKB;
          tc::mbar_arrive_expect_tx(&ctl->k_full[st], kTile);
          tc::tma_load_3d(k, &mapK, &ctl->k_full[st], 0, kvh, z);
          tc::tma_load_3d(k + kHalf, &mapK, &ctl->k_full[st], 64, kvh, z);
        }
      }
      // let copies in flight land before the CTA may exit
      if (i > 0) tc::mbar_wait(&ctl->q_full, (i - 1) & 1);
      for (uint32_t c = (kc > (uint32_t)kKStages ? kc - kKStages : 0); c < kc; ++c)
        tc::mbar_wait(&ctl->k_full[c % kKStages], (c / kKStages) & 1);
    }
  } else if (warp == kWarpV) {
    // ------------------------------ V loads ------------------------------
    if (lane == 0) {
      uint32_t vc = 0;
      bool ok = true;
      int4 T = unit_at(0) < n_units ? tile_of(a, unit_at(0)) : make_int4(0, 0, 0, 0);
      for (int i = 0; unit_at(i) < n_units && ok; ++i) {
        const int u = unit_at(i);
        const int4 cur = T;
        if (unit_at(i + 1) < n_units) T = tile_of(a, unit_at(i + 1));
        const int kvh = u % a.Hkv;
        for (int j = 0; j < cur.w; ++j, ++vc) {
          const int st = vc % kVStages;
          if (!wait_or_abort(&ctl->v_empty[st], ((vc / kVStages) & 1) ^ 1, ctl)) {
            abort_kernel(ctl, a.err, W_V_EMPTY, j);
            ok = false;
            break;
          }
          uint8_t* v = sV + st * kTile;
          const int z = cur.y + j * kKB;
          tc::mbar_arrive_expect_tx(&ctl->v_full[st], kTile);
          tc::tma_load_3d(v, &mapV, &ctl->v_full[st], 0, kvh, z);
          tc::tma_load_3d(v + kHalf, &mapV, &ctl->v_full[st], 64, kvh, z);
        }
      }
      for (uint32_t c = (vc > (uint32_t)kVStages ? vc - kVStages : 0); c < vc; ++c)
        tc::mbar_wait(&ctl->v_full[c % kVStages], (c / kVStages) & 1);
    }
  } else if (warp == kWarpS) {
    // ------------------------------ S = Q K^T ------------------------------
    if (lane == 0) {
      const uint32_t idesc_s = tc::idesc_bf16_f32(128, kKB);
      const uint32_t q_addr = tc::smem_u32(sQ);
      uint32_t kc = 0, b = 0;
      bool ok = true;
      int4 T = unit_at(0) < n_units ? tile_of(a, unit_at(0)) : make_int4(0, 0, 0, 0);
      for (int i = 0; unit_at(i) < n_units && ok; ++i) {
        const int nkb = T.w;
        if (unit_at(i + 1) < n_units) T = tile_of(a, unit_at(i + 1));
        if (!wait_or_abort(&ctl->q_full, i & 1, ctl)) {
          abort_kernel(ctl, a.err, W_Q_FULL, 0);
          break;
        }
        for (int j = 0; j < nkb; ++j, ++kc, ++b) {
          const int st = kc % kKStages;
          if (!wait_or_abort(&ctl->k_full[st], (kc / kKStages) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_K_FULL, j);
            ok = false;
            break;
          }
          // buffer b & 1 holds P of block b - 2 until that block's P.V is done
          if (!wait_or_abort(&ctl->pv_done[b & 1], ((b >> 1) & 1) ^ 1, ctl)) {
            abort_kernel(ctl, a.err, W_S_FREE, j);
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t kaddr = tc::smem_u32(sK + st * kTile);
          const uint32_t d = tmem + (b & 1) * kKB;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            tc::mma_bf16(d, kmajor_step(q_addr, kk), kmajor_step(kaddr, kk), idesc_s, kk != 0);
          tc::mma_commit(&ctl->s_full[b & 1]);
          tc::mma_commit(&ctl->k_empty[st]);
        }
        if (!ok) break;
        tc::mma_commit(&ctl->q_empty);
      }
    }
  } else if (warp == kWarpPV) {
    // ------------------------------ O_i += P V ------------------------------
    if (lane == 0) {
      const uint32_t idesc_o = tc::idesc_bf16_f32(128, kD, /*b_mn_major=*/true);
      uint32_t vc = 0, b = 0;
      bool ok = true;
      int4 T = unit_at(0) < n_units ? tile_of(a, unit_at(0)) : make_int4(0, 0, 0, 0);
      for (int i = 0; unit_at(i) < n_units && ok; ++i) {
        const int nkb = T.w;
        if (unit_at(i + 1) < n_units) T = tile_of(a, unit_at(i + 1));
        const uint32_t o = tmem + kColO + (i & 1) * kD;
        // O_(i & 1) was last read by the output warps for unit i - 2
        if (!wait_or_abort(&ctl->o_empty[i & 1], ((i >> 1) & 1) ^ 1, ctl)) {
          abort_kernel(ctl, a.err, W_O_EMPTY, 0);
          break;
        }
        for (int j = 0; j < nkb; ++j, ++vc, ++b) {
          if (!wait_or_abort(&ctl->p_full[b & 1], (b >> 1) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_P_FULL, j);
            ok = false;
            break;
          }
          const int st = vc % kVStages;
          if (!wait_or_abort(&ctl->v_full[st], (vc / kVStages) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_V_FULL, j);
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t vaddr = tc::smem_u32(sV + st * kTile);
          const uint32_t pa = tmem + (b & 1) * kKB;
#pragma unroll
          for (int kk = 0; kk < kKB / 16; ++kk)
            tc::mma_bf16_ts(o, pa + kk * 8, tc::smem_desc_mn128(vaddr + kk * 16 * 128, kHalf),
                            idesc_o, (j | kk) != 0 ? 1u : 0u);
          tc::mma_commit(&ctl->pv_done[b & 1]);
          tc::mma_commit(&ctl->v_empty[st]);
        }
        if (!ok) break;
        tc::mma_commit(&ctl->o_full[i & 1]);
      }
    }
  } else if (warp < kWarpOut) {
    // ------------------------------- softmax -------------------------------
    const int quarter = warp & 3;                      // TMEM lane quarter
    const int m = quarter * 32 + lane;                 // M row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float scale = a.scale_log2;
    const int rl = m / a.g;
    uint32_t b = 0;
    // this unit's record and positions, read one unit ahead
    int4 T = unit_at(0) < n_units ? tile_of(a, unit_at(0)) : make_int4(0, 0, 1, 0);
    int p_next = 0, pf_next = 0;
    if (unit_at(0) < n_units) {
      p_next = a.rows[T.x + min(rl, T.z - 1)].pos;
      pf_next = a.rows[T.x].pos;
    }
    for (int i = 0; unit_at(i) < n_units; ++i) {
      const int nkb = T.w;
      const int p = p_next;
      const int p_first = pf_next;                     // rows ascend: the tile's smallest
      const bool more = unit_at(i + 1) < n_units;
      if (more) T = tile_of(a, unit_at(i + 1));
      const uint32_t tO = tmem + lane_off + kColO + (i & 1) * kD;
      float mu = kFloor, l = 0.f;                      // running max (log2 units), sum
      bool ok = true;
      for (int j = 0; j < nkb; ++j, ++b) {
        if (!warp_wait_or_abort(&ctl->s_full[b & 1], (b >> 1) & 1, ctl)) {
          abort_kernel(ctl, a.err, W_S_FULL, j);
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t tS = tmem + lane_off + (b & 1) * kKB;
        const int key0 = j * kKB;
        const bool mask = key0 + kKB - 1 > p_first;     // warp-uniform
        // the whole row of scores in registers: one TMEM round trip
        uint32_t r[128];
        tc::tmem_ld_32x32b_x32(tS, *reinterpret_cast<uint32_t(*)[32]>(r));
        tc::tmem_ld_32x32b_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tc::tmem_ld_32x32b_x32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(r + 64));
        tc::tmem_ld_32x32b_x32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(r + 96));
        tc::tmem_ld_wait();
        if (mask) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (key0 + c > p) r[c] = __float_as_uint(-1e30f);
        }
        float mx;
        {                                              // four running maxima, then one
          float t0 = __uint_as_float(r[0]), t1 = __uint_as_float(r[1]);
          float t2 = __uint_as_float(r[2]), t3 = __uint_as_float(r[3]);
#pragma unroll
          for (int q = 4; q < 128; q += 8) {
            t0 = max3(t0, __uint_as_float(r[q]), __uint_as_float(r[q + 4]));
            t1 = max3(t1, __uint_as_float(r[q + 1]), __uint_as_float(r[q + 5]));
            t2 = max3(t2, __uint_as_float(r[q + 2]), __uint_as_float(r[q + 6]));
            t3 = max3(t3, __uint_as_float(r[q + 3]), __uint_as_float(r[q + 7]));
          }
          t0 = max3(t0, __uint_as_float(r[124]), __uint_as_float(r[125]));
          t1 = max3(t1, __uint_as_float(r[126]), __uint_as_float(r[127]));
          mx = fmaxf(max3(t0, t1, t2), t3);
        }
        const float mxs = mx * scale;
        float mnew = mu;
        bool rescale = false;
        if (j == 0) {
          mnew = fmaxf(mxs, kFloor);
        } else if (mxs > mu + kRescaleThreshold) {
          mnew = mxs;
          rescale = true;
        }
        const float alpha = rescale ? ex2(mu - mnew) : 1.f;
        // probabilities, written as bf16 over the scores
        const float neg = -mnew;
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
          float e[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) e[q] = ex2(fmaf(__uint_as_float(r[32 * c + q]), scale, neg));
#pragma unroll
          for (int q = 0; q < 32; q += 2) pk[q / 2] = pack_bf16x2(e[q], e[q + 1]);
#pragma unroll
          for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
            for (int q = 0; q < w; ++q) e[q] += e[q + w];
          sum += e[0];
          tc::tmem_st_32x32b_x16(tS + 16 * c, pk);
        }
        // tcgen05.ld/st are warp-collective (.sync.aligned): the whole warp
        // rescales its rows of O when any of them needs it (alpha is 1 for the
        // others); O must hold the previous block's P.V
        if (__any_sync(0xffffffffu, rescale)) {
          if (!warp_wait_or_abort(&ctl->pv_done[(b - 1) & 1], ((b - 1) >> 1) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_PV_DONE, j);
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kD; c += 32) {
            uint32_t o[32];
            tc::tmem_ld_32x32b_x32(tO + c, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
            tc::tmem_st_32x32b_x32(tO + c, o);
          }
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(&ctl->p_full[b & 1]);
        l = l * alpha + sum;
        mu = mnew;
      }
      if (!ok) break;
      if (more) {
        p_next = a.rows[T.x + min(rl, T.z - 1)].pos;
        pf_next = a.rows[T.x].pos;
      }
      // the row sum of unit i, once the output warps have read that of unit i - 2
      if (!warp_wait_or_abort(&ctl->o_empty[i & 1], ((i >> 1) & 1) ^ 1, ctl)) {
        abort_kernel(ctl, a.err, W_L_FREE, nkb);
        break;
      }
      ctl->xl[i & 1][m] = l;
      tc::mbar_arrive(&ctl->l_full[i & 1]);
    }
  } else {
    // ---------------------------- output O / l ----------------------------
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int rl = m / a.g;
    const int hh = m % a.g;
    int4 T = unit_at(0) < n_units ? tile_of(a, unit_at(0)) : make_int4(0, 0, 0, 0);
    for (int i = 0; unit_at(i) < n_units; ++i) {
      const int u = unit_at(i);
      const int4 cur = T;
      if (unit_at(i + 1) < n_units) T = tile_of(a, unit_at(i + 1));
      const int kvh = u % a.Hkv;
      if (!warp_wait_or_abort(&ctl->o_full[i & 1], (i >> 1) & 1, ctl)) {
        abort_kernel(ctl, a.err, W_O_FULL, cur.w);
        break;
      }
      if (!warp_wait_or_abort(&ctl->l_full[i & 1], (i >> 1) & 1, ctl)) {
        abort_kernel(ctl, a.err, W_L_FULL, cur.w);
        break;
      }
      tc::tc_fence_after();
      const float inv = 1.f / ctl->xl[i & 1][m];
      const bool valid = rl < cur.z;
      __nv_bfloat16* dst = a.O + ((int64_t)(cur.x + rl) * a.Hq + kvh * a.g + hh) * kD;
      const uint32_t tO = tmem + lane_off + kColO + (i & 1) * kD;
#pragma unroll 1
      for (int c = 0; c < kD; c += 32) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tO + c, r);
        tc::tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * inv, __uint_as_float(r[8 * q + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv, __uint_as_float(r[8 * q + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv, __uint_as_float(r[8 * q + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv, __uint_as_float(r[8 * q + 7]) * inv);
            reinterpret_cast<uint4*>(dst + c)[q] = w;
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&ctl->o_empty[i & 1]);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kWarpS) tc::tmem_dealloc(tmem, kTmemCols);
}

__global__ void attn_tiles_kernel(const fuse_request_t* reqs, int n_req, const int32_t* idx,
                                  int rtile, int4* tiles) {
  build_attn_tiles(reqs, n_req, idx, rtile, tiles);
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

int attention_rtile(const fuse_layer_desc_t& d) { return 128 / (d.n_q_heads / d.n_kv_heads); }

size_t attention_tiles_bytes(int64_t n_out, int n_req) {
  return (size_t)(n_out / 16 + n_req + 1) * sizeof(int4);
}

bool tc_attention_supported(const fuse_layer_desc_t& d) {
  const int g = d.n_q_heads / d.n_kv_heads;
  return d.dtype == FUSE_BF16 && d.head_dim == kD && (g == 1 || g == 2 || g == 4 || g == 8) &&
         tma_encode_available();
}

cudaError_t launch_attention_tc(const fuse_layer_desc_t& d, const fuse_requests_t& reqs,
                                int64_t n_out, int64_t n_tok, const WorkRow* rows,
                                const int32_t* idx, const void* Q, const void* Kf, const void* Vf,
                                void* O, void* tiles_ws, bool tiles_ready, uint32_t* err,
                                cudaStream_t s) {
  const int g = d.n_q_heads / d.n_kv_heads;
  const int rtile = 128 / g;
  int n_tiles = 0;
  for (int r = 0; r < reqs.n_req; ++r) {
    const int R = reqs.h_req[r].k + reqs.h_req[r].n_query;
    n_tiles += (R + rtile - 1) / rtile;
  }
  if (n_tiles == 0) return cudaSuccess;
  int4* tiles = reinterpret_cast<int4*>(tiles_ws);
  cudaError_t e = cudaSuccess;
  if (!tiles_ready) {
    attn_tiles_kernel<<<1, 128, 0, s>>>(reqs.d_req, reqs.n_req, idx, rtile, tiles);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }

  CUtensorMap mQ, mK, mV;
  const uint64_t dq[3] = {(uint64_t)kD, (uint64_t)d.n_q_heads, (uint64_t)n_out};
  const uint64_t sq[2] = {(uint64_t)kD * 2, (uint64_t)d.n_q_heads * kD * 2};
  const uint32_t bq[3] = {64, (uint32_t)g, (uint32_t)rtile};
  const uint64_t dk[3] = {(uint64_t)kD, (uint64_t)d.n_kv_heads, (uint64_t)n_tok};
  const uint64_t sk[2] = {(uint64_t)kD * 2, (uint64_t)d.n_kv_heads * kD * 2};
  const uint32_t bk[3] = {64, 1, (uint32_t)kKB};
  if (!make_map_3d(&mQ, Q, dq, sq, bq) || !make_map_3d(&mK, Kf, dk, sk, bk) ||
      !make_map_3d(&mV, Vf, dk, sk, bk))
    return cudaErrorInvalidValue;

  AttnArgs a;
  a.tiles = tiles;
  a.n_tiles = n_tiles;
  a.n_units = n_tiles * d.n_kv_heads;
  a.reqs = reqs.d_req;
  a.rows = rows;
  a.O = reinterpret_cast<__nv_bfloat16*>(O);
  a.Hq = d.n_q_heads;
  a.Hkv = d.n_kv_heads;
  a.g = g;
  a.rtile = rtile;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)kD);
  a.err = err;
  e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = a.n_units < sm_count() ? a.n_units : sm_count();
  attn_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(mQ, mK, mV, a);
  return cudaGetLastError();
}

}  // namespace fusekv
