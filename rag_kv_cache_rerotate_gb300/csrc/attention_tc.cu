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
// blocks of 128 up to the tile's last position:
//   S_b = Q K_b^T            tcgen05.mma into one of two TMEM S buffers
//   P_b = exp2(S_b - m)      four softmax warpgroups, each thread one M row and
//                            one 32-key quarter of the block (the quarters of
//                            a row exchange their maxima and sums through
//                            shared memory); causal mask by position on the
//                            blocks that need it; P (bf16) stored to one of
//                            two TMEM P buffers
//   O  += P_b V_b            tcgen05.mma with A = P in TMEM, V read from
//                            shared memory as an MN-major operand
// The running maximum m is raised only when a block exceeds it by more than
// 2^8 (then O in TMEM and the running sum are rescaled), so most blocks skip
// the rescale.  Six roles run decoupled, each behind its own mbarriers:
// warp 0 loads Q and K blocks (3-stage ring), warp 18 loads V blocks (2-stage
// ring), warp 1 issues the S MMAs, warp 19 the P.V MMAs, warps 2-17 run the
// softmax and the epilogue.  A K stage is released as soon as its S MMA has
// completed and an S buffer as soon as the softmax has read it, so loads and
// S MMAs run ahead of the softmax.  The kernel is persistent; units are taken
// heaviest first.
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
constexpr int kWG = 4;                        // softmax warpgroups
constexpr int kCols = kKB / kWG;              // keys of a block per softmax thread
constexpr int kSoftThreads = 128 * kWG;
constexpr int kThreads = 128 + kSoftThreads;  // K/Q loads, S MMAs, softmax, V loads, P.V MMAs
constexpr int kWarpVLoad = 2 + kSoftThreads / 32;
constexpr int kWarpPV = kWarpVLoad + 1;
constexpr int kTmemCols = 512;                // S0 | S1 | O | P0 | P1
constexpr int kColS = 0;                      // + 128 * (b & 1)
constexpr int kColO = 256;
constexpr int kColP = 384;                    // + 64 * (b & 1); bf16 pairs
constexpr int kSmemBytes = (1 + kKStages + kVStages) * kTile + 1024 + 12288;
constexpr float kRescaleThreshold = 8.0f;     // log2 units

struct AttnTile {
  int32_t req;
  int32_t r0;     // first row of the tile within the request's recomputed rows
  int32_t n;      // rows in the tile
  int32_t pad;
};

struct AttnArgs {
  const AttnTile* tiles;
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
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], pv_done[2], o_empty;   // [block parity]
  uint32_t tmem_base;
  volatile int abort_flag;
  uint64_t xmax_bar[2][4];  // [block parity][lane quarter]: all partial row maxima written
  uint64_t xsum_bar[2][4];  // [unit parity][lane quarter]: all partial row sums written
  float xmax[2][kWG][128];   // [block parity][warpgroup][row]: partial row maxima
  float xsum[2][kWG][128];   // [unit parity][warpgroup][row]: partial row sums
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Ctl* ctl) {
  return tc::mbar_wait(bar, parity, &ctl->abort_flag);
}

// The softmax warps issue warp-collective TMEM loads after their waits.
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t* bar, uint32_t parity, Ctl* ctl) {
  return tc::mbar_wait_warp(bar, parity, &ctl->abort_flag);
}

// Which wait gave up: info = wait id (4 bits) << 20 | CTA (8 bits) << 12 | key block (12 bits).
enum AttnWait : uint32_t {
  W_Q_EMPTY = 1, W_K_EMPTY, W_V_EMPTY, W_Q_FULL, W_K_FULL, W_S_EMPTY, W_P_FULL, W_O_EMPTY,
  W_V_FULL, W_S_FULL, W_PV_DONE, W_PV_LAST, W_XCHG
};

__device__ __forceinline__ void abort_kernel(Ctl* ctl, uint32_t* err, uint32_t which = 0,
                                             int j = 0) {
  const bool first = ctl->abort_flag == 0;
  ctl->abort_flag = 1;
  if (first)
    report_error(err, FUSE_ERR_TIMEOUT, SITE_ATTN_TIMEOUT,
                 (which << 20) | ((blockIdx.x & 0xFFu) << 12) | ((uint32_t)j & 0xFFFu));
}

struct Unit {
  int kvh, out0, row0, r0, n, pmax, nkb;
};

__device__ __forceinline__ Unit unit_of(const AttnArgs& a, int u) {
  Unit x;
  const AttnTile t = a.tiles[a.n_tiles - 1 - u / a.Hkv];   // heaviest tiles first
  x.kvh = u % a.Hkv;
  const fuse_request_t& R = a.reqs[t.req];
  x.out0 = (int)R.out0;
  x.row0 = (int)R.row0;
  x.r0 = t.r0;
  x.n = t.n;
  x.pmax = a.rows[R.out0 + t.r0 + t.n - 1].pos;
  x.nkb = x.pmax / kKB + 1;
  return x;
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
    for (int par = 0; par < 2; ++par) {
      tc::mbar_init(&ctl->s_full[par], 1);
      tc::mbar_init(&ctl->s_empty[par], kSoftThreads);
    }
    for (int par = 0; par < 2; ++par) {
      tc::mbar_init(&ctl->p_full[par], kSoftThreads);
      tc::mbar_init(&ctl->pv_done[par], 1);
    }
    tc::mbar_init(&ctl->o_empty, kSoftThreads);
    // the warps (one per softmax warpgroup) owning a TMEM lane quarter
    // exchange partial row values through these
    for (int par = 0; par < 2; ++par)
      for (int q = 0; q < 4; ++q) {
        tc::mbar_init(&ctl->xmax_bar[par][q], 32 * kWG);
        tc::mbar_init(&ctl->xsum_bar[par][q], 32 * kWG);
      }
    ctl->abort_flag = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&mapQ);
    tc::tma_prefetch_desc(&mapK);
    tc::tma_prefetch_desc(&mapV);
  }
  if (warp == 1) tc::tmem_alloc(&ctl->tmem_base, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // --------------------------- Q and K loads ---------------------------
    if (lane == 0) {
      uint32_t uc = 0, kc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x, ++uc) {
        const Unit x = unit_of(a, u);
        if (!wait_or_abort(&ctl->q_empty, (uc & 1) ^ 1, ctl)) {
          abort_kernel(ctl, a.err, W_Q_EMPTY, 0);
          break;
        }
        tc::mbar_arrive_expect_tx(&ctl->q_full, kTile);
        tc::tma_load_3d(sQ, &mapQ, &ctl->q_full, 0, x.kvh * a.g, x.out0 + x.r0);
        tc::tma_load_3d(sQ + kHalf, &mapQ, &ctl->q_full, 64, x.kvh * a.g, x.out0 + x.r0);
        for (int j = 0; j < x.nkb; ++j, ++kc) {
          const int st = kc % kKStages;
          if (!wait_or_abort(&ctl->k_empty[st], ((kc / kKStages) & 1) ^ 1, ctl)) {
            abort_kernel(ctl, a.err, W_K_EMPTY, j);
            ok = false;
            break;
          }
          uint8_t* k = sK + st * kTile;
          const int z = x.row0 + j * kKB;
          tc::mbar_arrive_expect_tx(&ctl->k_full[st], kTile);
          tc::tma_load_3d(k, &mapK, &ctl->k_full[st], 0, x.kvh, z);
          tc::tma_load_3d(k + kHalf, &mapK, &ctl->k_full[st], 64, x.kvh, z);
        }
      }
      // let copies in flight land before the CTA may exit
      tc::mbar_wait(&ctl->q_full, (uc & 1) ^ 1);
      for (uint32_t i = (kc > (uint32_t)kKStages ? kc - kKStages : 0); i < kc; ++i)
        tc::mbar_wait(&ctl->k_full[i % kKStages], (i / kKStages) & 1);
    }
  } else if (warp == kWarpVLoad) {
    // ------------------------------ V loads ------------------------------
    if (lane == 0) {
      uint32_t vc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
        const Unit x = unit_of(a, u);
        for (int j = 0; j < x.nkb; ++j, ++vc) {
          const int st = vc % kVStages;
          if (!wait_or_abort(&ctl->v_empty[st], ((vc / kVStages) & 1) ^ 1, ctl)) {
            abort_kernel(ctl, a.err, W_V_EMPTY, j);
            ok = false;
            break;
          }
          uint8_t* v = sV + st * kTile;
          const int z = x.row0 + j * kKB;
          tc::mbar_arrive_expect_tx(&ctl->v_full[st], kTile);
          tc::tma_load_3d(v, &mapV, &ctl->v_full[st], 0, x.kvh, z);
          tc::tma_load_3d(v + kHalf, &mapV, &ctl->v_full[st], 64, x.kvh, z);
        }
      }
      for (uint32_t i = (vc > (uint32_t)kVStages ? vc - kVStages : 0); i < vc; ++i)
        tc::mbar_wait(&ctl->v_full[i % kVStages], (i / kVStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------ S = Q K^T ------------------------------
    if (lane == 0) {
      const uint32_t idesc_s = tc::idesc_bf16_f32(128, kKB);
      const uint32_t q_addr = tc::smem_u32(sQ);
      uint32_t uc = 0, kc = 0, bc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x, ++uc) {
        const Unit x = unit_of(a, u);
        if (!wait_or_abort(&ctl->q_full, uc & 1, ctl)) {
          abort_kernel(ctl, a.err, W_Q_FULL, 0);
          break;
        }
        for (int j = 0; j < x.nkb; ++j, ++kc) {
          const uint32_t b = bc + j;
          const int st = kc % kKStages;
          if (!wait_or_abort(&ctl->k_full[st], (kc / kKStages) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_K_FULL, j);
            ok = false;
            break;
          }
          // S buffer b & 1 is free once the softmax has read S of block b - 2
          if (b >= 2 && !wait_or_abort(&ctl->s_empty[b & 1], ((b - 2) >> 1) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_S_EMPTY, j);
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t kaddr = tc::smem_u32(sK + st * kTile);
          const uint32_t d = tmem + kColS + (b & 1) * kKB;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            tc::mma_bf16(d, kmajor_step(q_addr, kk), kmajor_step(kaddr, kk), idesc_s, kk != 0);
          tc::mma_commit(&ctl->s_full[b & 1]);
          tc::mma_commit(&ctl->k_empty[st]);
        }
        if (!ok) break;
        tc::mma_commit(&ctl->q_empty);
        bc += x.nkb;
      }
    }
  } else if (warp == kWarpPV) {
    // ------------------------------ O += P V ------------------------------
    if (lane == 0) {
      const uint32_t idesc_o = tc::idesc_bf16_f32(128, kD, /*b_mn_major=*/true);
      uint32_t uc = 0, vc = 0, bc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x, ++uc) {
        const Unit x = unit_of(a, u);
        for (int j = 0; j < x.nkb; ++j, ++vc) {
          const uint32_t b = bc + j;
          if (!wait_or_abort(&ctl->p_full[b & 1], (b >> 1) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_P_FULL, j);
            ok = false;
            break;
          }
          if (j == 0 && !wait_or_abort(&ctl->o_empty, (uc & 1) ^ 1, ctl)) {
            abort_kernel(ctl, a.err, W_O_EMPTY, j);
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
          const uint32_t o = tmem + kColO;
          const uint32_t pa = tmem + kColP + (b & 1) * (kKB / 2);
#pragma unroll
          for (int kk = 0; kk < kKB / 16; ++kk)
            tc::mma_bf16_ts(o, pa + kk * 8, tc::smem_desc_mn128(vaddr + kk * 16 * 128, kHalf),
                            idesc_o, (j | kk) != 0);
          tc::mma_commit(&ctl->pv_done[b & 1]);
          tc::mma_commit(&ctl->v_empty[st]);
        }
        bc += x.nkb;
      }
    }
  } else {
    // --------------------------- softmax + epilogue ---------------------------
    const int wg = (warp - 2) >> 2;                    // key quarter of this warpgroup
    const int quarter = warp % 4;                      // TMEM lane quarter
    const int m = quarter * 32 + lane;                 // M row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int c_off = wg * kCols;                      // first S / O column of this thread
    uint32_t uc = 0, bc = 0;
    for (int u = blockIdx.x; u < a.n_units; u += gridDim.x, ++uc) {
      const Unit x = unit_of(a, u);
      const int rl = m / a.g;
      const int hh = m % a.g;
      const bool valid = rl < x.n;
      const int p = a.rows[x.out0 + x.r0 + (valid ? rl : x.n - 1)].pos;
      const int p_first = a.rows[x.out0 + x.r0].pos;   // rows ascend: the tile's smallest
      float mu = -1e30f, l = 0.f;                      // running max (log2 units), partial sum
      bool ok = true;
      for (int j = 0; j < x.nkb; ++j) {
        const uint32_t b = bc + j;
        if (!warp_wait_or_abort(&ctl->s_full[b & 1], (b >> 1) & 1, ctl)) {
          abort_kernel(ctl, a.err, W_S_FULL, j);
          ok = false;
          break;
        }
        tc::tc_fence_after();
        float s[kCols];
        {
          uint32_t r[32];
          tc::tmem_ld_32x32b_x32(tmem + lane_off + kColS + (b & 1) * kKB + c_off, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < kCols; ++i) s[i] = __uint_as_float(r[i]);
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&ctl->s_empty[b & 1]);
        const int key0 = j * kKB + c_off;
        if (key0 + kCols - 1 > p_first) {              // warp-uniform: some key may be masked
#pragma unroll
          for (int c = 0; c < kCols; ++c) s[c] = (key0 + c <= p) ? s[c] : -1e30f;
        }
        float mx;
        {                                              // tree maximum of the 32 scores
          float t[11];
#pragma unroll
          for (int i = 0; i < 10; ++i) t[i] = max3(s[3 * i], s[3 * i + 1], s[3 * i + 2]);
          t[10] = fmaxf(s[30], s[31]);
          const float u0 = max3(t[0], t[1], t[2]), u1 = max3(t[3], t[4], t[5]);
          const float u2 = max3(t[6], t[7], t[8]), u3 = fmaxf(t[9], t[10]);
          mx = fmaxf(max3(u0, u1, u2), u3);
        }
        ctl->xmax[b & 1][wg][m] = mx;
        tc::mbar_arrive(&ctl->xmax_bar[b & 1][quarter]);
        if (!warp_wait_or_abort(&ctl->xmax_bar[b & 1][quarter], (b >> 1) & 1, ctl)) {
          abort_kernel(ctl, a.err, W_XCHG, j);
          ok = false;
          break;
        }
        {
          const float* xm = &ctl->xmax[b & 1][0][m];
          mx = fmaxf(max3(xm[0], xm[128], xm[256]), xm[384]) * a.scale_log2;
        }
        float mnew = mu;
        bool rescale = false;
        if (j == 0) {
          mnew = mx;
        } else if (mx > mu + kRescaleThreshold) {
          mnew = mx;
          rescale = true;
        }
        const float neg = -mnew;
        float e[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c) e[c] = ex2(fmaf(s[c], a.scale_log2, neg));
        uint32_t pk[kCols / 2];
#pragma unroll
        for (int c = 0; c < kCols; c += 2) pk[c / 2] = pack_bf16x2(e[c], e[c + 1]);
        float sum;
        {                                              // tree sum of the 32 probabilities
#pragma unroll
          for (int w = kCols / 2; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) e[i] += e[i + w];
          sum = e[0];
        }
        const float alpha = rescale ? ex2(mu - mnew) : 1.f;
        l = l * alpha + sum;
        // P buffer b & 1 was last read by the P.V of block b - 2; a rescale of
        // O also needs the P.V of block b - 1 done (commits complete in order)
        const bool any_rescale = __any_sync(0xffffffffu, rescale);
        if (j >= 1 && (any_rescale || j >= 2)) {
          const uint32_t wb = any_rescale ? b - 1 : b - 2;
          if (!warp_wait_or_abort(&ctl->pv_done[wb & 1], (wb >> 1) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_PV_DONE, j);
            ok = false;
            break;
          }
          tc::tc_fence_after();
        }
        // tcgen05.ld/st are warp-collective (.sync.aligned): the whole warp
        // rescales its columns of O when any of its rows needs it (alpha is 1
        // for the others); all warps of a lane quarter decide alike
        if (any_rescale) {
          uint32_t r[32];
          const uint32_t to = tmem + lane_off + kColO + c_off;
          tc::tmem_ld_32x32b_x32(to, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tc::tmem_st_32x32b_x32(to, r);
        }
        // this thread's 32 keys of P row m: 32 bf16 in 16 TMEM columns
        tc::tmem_st_32x32b_x16(tmem + lane_off + kColP + (b & 1) * (kKB / 2) + wg * (kCols / 2), pk);
        tc::tmem_st_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(&ctl->p_full[b & 1]);
        mu = mnew;
      }
      if (!ok) break;
      ctl->xsum[uc & 1][wg][m] = l;
      const uint32_t last = bc + x.nkb - 1;
      if (!warp_wait_or_abort(&ctl->pv_done[last & 1], (last >> 1) & 1, ctl)) {
        abort_kernel(ctl, a.err, W_PV_LAST, x.nkb);
        break;
      }
      tc::tc_fence_after();
      tc::mbar_arrive(&ctl->xsum_bar[uc & 1][quarter]);
      if (!warp_wait_or_abort(&ctl->xsum_bar[uc & 1][quarter], (uc >> 1) & 1, ctl)) {
        abort_kernel(ctl, a.err, W_XCHG, x.nkb);
        break;
      }
      {
        const float* xs = &ctl->xsum[uc & 1][0][m];
        const float inv = 1.f / ((xs[0] + xs[128]) + (xs[256] + xs[384]));
        __nv_bfloat16* dst =
            a.O + ((int64_t)(x.out0 + x.r0 + rl) * a.Hq + x.kvh * a.g + hh) * kD + c_off;
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tmem + lane_off + kColO + c_off, r);
        tc::tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * inv, __uint_as_float(r[8 * q + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv, __uint_as_float(r[8 * q + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv, __uint_as_float(r[8 * q + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv, __uint_as_float(r[8 * q + 7]) * inv);
            reinterpret_cast<uint4*>(dst)[q] = w;
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&ctl->o_empty);
      bc += x.nkb;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// One block: the tiles of every request, in request order.
__global__ void attn_tiles_kernel(const fuse_request_t* reqs, int n_req, int rtile, AttnTile* tiles) {
  if (threadIdx.x != 0) return;
  int t = 0;
  for (int r = 0; r < n_req; ++r) {
    const int R = reqs[r].k + reqs[r].n_query;
    for (int r0 = 0; r0 < R; r0 += rtile) {
      AttnTile x;
      x.req = r;
      x.r0 = r0;
      x.n = min(rtile, R - r0);
      x.pad = 0;
      tiles[t++] = x;
    }
  }
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
  return (size_t)(n_out / 16 + n_req + 1) * sizeof(AttnTile);
}

bool tc_attention_supported(const fuse_layer_desc_t& d) {
  const int g = d.n_q_heads / d.n_kv_heads;
  return d.dtype == FUSE_BF16 && d.head_dim == kD && (g == 1 || g == 2 || g == 4 || g == 8) &&
         tma_encode_available();
}

cudaError_t launch_attention_tc(const fuse_layer_desc_t& d, const fuse_requests_t& reqs,
                                int64_t n_out, int64_t n_tok, const WorkRow* rows, const void* Q,
                                const void* Kf, const void* Vf, void* O, void* tiles_ws,
                                bool tiles_ready, uint32_t* err, cudaStream_t s) {
  const int g = d.n_q_heads / d.n_kv_heads;
  const int rtile = 128 / g;
  int n_tiles = 0;
  for (int r = 0; r < reqs.n_req; ++r) {
    const int R = reqs.h_req[r].k + reqs.h_req[r].n_query;
    n_tiles += (R + rtile - 1) / rtile;
  }
  if (n_tiles == 0) return cudaSuccess;
  AttnTile* tiles = reinterpret_cast<AttnTile*>(tiles_ws);
  cudaError_t e = cudaSuccess;
  if (!tiles_ready) {
    attn_tiles_kernel<<<1, 32, 0, s>>>(reqs.d_req, reqs.n_req, rtile, tiles);
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
