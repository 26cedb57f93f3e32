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
//   S = Q K_b^T          tcgen05.mma into TMEM buffer b % 3 (columns
//                        [128 (b % 3), 128 (b % 3) + 128)), so the scores of
//                        the next blocks are formed during this block's
//                        softmax
//   P = 2^(S - m)        eight warps; each thread holds two M rows x 32 keys
//                        of the block in registers (TMEM shape 16x256b: rows
//                        t/4 and t/4 + 8 of the warp's 16 lanes, key pairs
//                        8q + 2(t%4) + {0, 1}), the four threads of a row
//                        exchange maxima by shuffles, and each key pair is
//                        one bf16x2 column of P (shape 16x128b: column
//                        4q + t%4), written back over S
//   O += P V_b           tcgen05.mma with A = P in TMEM, V read from shared
//                        memory as an MN-major operand, O in TMEM columns
//                        [384, 512)
// The running maximum m is raised only when a block exceeds it by more than
// 2^16 (then O and the running sum l are rescaled).  A separate warpgroup
// writes O / l of a unit while the softmax starts on the next one (whose
// first P.V waits until O has been read).
// Roles, each behind its own mbarriers: warp 0 loads Q (two buffers in the
// single-CTA form, so that the next unit's Q lands while this one's scores
// are formed; one in the paired form) and K blocks (a 3-stage ring; 4 in the
// paired form), warp 2 V blocks (2-stage ring), warp 1 issues the S MMAs, warp 3 the
// P.V MMAs, warps 4-11 the softmax, warps 12-15 the output.  Every role reads
// the unit's tile record (first output row, first fused row, rows, key
// blocks) one unit ahead.  The kernel is persistent; units are taken heaviest
// first, snake-ordered over the CTAs (round r visits the CTAs upwards when r
// is even and downwards when r is odd).
// For requests of 16 384 tokens and more, tiles go in pairs: a cluster of
// two CTAs takes two neighbouring tiles (by key-block count) of one KV head
// (units are then pairs of tiles), and when both belong to one request every
// K and V block is fetched from L2 once for both: each CTA loads one
// 64-column half with TMA multicast into both CTAs' rings, and a stage is
// refilled once both CTAs' MMAs have released it (their commits arrive on
// both CTAs' barriers).  On long contexts this halves the ~16 GB of K and V
// a layer-step moves from L2 to the SMs; the time at a fixed clock is the
// same, but the energy saved lets the SMs hold a higher clock under the
// board's power cap, where long steps run.
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <mutex>

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
// Ring depths: the single-CTA form double-buffers Q (its units can be short,
// and the next unit's Q then lands while this one runs); the paired form, for
// long requests whose units run over a hundred key blocks, trades the second
// Q buffer for a fourth K stage (the same shared memory), which keeps the two
// CTAs' shared rings fed (+0.5 % on the long-context step)
constexpr int kQBufs = 2;                     // Q tiles in flight, at most
constexpr int64_t kPairMinTokens = 16384;     // longest request from which tiles go in pairs
constexpr int kKStages = 4;                   // K stages, at most
template <bool PAIR> struct Ring {
  static constexpr int QB = PAIR ? 1 : 2;     // Q buffers
  static constexpr int KS = PAIR ? 4 : 3;     // K stages
};
static_assert(Ring<true>::QB + Ring<true>::KS == Ring<false>::QB + Ring<false>::KS,
              "both forms lay out the same shared memory");
constexpr int kVStages = 2;
constexpr int kWarpQK = 0, kWarpS = 1, kWarpV = 2, kWarpPV = 3, kWarpSoft = 4, kWarpOut = 12;
constexpr int kSoftThreads = 256;
constexpr int kThreads = 16 * 32;
constexpr int kTmemCols = 512;                // S0 | S1 | S2 | O
constexpr int kSBufs = 3;
constexpr int kColO = 384;
// log2 units.  P is rounded to bf16 and summed in fp32 at the same relative
// precision whatever its size, so a reference up to 2^16 below the true
// maximum costs no accuracy (P, l and O stay far from overflow: at most
// 2^16 x keys x |V|); a larger threshold means fewer O rescales.
constexpr float kRescaleThreshold = 16.0f;
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
  int st32;               // O 32-byte aligned: 256-bit stores
  int records_ready;      // tiles and rows complete before the previous kernel's release
};

struct Ctl {
  uint64_t q_full[kQBufs], q_empty[kQBufs];
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[kSBufs], p_full[kSBufs], pv_done[kSBufs];   // [block % 3]
  uint64_t o_full, o_empty, l_full;                            // once per unit
  uint32_t tmem_base;
  volatile int abort_flag;
  float xl[128];          // [row] softmax row sum of the unit being written
};
constexpr int kSmemBytes =
    (Ring<false>::QB + Ring<false>::KS + kVStages) * kTile + 1024 + (int)sizeof(Ctl);
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

// The unit that a CTA (a cluster of two CTAs when PAIR) takes in its i-th
// round: round i visits them upwards when i is even and downwards when i is
// odd.  Units past the end stay past it in later rounds.
template <bool PAIR>
__device__ __forceinline__ int unit_at(int i) {
  const int G = PAIR ? (int)gridDim.x / 2 : (int)gridDim.x;
  const int c = PAIR ? (int)blockIdx.x / 2 : (int)blockIdx.x;
  return i * G + ((i & 1) ? G - 1 - c : c);
}

// What one CTA does for a unit.
struct Unit {
  int4 t;       // its tile record; rows 0 and key blocks 0 when it has no tile
  int kvh;
  int nkb;      // key blocks its K and V rings step through
  int shared;   // PAIR: both tiles start at the same fused row, and each CTA
                // loads one 64-column half of every K and V block for both
};

// Unit u.  Single CTAs: the tile u / Hkv places from the heaviest end of the
// list.  Pairs: the tiles 2p and 2p + 1 places from the heaviest end
// (p = u / Hkv), the first for cluster rank 0 and the second for rank 1;
// both CTAs' rings step through the larger key-block count of the two, so
// that they stay in step (a CTA past its own blocks only passes stages on).
template <bool PAIR>
__device__ __forceinline__ Unit unit_rec(const AttnArgs& a, int u, uint32_t rank) {
  Unit r;
  r.kvh = u % a.Hkv;
  if (!PAIR) {
    r.t = a.tiles[a.n_tiles - 1 - u / a.Hkv];
    r.nkb = r.t.w;
    r.shared = 0;
    return r;
  }
  const int i0 = a.n_tiles - 1 - 2 * (u / a.Hkv);
  const int4 t0 = a.tiles[i0];
  const int4 t1 = i0 > 0 ? a.tiles[i0 - 1] : make_int4(t0.x, t0.y, 0, 0);
  r.t = rank ? t1 : t0;
  r.nkb = max(t0.w, t1.w);
  r.shared = t0.y == t1.y;
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of floats for the f32x2 arithmetic of sm_100 and later: one
// instruction does the operation on both halves.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 3-D tiled load delivered to the same shared-memory offset in every CTA of
// `mask` (bit r: cluster rank r); each destination CTA counts the bytes on the
// mbarrier at `bar`'s offset in its own shared memory.
__device__ __forceinline__ void tma_load_3d_multicast(void* dst, const CUtensorMap* map,
                                                      uint64_t* bar, int x, int y, int z,
                                                      uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(tc::smem_u32(bar)), "h"(mask)
      : "memory");
}

// Arrive on the mbarrier at this offset in every CTA of `mask` once every
// tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(tc::smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// descriptor of K-step kk (16 columns) of a 128-row K-major tile stored as two
// 64-column halves
__device__ __forceinline__ uint64_t kmajor_step(uint32_t tile, int kk) {
  return tc::smem_desc_k128(tile + (kk >> 2) * kHalf + (kk & 3) * 32);
}

// PAIR: clusters of two CTAs, each on its own tile of one KV head; when both
// tiles read the same fused rows, every K and V block is read from L2 once
// for the pair (each CTA loads one half with TMA multicast into both), and a
// ring stage is refilled once both CTAs' MMAs are done with it.
template <bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                   const __grid_constant__ CUtensorMap mapV, const AttnArgs a) {
  constexpr int kQB = Ring<PAIR>::QB, kKS = Ring<PAIR>::KS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                               // Q buffer q at sQ + q * kTile
  uint8_t* sK = smem + kQB * kTile;              // K stage s at sK + s * kTile
  uint8_t* sV = sK + kKS * kTile;              // V stage s at sV + s * kTile
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (kQB + kKS + kVStages) * kTile);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = PAIR ? tc::cluster_rank() : 0u;
  constexpr uint16_t kBoth = 0x3;                   // both CTAs of the cluster
  constexpr uint32_t kUsers = PAIR ? 2 : 1;         // MMA warps that release a K / V stage
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int q = 0; q < kQB; ++q) {
      tc::mbar_init(&ctl->q_full[q], 1);
      tc::mbar_init(&ctl->q_empty[q], 1);
    }
    for (int s = 0; s < kKS; ++s) {
      tc::mbar_init(&ctl->k_full[s], 1);
      tc::mbar_init(&ctl->k_empty[s], kUsers);
    }
    for (int s = 0; s < kVStages; ++s) {
      tc::mbar_init(&ctl->v_full[s], 1);
      tc::mbar_init(&ctl->v_empty[s], kUsers);
    }
    for (int s = 0; s < kSBufs; ++s) {
      tc::mbar_init(&ctl->s_full[s], 1);
      tc::mbar_init(&ctl->p_full[s], kSoftThreads);
      tc::mbar_init(&ctl->pv_done[s], 1);
    }
    tc::mbar_init(&ctl->o_full, 1);
    tc::mbar_init(&ctl->o_empty, 128);
    tc::mbar_init(&ctl->l_full, kSoftThreads);
    ctl->abort_flag = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&mapQ);
    tc::tma_prefetch_desc(&mapK);
    tc::tma_prefetch_desc(&mapV);
  }
  if (warp == kWarpS) tc::tmem_alloc(&ctl->tmem_base, kTmemCols);
  tc::tc_fence_before();
  if (PAIR) {
    __syncwarp();
    tc::cluster_sync_all();   // both CTAs' barriers exist before any copy or arrival crosses
  } else {
    __syncthreads();
  }
  tc::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int n_units = a.n_units;
  // The first unit's records, and for the softmax threads the positions of
  // their rows.  When the records come from a kernel that finished before the
  // previous one could release its dependents, they are read before waiting.
  const bool have0 = unit_at<PAIR>(0) < n_units;
  Unit U0;
  U0.t = make_int4(0, 0, 0, 0);
  U0.kvh = U0.nkb = U0.shared = 0;
  int pos0[3] = {0, 0, 0};                          // softmax: rows R0, R1, the tile's first
  auto first_records = [&]() {
    if (!have0) return;
    U0 = unit_rec<PAIR>(a, unit_at<PAIR>(0), rank);
    if (warp >= kWarpSoft && warp < kWarpOut && U0.t.z > 0) {
      const int R0 = (warp & 3) * 32 + ((warp - kWarpSoft) >> 2) * 16 + (lane >> 2);
      pos0[0] = a.rows[U0.t.x + min(R0 / a.g, U0.t.z - 1)].pos;
      pos0[1] = a.rows[U0.t.x + min((R0 + 8) / a.g, U0.t.z - 1)].pos;
      pos0[2] = a.rows[U0.t.x].pos;
    }
  };
  if (a.records_ready) first_records();
  pdl_wait();                 // inputs of the previous kernel complete and visible
  if (!a.records_ready) first_records();

  if (warp == kWarpQK) {
    // --------------------------- Q and K loads ---------------------------
    if (lane == 0) {
      uint32_t kc = 0;
      int i = 0;
      bool ok = true;
      Unit U = U0;
      for (; unit_at<PAIR>(i) < n_units && ok; ++i) {
        const Unit cur = U;
        if (unit_at<PAIR>(i + 1) < n_units) U = unit_rec<PAIR>(a, unit_at<PAIR>(i + 1), rank);
        const int qb = i % kQB;
        if (!wait_or_abort(&ctl->q_empty[qb], ((i / kQB) & 1) ^ 1, ctl)) {
          abort_kernel(ctl, a.err, W_Q_EMPTY, 0);
          break;
        }
        uint8_t* q = sQ + qb * kTile;
        if (cur.t.z > 0) {
          tc::mbar_arrive_expect_tx(&ctl->q_full[qb], kTile);
          tc::tma_load_3d(q, &mapQ, &ctl->q_full[qb], 0, cur.kvh * a.g, cur.t.x);
          tc::tma_load_3d(q + kHalf, &mapQ, &ctl->q_full[qb], 64, cur.kvh * a.g, cur.t.x);
        } else {
          tc::mbar_arrive(&ctl->q_full[qb]);
        }
        for (int j = 0; j < cur.nkb; ++j, ++kc) {
          const int st = kc % kKS;
          if (!wait_or_abort(&ctl->k_empty[st], ((kc / kKS) & 1) ^ 1, ctl)) {
            abort_kernel(ctl, a.err, W_K_EMPTY, j);
            ok = false;
            break;
          }
          uint8_t* k = sK + st * kTile;
          const int z = cur.t.y + j * kKB;
          // the stage counts kTile bytes: both halves from this CTA, or one
          // from each CTA of the pair (the other's may land first)
          if (PAIR && cur.shared) {
            tc::mbar_arrive_expect_tx(&ctl->k_full[st], kTile);
            tma_load_3d_multicast(k + rank * kHalf, &mapK, &ctl->k_full[st], 64 * (int)rank,
                                      cur.kvh, z, kBoth);
          } else if (j < cur.t.w) {
            tc::mbar_arrive_expect_tx(&ctl->k_full[st], kTile);
            tc::tma_load_3d(k, &mapK, &ctl->k_full[st], 0, cur.kvh, z);
            tc::tma_load_3d(k + kHalf, &mapK, &ctl->k_full[st], 64, cur.kvh, z);
          } else {
            tc::mbar_arrive(&ctl->k_full[st]);
          }
        }
      }
      // let copies in flight land (and, in a pair, the other CTA's releases
      // of the last stages arrive) before the CTA may exit
      for (int k = (i > kQB ? i - kQB : 0); k < i; ++k)
        tc::mbar_wait(&ctl->q_full[k % kQB], (k / kQB) & 1);
      for (uint32_t c = (kc > (uint32_t)kKS ? kc - kKS : 0); c < kc; ++c) {
        tc::mbar_wait(&ctl->k_full[c % kKS], (c / kKS) & 1);
        if (PAIR) tc::mbar_wait(&ctl->k_empty[c % kKS], (c / kKS) & 1);
      }
    }
  } else if (warp == kWarpV) {
    // ------------------------------ V loads ------------------------------
    if (lane == 0) {
      uint32_t vc = 0;
      bool ok = true;
      Unit U = U0;
      for (int i = 0; unit_at<PAIR>(i) < n_units && ok; ++i) {
        const Unit cur = U;
        if (unit_at<PAIR>(i + 1) < n_units) U = unit_rec<PAIR>(a, unit_at<PAIR>(i + 1), rank);
        for (int j = 0; j < cur.nkb; ++j, ++vc) {
          const int st = vc % kVStages;
          if (!wait_or_abort(&ctl->v_empty[st], ((vc / kVStages) & 1) ^ 1, ctl)) {
            abort_kernel(ctl, a.err, W_V_EMPTY, j);
            ok = false;
            break;
          }
          uint8_t* v = sV + st * kTile;
          const int z = cur.t.y + j * kKB;
          if (PAIR && cur.shared) {
            tc::mbar_arrive_expect_tx(&ctl->v_full[st], kTile);
            tma_load_3d_multicast(v + rank * kHalf, &mapV, &ctl->v_full[st], 64 * (int)rank,
                                      cur.kvh, z, kBoth);
          } else if (j < cur.t.w) {
            tc::mbar_arrive_expect_tx(&ctl->v_full[st], kTile);
            tc::tma_load_3d(v, &mapV, &ctl->v_full[st], 0, cur.kvh, z);
            tc::tma_load_3d(v + kHalf, &mapV, &ctl->v_full[st], 64, cur.kvh, z);
          } else {
            tc::mbar_arrive(&ctl->v_full[st]);
          }
        }
      }
      for (uint32_t c = (vc > (uint32_t)kVStages ? vc - kVStages : 0); c < vc; ++c) {
        tc::mbar_wait(&ctl->v_full[c % kVStages], (c / kVStages) & 1);
        if (PAIR) tc::mbar_wait(&ctl->v_empty[c % kVStages], (c / kVStages) & 1);
      }
    }
  } else if (warp == kWarpS) {
    // ------------------------------ S = Q K^T ------------------------------
    if (lane == 0) {
      const uint32_t idesc_s = tc::idesc_bf16_f32(128, kKB);
      uint32_t kc = 0, b = 0;
      bool ok = true;
      Unit U = U0;
      for (int i = 0; unit_at<PAIR>(i) < n_units && ok; ++i) {
        const Unit cur = U;
        if (unit_at<PAIR>(i + 1) < n_units) U = unit_rec<PAIR>(a, unit_at<PAIR>(i + 1), rank);
        const int qb = i % kQB;
        if (!wait_or_abort(&ctl->q_full[qb], (i / kQB) & 1, ctl)) {
          abort_kernel(ctl, a.err, W_Q_FULL, 0);
          break;
        }
        const uint32_t q_addr = tc::smem_u32(sQ + qb * kTile);
        for (int j = 0; j < cur.nkb; ++j, ++kc) {
          const int st = kc % kKS;
          // a stage is released only after its copies have landed, also when
          // this CTA does not use it (the next copies into it count on the
          // next phase)
          if (!wait_or_abort(&ctl->k_full[st], (kc / kKS) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_K_FULL, j);
            ok = false;
            break;
          }
          if (j < cur.t.w) {
            // buffer b % 3 holds P of block b - 3 until that block's P.V is done
            const uint32_t sb = b % kSBufs;
            if (!wait_or_abort(&ctl->pv_done[sb], ((b / kSBufs) & 1) ^ 1, ctl)) {
              abort_kernel(ctl, a.err, W_S_FREE, j);
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const uint32_t kaddr = tc::smem_u32(sK + st * kTile);
            const uint32_t d = tmem + sb * kKB;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              tc::mma_bf16(d, kmajor_step(q_addr, kk), kmajor_step(kaddr, kk), idesc_s, kk != 0);
            tc::mma_commit(&ctl->s_full[sb]);
            ++b;
          }
          if (PAIR)
            mma_commit_multicast(&ctl->k_empty[st], kBoth);
          else
            tc::mma_commit(&ctl->k_empty[st]);
        }
        if (!ok) break;
        tc::mma_commit(&ctl->q_empty[qb]);
      }
    }
  } else if (warp == kWarpPV) {
    // ------------------------------ O_i += P V ------------------------------
    if (lane == 0) {
      const uint32_t idesc_o = tc::idesc_bf16_f32(128, kD, /*b_mn_major=*/true);
      uint32_t vc = 0, b = 0;
      bool ok = true;
      Unit U = U0;
      for (int i = 0; unit_at<PAIR>(i) < n_units && ok; ++i) {
        const Unit cur = U;
        if (unit_at<PAIR>(i + 1) < n_units) U = unit_rec<PAIR>(a, unit_at<PAIR>(i + 1), rank);
        const uint32_t o = tmem + kColO;
        // O was last read by the output warps for unit i - 1
        if (!wait_or_abort(&ctl->o_empty, (i & 1) ^ 1, ctl)) {
          abort_kernel(ctl, a.err, W_O_EMPTY, 0);
          break;
        }
        for (int j = 0; j < cur.nkb; ++j, ++vc) {
          const int st = vc % kVStages;
          const bool use = j < cur.t.w;
          const uint32_t sb = b % kSBufs;
          if (use && !wait_or_abort(&ctl->p_full[sb], (b / kSBufs) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_P_FULL, j);
            ok = false;
            break;
          }
          if (!wait_or_abort(&ctl->v_full[st], (vc / kVStages) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_V_FULL, j);
            ok = false;
            break;
          }
          if (use) {
            tc::tc_fence_after();
            const uint32_t vaddr = tc::smem_u32(sV + st * kTile);
            const uint32_t pa = tmem + sb * kKB;
#pragma unroll
            for (int kk = 0; kk < kKB / 16; ++kk)
              tc::mma_bf16_ts(o, pa + kk * 8, tc::smem_desc_mn128(vaddr + kk * 16 * 128, kHalf),
                              idesc_o, (j | kk) != 0 ? 1u : 0u);
            tc::mma_commit(&ctl->pv_done[sb]);
            ++b;
          }
          if (PAIR)
            mma_commit_multicast(&ctl->v_empty[st], kBoth);
          else
            tc::mma_commit(&ctl->v_empty[st]);
        }
        if (!ok) break;
        tc::mma_commit(&ctl->o_full);
      }
    }
  } else if (warp < kWarpOut) {
    // ------------------------------- softmax -------------------------------
    // warp w: TMEM lane quarter w % 4, half (w - 4) / 4 of it: 16 M rows
    const int base = (warp & 3) * 32 + ((warp - kWarpSoft) >> 2) * 16;
    const uint32_t lane_off = (uint32_t)base << 16;
    const int c4 = lane & 3;
    const int R0 = base + (lane >> 2), R1 = R0 + 8;    // this thread's two M rows
    const int rl0 = R0 / a.g, rl1 = R1 / a.g;
    const float scale = a.scale_log2;
    uint32_t b = 0;
    // this unit's record and positions, read one unit ahead
    Unit U = U0;
    int p0n = pos0[0], p1n = pos0[1], pfn = pos0[2];
    for (int i = 0; unit_at<PAIR>(i) < n_units; ++i) {
      const int nkb = U.t.w;
      const int p0 = p0n, p1 = p1n;
      const int p_first = pfn;                         // rows ascend: the tile's smallest
      const bool more = unit_at<PAIR>(i + 1) < n_units;
      if (more) U = unit_rec<PAIR>(a, unit_at<PAIR>(i + 1), rank);
      const uint32_t tO = tmem + lane_off + kColO;
      float mu0 = kFloor, mu1 = kFloor;                // running maxima (log2 units)
      float l0 = 0.f, l1 = 0.f;                        // this thread's part of the row sums
      bool ok = true;
      for (int j = 0; j < nkb; ++j, ++b) {
        const uint32_t sb = b % kSBufs;
        if (!warp_wait_or_abort(&ctl->s_full[sb], (b / kSBufs) & 1, ctl)) {
          abort_kernel(ctl, a.err, W_S_FULL, j);
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t tS = tmem + lane_off + sb * kKB;
        const int key0 = j * kKB;
        uint32_t r[64];
        tc::tmem_ld_16x256b_x8(tS, *reinterpret_cast<uint32_t(*)[32]>(r));
        tc::tmem_ld_16x256b_x8(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tc::tmem_ld_wait();
        if (key0 + kKB - 1 > p_first) {                // warp-uniform: some key may be masked
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int k = key0 + 8 * q + 2 * c4;
            if (k > p0) r[4 * q] = __float_as_uint(-1e30f);
            if (k + 1 > p0) r[4 * q + 1] = __float_as_uint(-1e30f);
            if (k > p1) r[4 * q + 2] = __float_as_uint(-1e30f);
            if (k + 1 > p1) r[4 * q + 3] = __float_as_uint(-1e30f);
          }
        }
        float m0, m1;
        {
          float a0 = __uint_as_float(r[0]), a1 = __uint_as_float(r[1]);
          float b0 = __uint_as_float(r[2]), b1 = __uint_as_float(r[3]);
#pragma unroll
          for (int q = 1; q < 15; q += 2) {                // repeats 1 .. 14 in pairs
            a0 = max3(a0, __uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 4]));
            a1 = max3(a1, __uint_as_float(r[4 * q + 1]), __uint_as_float(r[4 * q + 5]));
            b0 = max3(b0, __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 6]));
            b1 = max3(b1, __uint_as_float(r[4 * q + 3]), __uint_as_float(r[4 * q + 7]));
          }
          m0 = max3(a0, a1, fmaxf(__uint_as_float(r[60]), __uint_as_float(r[61])));   // repeat 15
          m1 = max3(b0, b1, fmaxf(__uint_as_float(r[62]), __uint_as_float(r[63])));
          m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
          m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
          m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
          m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
        }
        const float ms0 = m0 * scale, ms1 = m1 * scale;
        float mn0 = mu0, mn1 = mu1;
        bool rs0 = false, rs1 = false;
        if (j == 0) {
          mn0 = fmaxf(ms0, kFloor);
          mn1 = fmaxf(ms1, kFloor);
        } else {
          if (ms0 > mu0 + kRescaleThreshold) { mn0 = ms0; rs0 = true; }
          if (ms1 > mu1 + kRescaleThreshold) { mn1 = ms1; rs1 = true; }
        }
        const float al0 = rs0 ? ex2(mu0 - mn0) : 1.f, al1 = rs1 ? ex2(mu1 - mn1) : 1.f;
        // probabilities: key pairs packed as bf16x2, in place over the scores;
        // the scaling and the row sums work on key pairs (f32x2)
        const uint64_t sc2 = pack2(scale, scale);
        const uint64_t ng0 = pack2(-mn0, -mn0), ng1 = pack2(-mn1, -mn1);
        uint64_t acc0 = 0, acc1 = 0;                    // (even keys, odd keys) of each row
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float2 x01 = unpack2(fma2(pack2(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1])), sc2, ng0));
          const float2 x23 = unpack2(fma2(pack2(__uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])), sc2, ng1));
          const float e0 = ex2(x01.x), e1 = ex2(x01.y), e2 = ex2(x23.x), e3 = ex2(x23.y);
          acc0 = add2(acc0, pack2(e0, e1));
          acc1 = add2(acc1, pack2(e2, e3));
          r[2 * q] = pack_bf16x2(e0, e1);
          r[2 * q + 1] = pack_bf16x2(e2, e3);
        }
        const float2 a0 = unpack2(acc0), a1 = unpack2(acc1);
        const float s0 = a0.x + a0.y, s1 = a1.x + a1.y;
        tc::tmem_st_16x128b_x16(tS, *reinterpret_cast<uint32_t(*)[32]>(r));
        // tcgen05.ld/st are warp-collective (.sync.aligned): the whole warp
        // rescales its rows of O when any of them needs it (the factor is 1
        // for the others); O must hold the previous block's P.V
        if (__any_sync(0xffffffffu, rs0 || rs1)) {
          if (!warp_wait_or_abort(&ctl->pv_done[(b - 1) % kSBufs], ((b - 1) / kSBufs) & 1, ctl)) {
            abort_kernel(ctl, a.err, W_PV_DONE, j);
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kD; c += 64) {
            uint32_t o[32];
            tc::tmem_ld_16x256b_x8(tO + c, o);
            tc::tmem_ld_wait();
            const uint64_t f0 = pack2(al0, al0), f1 = pack2(al1, al1);
#pragma unroll
            for (int q = 0; q < 32; q += 2) {
              const float2 v = unpack2(mul2(pack2(__uint_as_float(o[q]), __uint_as_float(o[q + 1])), (q & 2) ? f1 : f0));
              o[q] = __float_as_uint(v.x);
              o[q + 1] = __float_as_uint(v.y);
            }
            tc::tmem_st_16x256b_x8(tO + c, o);
          }
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(&ctl->p_full[sb]);
        l0 = l0 * al0 + s0;
        l1 = l1 * al1 + s1;
        mu0 = mn0;
        mu1 = mn1;
      }
      if (!ok) break;
      if (more && U.t.z > 0) {
        p0n = a.rows[U.t.x + min(rl0, U.t.z - 1)].pos;
        p1n = a.rows[U.t.x + min(rl1, U.t.z - 1)].pos;
        pfn = a.rows[U.t.x].pos;
      }
      // row sums: the four threads of a row, in a fixed order
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      // the row sums of unit i, once the output warps are done with unit i - 1
      if (!warp_wait_or_abort(&ctl->o_empty, (i & 1) ^ 1, ctl)) {
        abort_kernel(ctl, a.err, W_L_FREE, nkb);
        break;
      }
      if (c4 == 0) {
        ctl->xl[R0] = l0;
        ctl->xl[R1] = l1;
      }
      tc::mbar_arrive(&ctl->l_full);
    }
  } else {
    // ---------------------------- output O / l ----------------------------
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int rl = m / a.g;
    const int hh = m % a.g;
    Unit U = U0;
    for (int i = 0; unit_at<PAIR>(i) < n_units; ++i) {
      const Unit cu = U;
      const int4 cur = cu.t;
      if (unit_at<PAIR>(i + 1) < n_units) U = unit_rec<PAIR>(a, unit_at<PAIR>(i + 1), rank);
      const int kvh = cu.kvh;
      if (!warp_wait_or_abort(&ctl->o_full, i & 1, ctl)) {
        abort_kernel(ctl, a.err, W_O_FULL, cur.w);
        break;
      }
      if (!warp_wait_or_abort(&ctl->l_full, i & 1, ctl)) {
        abort_kernel(ctl, a.err, W_L_FULL, cur.w);
        break;
      }
      tc::tc_fence_after();
      const float inv = 1.f / ctl->xl[m];
      const bool valid = rl < cur.z;
      __nv_bfloat16* dst = a.O + ((int64_t)(cur.x + rl) * a.Hq + kvh * a.g + hh) * kD;
      const uint32_t tO = tmem + lane_off + kColO;
#pragma unroll 1
      for (int c = 0; c < kD; c += 32) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tO + c, r);
        tc::tmem_ld_wait();
        if (valid && a.st32) {
          // one 256-bit store per 16 values: the 32 bytes fill one sector
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = pack_bf16x2(__uint_as_float(r[16 * q + 2 * e]) * inv,
                                 __uint_as_float(r[16 * q + 2 * e + 1]) * inv);
            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + c + 16 * q),
                         "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                         "r"(w[7])
                         : "memory");
          }
        } else if (valid) {
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
      tc::mbar_arrive(&ctl->o_empty);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (PAIR) {
    // the other CTA has no copy into, nor arrival on, this one's shared
    // memory in flight (its producers waited for the last phases above)
    __syncwarp();
    tc::cluster_sync_all();
  }
  tc::tc_fence_after();
  if (warp == kWarpS) tc::tmem_dealloc(tmem, kTmemCols);
}

__global__ void attn_tiles_kernel(const fuse_request_t* reqs, int n_req, const int32_t* idx,
                                  int rtile, int4* tiles) {
  pdl_trigger();
  pdl_wait();
  build_attn_tiles(reqs, n_req, idx, rtile, tiles);
}

// Clusters of two CTAs of the paired kernel that can be resident at once
// (two free SMs of one GPC each), per device; 0 when none can.
int resident_pairs() {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  const void* kernel = reinterpret_cast<const void*>(attn_tc_kernel<true>);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (set_dyn_smem_once(kernel, kSmemBytes) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters < 0) {
    cudaGetLastError();
    clusters = 0;
  }
  cache[dev] = clusters;
  return clusters;
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
    e = launch_pdl(attn_tiles_kernel, dim3(1), dim3(128), 0, s, reqs.d_req, reqs.n_req, idx, rtile,
                   tiles);
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
  a.reqs = reqs.d_req;
  a.rows = rows;
  a.O = reinterpret_cast<__nv_bfloat16*>(O);
  a.Hq = d.n_q_heads;
  a.Hkv = d.n_kv_heads;
  a.g = g;
  a.rtile = rtile;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)kD);
  a.err = err;
  a.st32 = (reinterpret_cast<uintptr_t>(O) & 31u) == 0;
  // the tile records and row tables come from the row preparation, which
  // finished before the QKV projection (launched after it) let this kernel
  // start; otherwise the tile kernel launched just above is still running
  a.records_ready = tiles_ready ? 1 : 0;
  // tiles in pairs (clusters of two CTAs) for long contexts, where K and V
  // dominate the data the kernel moves: on a 33 024-token request the pairs
  // raise the power-capped clock and the layer-step's rate by ~1 %; on
  // requests of 4–10 K tokens they cost 0.5–3 % at the full clock
  int64_t longest = 0;
  for (int r = 0; r < reqs.n_req; ++r)
    longest = std::max<int64_t>(longest, reqs.h_req[r].n_ctx + reqs.h_req[r].n_query);
  const int pairs = (n_tiles >= 2 && longest >= kPairMinTokens) ? resident_pairs() : 0;
  if (pairs > 0) {
    a.n_units = (n_tiles + 1) / 2 * d.n_kv_heads;
    const int grid = 2 * (a.n_units < pairs ? a.n_units : pairs);
    return launch_pdl_pairs(attn_tc_kernel<true>, dim3(grid), dim3(kThreads), kSmemBytes, s, mQ,
                            mK, mV, a);
  }
  a.n_units = n_tiles * d.n_kv_heads;
  e = set_dyn_smem_once(reinterpret_cast<const void*>(attn_tc_kernel<false>), kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = a.n_units < sm_count() ? a.n_units : sm_count();
  return launch_pdl(attn_tc_kernel<false>, dim3(grid), dim3(kThreads), kSmemBytes, s, mQ, mK, mV,
                    a);
}

}  // namespace fusekv
