// Tensor-core projection GEMMs for bf16 layers: tcgen05.mma with fp32
// accumulators in tensor memory, operands staged by TMA with 128-byte
// swizzling, fused epilogues.
//
//   deviation (KVBoost Alg. 2 step 2, on V):  C = H W_V^T, and per (token,
//     KV head) the cosine between the fresh V row of the tile and the cached
//     V row, the two heads of a tile summed -> partial[slot, h / 2] (the
//     score, 1 - the sum of a token's partials / Hkv, is formed by the top-k
//     kernel);
//   recompute (QCFuse Eqs. 6-7; KVBoost Eqs. 1-3):  C = Hs [W_Q; W_K; W_V]^T
//     over the gathered rows S, RoPE at each row's request position on Q and
//     K heads, Q to a compact buffer, K and V scattered into the fused cache.
//
// A CTA pair (cluster of two) computes a 256 x 256 output tile with 2-SM MMAs
// (tcgen05.mma.cta_group::2): each CTA holds 128 rows of A and the 128 weight
// rows of one head (the tile's two heads, each from the weight matrix of its
// own head), and the pair's MMA gives each CTA its 128 rows x both heads in
// its own TMEM.  Each SM thus takes in 32 KB of operands per 64-deep step
// instead of the 48 KB a single-SM 128 x 256 tile needs, which is what one
// SM's L2 port can feed at the MMA rate.  The kernel is persistent (one pair
// per two SMs) and warp specialised: warp 0 of each CTA issues TMA loads into
// a 6-stage ring; in the even CTA warp 1 issues the MMAs into one of two TMEM
// accumulators, in the odd CTA warp 1 tells the even one (remote mbarrier
// arrivals) when its stages have landed and its accumulator has been read;
// warps 2-9 (one warpgroup per head) drain the other accumulator through
// tcgen05.ld and run the epilogue, so the epilogue of tile i overlaps the main
// loop of tile i + 1.  The epilogue warps load what they
// read from global memory (cached V rows; work rows and RoPE factors) before
// they wait for the accumulator, so those loads overlap the main loop.
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace fusekv {

namespace {

constexpr int BM = 128;                             // rows of A per CTA (256 per pair)
constexpr int BMP = 2 * BM;                         // rows of a pair tile
constexpr int BN = 128;                             // one head
constexpr int BN2 = 2 * BN;                         // one tile: two heads
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int kTileBytes = BM * BK * 2;             // 16 KB: A, or one head's B rows
constexpr int kStageBytes = 2 * kTileBytes;         // this CTA's A rows + its head's B rows
constexpr int kAccCols = BN2;
constexpr int kTmemCols = 2 * kAccCols;             // two accumulators: all 512 columns
constexpr int kEpiThreads = 256;                    // two warpgroups, one per head
constexpr int kThreads = 64 + kEpiThreads;

enum Mode : int { MODE_DEVIATION = 0, MODE_RECOMPUTE = 1, MODE_SPLITK = 2 };

struct TcArgs {
  int M;                 // rows of A
  int K;                 // hidden
  int m_tiles;           // pair tiles of 256 rows
  int n_tiles;
  int h0, h1;            // heads taken by B map 0 and 1 (map 2 takes the rest)
  int mode;
  int n_q_heads;
  int n_kv_heads;
  // deviation
  const __nv_bfloat16* Vf;
  // cached V read from the chunk caches (bf16, same type as the layer) instead
  // of Vf, so that the stitch may run alongside; null: read Vf
  const fuse_chunk_t* chunks;    // sorted by dst_row, non-overlapping
  int n_chunks;
  int kv_paged;
  int block_size;
  int64_t n_pool_blocks;
  const int32_t* map;            // score slot of every packed row, or null: search reqs
  const fuse_request_t* reqs;    // sorted by row0, non-overlapping (when map is null)
  int n_req;
  float* partial;
  // recompute
  const WorkRow* rows;
  const float2* rope;
  __nv_bfloat16* Q;
  __nv_bfloat16* Kf;
  __nv_bfloat16* Vout;
  uint32_t* err;
  int st32;              // Q, Kf and Vout 32-byte aligned: one 256-bit store per 16 values
  // split over K (MODE_SPLITK): tile t of the K range [ks K / k_splits,
  // (ks + 1) K / k_splits) writes its fp32 accumulator to
  // split_out[(ks * M + m) * split_cols + head * 128 + c]
  int k_splits;
  float* split_out;
  int split_cols;
};

struct SharedCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t peer_tempty[2];     // even CTA: the odd CTA's epilogue has read the accumulator
  uint64_t xc_bar[2];          // [accumulator]: the second head's cosines written
  float xc[2][BM];             // [accumulator][row]: cosine of the tile's second head
  uint32_t tmem_base;
  volatile int abort_flag;
};

// The stages, then the control block, after aligning the base to 1024 bytes
// (up to 1023 bytes of slack).
constexpr int kSmemBytes = STAGES * kStageBytes + 1024 + (int)sizeof(SharedCtl);
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, SharedCtl* ctl) {
  return tc::mbar_wait(bar, parity, &ctl->abort_flag);
}

__device__ __forceinline__ void abort_kernel(SharedCtl* ctl, uint32_t* err) {
  ctl->abort_flag = 1;
  report_error(err, FUSE_ERR_TIMEOUT, SITE_GEMM_TIMEOUT, blockIdx.x);
}

// ---- epilogues (one thread = one row of the tile) -------------------------

// Score slot of packed row m: score0 + t for context token t of its request,
// -1 for query rows and rows outside every request.
__device__ __forceinline__ int32_t row_slot(const TcArgs& a, int m) {
  if (a.map) return a.map[m];
  int lo = 0, hi = a.n_req - 1;
  while (lo < hi) {                       // last request with row0 <= m
    const int mid = (lo + hi + 1) >> 1;
    if (a.reqs[mid].row0 <= m) lo = mid; else hi = mid - 1;
  }
  const fuse_request_t& R = a.reqs[lo];
  const int64_t t = m - R.row0;
  return (t >= 0 && t < R.n_ctx) ? (int32_t)(R.score0 + t) : -1;
}

// Operands of the deviation epilogue of one row and head, loaded before the
// accumulator is ready: the score slot and the cached V row.
struct DevPre {
  int32_t slot;
  uint4 v[BN / 8];
};

// Where the cached V row of packed row m lives: in the chunk cache whose
// fused rows hold m (what the stitch writes to Vf[m]), else in Vf itself (a
// row no chunk covers keeps its contents).  Returns the chunk (null for Vf)
// and the source row (pool row when paged; -1 for an out-of-pool block id,
// which the stitch reports).
__device__ __forceinline__ const fuse_chunk_t* cached_v_chunk(const TcArgs& a, int m,
                                                              int64_t* tok) {
  if (!a.chunks || a.n_chunks == 0) return nullptr;
  int lo = 0, hi = a.n_chunks - 1;
  while (lo < hi) {                       // last chunk with dst_row <= m
    const int mid = (lo + hi + 1) >> 1;
    if (a.chunks[mid].dst_row <= m) lo = mid; else hi = mid - 1;
  }
  const fuse_chunk_t* c = &a.chunks[lo];
  const int64_t r = m - c->dst_row;
  if (r < 0 || r >= c->len) return nullptr;
  *tok = r;
  if (a.kv_paged) {
    const int32_t b = __ldg(c->block_table + r / a.block_size);
    *tok = (b < 0 || b >= a.n_pool_blocks) ? -1 : (int64_t)b * a.block_size + r % a.block_size;
  }
  return c;
}

__device__ __forceinline__ void pre_deviation(const TcArgs& a, int m, int head, DevPre& p) {
  p.slot = m < a.M ? row_slot(a, m) : -1;
  if (p.slot < 0) return;
  int64_t tok = 0;
  const fuse_chunk_t* c = cached_v_chunk(a, m, &tok);
  if (c && tok < 0) {
#pragma unroll
    for (int q = 0; q < BN / 8; ++q) p.v[q] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* vrow = reinterpret_cast<const uint4*>(
      c ? reinterpret_cast<const __nv_bfloat16*>(c->v) + (tok * a.n_kv_heads + head) * BN
        : a.Vf + ((int64_t)m * a.n_kv_heads + head) * BN);
#pragma unroll
  for (int q = 0; q < BN / 8; ++q) p.v[q] = __ldg(vrow + q);
}

// Cosine of this row and head (0 for rows without a score slot).
__device__ __forceinline__ float epi_deviation(uint32_t taddr, const DevPre& p) {
  float dot = 0.f, na = 0.f, nb = 0.f;
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 32) {
    uint32_t r[32];
    tc::tmem_ld_32x32b_x32(taddr + c0, r);
    tc::tmem_ld_wait();
    if (p.slot >= 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = p.v[c0 / 8 + q];
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float f0 = bf16_lo(ww[e]), f1 = bf16_hi(ww[e]);
          const float v0 = __uint_as_float(r[8 * q + 2 * e]);
          const float v1 = __uint_as_float(r[8 * q + 2 * e + 1]);
          dot = fmaf(v0, f0, fmaf(v1, f1, dot));
          na = fmaf(v0, v0, fmaf(v1, v1, na));
          nb = fmaf(f0, f0, fmaf(f1, f1, nb));
        }
      }
    }
  }
  return p.slot >= 0 ? dot / fmaxf(sqrtf(na) * sqrtf(nb), 1e-30f) : 0.f;
}

__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* dst, const float (&x)[16]) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint4 w;
    w.x = pack_bf16x2(x[8 * q + 0], x[8 * q + 1]);
    w.y = pack_bf16x2(x[8 * q + 2], x[8 * q + 3]);
    w.z = pack_bf16x2(x[8 * q + 4], x[8 * q + 5]);
    w.w = pack_bf16x2(x[8 * q + 6], x[8 * q + 7]);
    reinterpret_cast<uint4*>(dst)[q] = w;
  }
}

// The same as one 256-bit store (dst 32-byte aligned): the 32 bytes a thread
// writes fill one sector in one instruction.
__device__ __forceinline__ void store_bf16x16_v8(__nv_bfloat16* dst, const float (&x)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) w[q] = pack_bf16x2(x[2 * q], x[2 * q + 1]);
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Operands of the recompute epilogue of one row and head loaded before the
// accumulator is ready: the destination row and the first RoPE factors.
constexpr int kRopeChunk = 16;                     // rotation pairs per step
struct RecPre {
  __nv_bfloat16* dst;    // null for rows past the end
  bool rot;
  float4 cs[kRopeChunk / 2];                       // (cos, sin) of pairs 0 .. 15
};

__device__ __forceinline__ void pre_recompute(const TcArgs& a, int m, int head, RecPre& p) {
  const int Hq = a.n_q_heads, Hkv = a.n_kv_heads;
  p.dst = nullptr;
  p.rot = head < Hq + Hkv;
  if (m >= a.M) return;
  if (head < Hq) {
    p.dst = a.Q + ((int64_t)m * Hq + head) * BN;
  } else {
    const WorkRow w = a.rows[m];
    p.dst = head < Hq + Hkv ? a.Kf + (w.dst_row * Hkv + (head - Hq)) * BN
                            : a.Vout + (w.dst_row * Hkv + (head - Hq - Hkv)) * BN;
  }
  if (p.rot) {
    // (cos, sin) of pairs 2i, 2i + 1: one float4 at i * M + m (rope_index)
    const float4* cs = reinterpret_cast<const float4*>(a.rope) + m;
#pragma unroll
    for (int i = 0; i < kRopeChunk / 2; ++i) p.cs[i] = __ldg(cs + (int64_t)i * a.M);
  }
}

__device__ __forceinline__ void epi_recompute(const TcArgs& a, uint32_t taddr, int m,
                                              const RecPre& p) {
  const float4* csrow = reinterpret_cast<const float4*>(a.rope) + m;
  float4 cs[kRopeChunk / 2];
#pragma unroll
  for (int i = 0; i < kRopeChunk / 2; ++i) cs[i] = p.cs[i];
#pragma unroll
  for (int j0 = 0; j0 < BN / 2; j0 += kRopeChunk) {
    // the next chunk's factors are on their way while this one is rotated
    float4 nx[kRopeChunk / 2];
    if (p.rot && p.dst && j0 + kRopeChunk < BN / 2) {
#pragma unroll
      for (int i = 0; i < kRopeChunk / 2; ++i)
        nx[i] = __ldg(csrow + (int64_t)((j0 + kRopeChunk) / 2 + i) * a.M);
    }
    uint32_t rx[kRopeChunk], ry[kRopeChunk];
    tc::tmem_ld_32x32b_x16(taddr + j0, rx);
    tc::tmem_ld_32x32b_x16(taddr + j0 + BN / 2, ry);
    tc::tmem_ld_wait();
    if (p.dst) {
      float x[kRopeChunk], y[kRopeChunk];
      if (p.rot) {
#pragma unroll
        for (int i = 0; i < kRopeChunk / 2; ++i) {
          const float4 c = cs[i];                    // (cos, sin) of pairs j0+2i, j0+2i+1
          const float x0 = __uint_as_float(rx[2 * i]), y0 = __uint_as_float(ry[2 * i]);
          const float x1 = __uint_as_float(rx[2 * i + 1]), y1 = __uint_as_float(ry[2 * i + 1]);
          x[2 * i] = fmaf(x0, c.x, -y0 * c.y);
          y[2 * i] = fmaf(y0, c.x, x0 * c.y);
          x[2 * i + 1] = fmaf(x1, c.z, -y1 * c.w);
          y[2 * i + 1] = fmaf(y1, c.z, x1 * c.w);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kRopeChunk; ++i) {
          x[i] = __uint_as_float(rx[i]);
          y[i] = __uint_as_float(ry[i]);
        }
      }
      if (a.st32) {
        store_bf16x16_v8(p.dst + j0, x);
        store_bf16x16_v8(p.dst + j0 + BN / 2, y);
      } else {
        store_bf16x16(p.dst + j0, x);
        store_bf16x16(p.dst + j0 + BN / 2, y);
      }
    }
    if (j0 + kRopeChunk < BN / 2) {
#pragma unroll
      for (int i = 0; i < kRopeChunk / 2; ++i) cs[i] = nx[i];
    }
  }
}

// Tile t of the pair grid: row tile, column tile (two heads) and K split.
// The dimension with fewer tiles varies fastest, so the pairs running at one
// time share the other operand's tiles: a row tile of a tall A (the
// deviation's H) is read from memory once for all its column tiles, a
// weight tile of a wide B (the recompute's) once for all row tiles.
struct TileIdx {
  int mt, nt, kb0, kb1, ks;
};
__device__ __forceinline__ TileIdx tile_idx(const TcArgs& a, int t, int k_blocks) {
  TileIdx x;
  const int mn = a.m_tiles * a.n_tiles;
  x.ks = t / mn;
  const int r = t % mn;
  if (a.n_tiles <= a.m_tiles) {
    x.nt = r % a.n_tiles;
    x.mt = r / a.n_tiles;
  } else {
    x.mt = r % a.m_tiles;
    x.nt = r / a.m_tiles;
  }
  x.kb0 = x.ks * k_blocks / a.k_splits;
  x.kb1 = (x.ks + 1) * k_blocks / a.k_splits;
  return x;
}

// Split-K epilogue: this row's fp32 accumulator of one head, as it is.
__device__ __forceinline__ void epi_splitk(const TcArgs& a, uint32_t taddr, int m, int head,
                                           int ks) {
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 32) {
    uint32_t r[32];
    tc::tmem_ld_32x32b_x32(taddr + c0, r);
    tc::tmem_ld_wait();
    if (m < a.M) {
      float4* dst = reinterpret_cast<float4*>(
          a.split_out + ((int64_t)ks * a.M + m) * a.split_cols + head * BN + c0);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                             __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
    }
  }
}

// B tensor map and first row of head `head` (the heads of map 0, then 1, then 2).
__device__ __forceinline__ void b_map_of(const TcArgs& a, int head, const CUtensorMap* m0,
                                         const CUtensorMap* m1, const CUtensorMap* m2,
                                         const CUtensorMap*& mb, int& nrow) {
  if (head < a.h0) {
    mb = m0;
    nrow = head * BN;
  } else if (head < a.h0 + a.h1) {
    mb = m1;
    nrow = (head - a.h0) * BN;
  } else {
    mb = m2;
    nrow = (head - a.h0 - a.h1) * BN;
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB0,
                   const __grid_constant__ CUtensorMap mapB1, const __grid_constant__ CUtensorMap mapB2,
                   const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + STAGES * kStageBytes);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = tc::cluster_rank();          // 0: issues the pair's MMAs
  const int total = a.m_tiles * a.n_tiles * a.k_splits;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int k_blocks = a.K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&ctl->full[s], 1);
      tc::mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl->tfull[b], 1);
      tc::mbar_init(&ctl->tempty[b], kEpiThreads);
      tc::mbar_init(&ctl->peer_tempty[b], 1);
      tc::mbar_init(&ctl->xc_bar[b], kEpiThreads / 2);
    }
    ctl->abort_flag = 0;
    tc::fence_barrier_init_cluster();
    tc::tma_prefetch_desc(&mapA);
    tc::tma_prefetch_desc(&mapB0);
    tc::tma_prefetch_desc(&mapB1);
    tc::tma_prefetch_desc(&mapB2);
  }
  if (warp == 1) tc::tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
  tc::tc_fence_before();
  tc::cluster_sync_all();      // both CTAs' barriers exist before any remote arrival
  tc::tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // The TMA producer requests the weights (B) of its first stages before
  // waiting on the previous kernel (they are the caller's inputs); every other
  // thread waits first.  Each thread lets the next kernel start only after its
  // own wait: the kernels before this one are then complete (a stitch launched
  // next may write the fused cache; the attention reads the row tables).
  const bool producer = warp == 0 && lane == 0;
  if (!producer) {
    pdl_wait();               // inputs of the previous kernel complete and visible
    pdl_trigger();
  }

  if (warp == 0) {
    // ---------------- TMA producer: this CTA's A rows and its head's B rows ----------------
    if (lane == 0) {
      const uint32_t leader_full = tc::peer_smem(&ctl->full[0], 0);
      int s = 0;
      uint32_t ph = 0;
      bool armed[STAGES];
      uint32_t armed_ph[STAGES];
      for (int i = 0; i < STAGES; ++i) armed[i] = false;
      bool ok = true;
      // B of the first tile's first stages, before the wait
      int pre = 0;
      if (pair < total) {
        const TileIdx t0 = tile_idx(a, pair, k_blocks);
        const int head = 2 * t0.nt + (int)rank;
        const CUtensorMap* mb;
        int nrow;
        b_map_of(a, head, &mapB0, &mapB1, &mapB2, mb, nrow);
        pre = t0.kb1 - t0.kb0 < STAGES ? t0.kb1 - t0.kb0 : STAGES;
        for (int i = 0; i < pre; ++i) {             // stage i, first use: no wait for it
          uint8_t* sa = smem + i * kStageBytes;
          const int kb = t0.kb0 + i;
          if (rank == 0) {
            tc::mbar_arrive_expect_tx(&ctl->full[i], 2 * kStageBytes);
            tc::tma_load_2d(sa + kTileBytes, mb, &ctl->full[i], kb * BK, nrow);
          } else {
            tc::tma_load_2d_pair(sa + kTileBytes, mb, leader_full + i * (uint32_t)sizeof(uint64_t),
                                 kb * BK, nrow);
          }
        }
      }
      pdl_wait();
      pdl_trigger();
      for (int tile = pair; tile < total && ok; tile += n_pairs) {
        const TileIdx tx = tile_idx(a, tile, k_blocks);
        const int head = 2 * tx.nt + (int)rank;
        const CUtensorMap* mb;
        int nrow;
        b_map_of(a, head, &mapB0, &mapB1, &mapB2, mb, nrow);
        const int arow = tx.mt * BMP + (int)rank * BM;
        for (int kb = tx.kb0; kb < tx.kb1; ++kb) {
          if (!wait_or_abort(&ctl->empty[s], ph ^ 1, ctl)) {
            abort_kernel(ctl, a.err);
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * kStageBytes;
          const bool b_done = tile == pair && kb - tx.kb0 < pre;   // armed and B requested above
          if (rank == 0) {
            // the stage is full once both CTAs' bytes have landed
            if (!b_done) tc::mbar_arrive_expect_tx(&ctl->full[s], 2 * kStageBytes);
            tc::tma_load_2d(sa, &mapA, &ctl->full[s], kb * BK, arow);
            if (!b_done) tc::tma_load_2d(sa + kTileBytes, mb, &ctl->full[s], kb * BK, nrow);
          } else {
            const uint32_t lf = leader_full + s * (uint32_t)sizeof(uint64_t);
            tc::tma_load_2d_pair(sa, &mapA, lf, kb * BK, arow);
            if (!b_done) tc::tma_load_2d_pair(sa + kTileBytes, mb, lf, kb * BK, nrow);
          }
          armed[s] = true;
          armed_ph[s] = ph;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // copies still in flight land before the CTA can exit: the even CTA's
      // full barriers count both CTAs' bytes, and the odd CTA leaves only
      // after the even one (cluster barrier at the end)
      if (rank == 0)
        for (int i = 0; i < STAGES; ++i)
          if (armed[i]) tc::mbar_wait(&ctl->full[i], armed_ph[i]);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer of the pair ----------------
      const uint32_t idesc = tc::idesc_bf16_f32(BMP, BN2);
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int tile = pair; tile < total && ok; tile += n_pairs) {
        // both CTAs' epilogues have read this accumulator (previous use)
        if (!wait_or_abort(&ctl->tempty[acc], acc_ph ^ 1, ctl) ||
            !tc::mbar_wait_cluster(&ctl->peer_tempty[acc], acc_ph, &ctl->abort_flag)) {
          abort_kernel(ctl, a.err);
          break;
        }
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kAccCols;
        const TileIdx tx = tile_idx(a, tile, k_blocks);
        for (int kb = tx.kb0; kb < tx.kb1; ++kb) {
          if (!wait_or_abort(&ctl->full[s], ph, ctl)) {
            abort_kernel(ctl, a.err);
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t sa = tc::smem_u32(smem + s * kStageBytes);
          const uint64_t da = tc::smem_desc_k128(sa);
          const uint64_t db = tc::smem_desc_k128(sa + kTileBytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc::mma_bf16_pair(d_tmem, da + 2 * k, db + 2 * k, idesc, (kb != tx.kb0) || k != 0);
          tc::mma_commit_pair(&ctl->empty[s], 0x3);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit_pair(&ctl->tfull[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_ph ^= 1;
      }
    } else if (lane == 0) {
      // ---------------- odd CTA: report its epilogue's reads of each accumulator ----------------
      const uint32_t leader_tempty = tc::peer_smem(&ctl->peer_tempty[0], 0);
      int acc = 0;
      uint32_t acc_ph = 0;
      for (int tile = pair; tile < total; tile += n_pairs) {
        if (!wait_or_abort(&ctl->tempty[acc], acc_ph ^ 1, ctl)) {
          abort_kernel(ctl, a.err);
          break;
        }
        tc::mbar_arrive_remote(leader_tempty + acc * (uint32_t)sizeof(uint64_t));
        acc ^= 1;
        if (acc == 0) acc_ph ^= 1;
      }
    }
  } else {
    // ---------------- epilogue warps 2..9 ----------------
    const int hb = (warp - 2) >> 2;          // head of the tile this warpgroup drains
    const int quarter = warp % 4;            // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int tile = pair; tile < total; tile += n_pairs) {
      const TileIdx tx = tile_idx(a, tile, k_blocks);
      const int nt = tx.nt;
      const int m = tx.mt * BMP + (int)rank * BM + row;
      const int head = 2 * nt + hb;
      // one of the two is used (MODE is a compile-time constant)
      DevPre dp;
      RecPre rp;
      if constexpr (MODE == MODE_DEVIATION)
        pre_deviation(a, m, head, dp);
      else if constexpr (MODE == MODE_RECOMPUTE)
        pre_recompute(a, m, head, rp);
      if (!tc::mbar_wait_warp(&ctl->tfull[acc], acc_ph, &ctl->abort_flag)) {
        abort_kernel(ctl, a.err);
        break;
      }
      tc::tc_fence_after();
      const uint32_t taddr =
          tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * kAccCols + hb * BN;
      if constexpr (MODE == MODE_DEVIATION) {
        const float c = epi_deviation(taddr, dp);
        if (hb == 1) {
          ctl->xc[acc][row] = c;
          tc::mbar_arrive(&ctl->xc_bar[acc]);
        } else {
          // the pair's sum, first head first; xc[acc] is rewritten only after
          // this warpgroup has released the accumulator (tempty) below
          if (!tc::mbar_wait_warp(&ctl->xc_bar[acc], acc_ph, &ctl->abort_flag)) {
            abort_kernel(ctl, a.err);
            break;
          }
          if (dp.slot >= 0) a.partial[(int64_t)dp.slot * (a.n_kv_heads / 2) + nt] = c + ctl->xc[acc][row];
        }
      } else if constexpr (MODE == MODE_RECOMPUTE) {
        epi_recompute(a, taddr, m, rp);
      } else {
        epi_splitk(a, taddr, m, head, tx.ks);
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&ctl->tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1;
    }
  }

  tc::tc_fence_before();
  __syncwarp();               // the cluster barrier is warp-aligned
  tc::cluster_sync_all();     // the pair's MMAs are done with both CTAs' memory
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc_pair(tmem_base, kTmemCols);
}

// ---- host side ---------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major bf16 matrix [rows, cols] read in boxes of 128 rows x 64 columns.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {BK, BM};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTA pairs of this kernel that can be resident at once (clusters of two
// need two free SMs of one GPC), cached per device and kernel.
int resident_pairs(const void* kernel) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> g(mu);
  auto it = cache.find({dev, kernel});
  if (it != cache.end()) return it->second;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int n = std::max(1, sms / 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * n);
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
  if (set_dyn_smem_once(kernel, kSmemBytes) == cudaSuccess &&
      cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) == cudaSuccess && clusters > 0)
    n = std::min(n, clusters);
  else
    cudaGetLastError();
  cache[{dev, kernel}] = n;
  return n;
}

cudaError_t launch(const CUtensorMap& mA, const CUtensorMap& mB0, const CUtensorMap& mB1,
                   const CUtensorMap& mB2, const TcArgs& a, cudaStream_t s) {
  const int total = a.m_tiles * a.n_tiles * a.k_splits;
  if (total == 0) return cudaSuccess;
  auto kernel = a.mode == MODE_DEVIATION   ? gemm_tc_kernel<MODE_DEVIATION>
                : a.mode == MODE_RECOMPUTE ? gemm_tc_kernel<MODE_RECOMPUTE>
                                           : gemm_tc_kernel<MODE_SPLITK>;
  cudaError_t e = set_dyn_smem_once(reinterpret_cast<const void*>(kernel), kSmemBytes);
  if (e != cudaSuccess) return e;
  const int pairs = std::min(total, resident_pairs(reinterpret_cast<const void*>(kernel)));
  return launch_pdl_pairs(kernel, dim3(2 * pairs), dim3(kThreads), kSmemBytes, s, mA, mB0, mB1,
                          mB2, a);
}

}  // namespace

bool tma_encode_available() { return encode_fn() != nullptr; }

// Row-major bf16 tensor of rank 3 (dims innermost first, byte strides of
// dims 1 and 2) read in boxes of `box` elements, 128-byte swizzled.
bool make_map_3d(CUtensorMap* m, const void* base, const uint64_t dims[3], const uint64_t strides[2],
                 const uint32_t box[3]) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t gs[2] = {strides[0], strides[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gd, gs, bx, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_gemm_supported(const fuse_layer_desc_t& d) {
  // tiles pair heads: even head counts keep a pair inside Q, inside K/V or
  // across the K/V boundary (handled by per-half weight maps)
  return d.dtype == FUSE_BF16 && d.head_dim == 128 && d.hidden % BK == 0 &&
         d.n_q_heads % 2 == 0 && d.n_kv_heads % 2 == 0 && encode_fn() != nullptr;
}

cudaError_t launch_deviation_partials_tc(const fuse_layer_desc_t& d, int64_t n_rows, const void* H,
                                         const void* Wv, const void* Vf, const int32_t* map,
                                         const fuse_request_t* d_req, int n_req, float* partial,
                                         const fuse_chunks_t* v_chunks, uint32_t* err,
                                         cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  CUtensorMap mA, mB;
  if (!make_map(&mA, H, n_rows, d.hidden) ||
      !make_map(&mB, Wv, (int64_t)d.n_kv_heads * d.head_dim, d.hidden))
    return cudaErrorInvalidValue;
  TcArgs a = {};
  a.M = (int)n_rows;
  a.K = d.hidden;
  a.m_tiles = (int)((n_rows + BMP - 1) / BMP);
  a.n_tiles = d.n_kv_heads / 2;
  a.h0 = d.n_kv_heads;
  a.h1 = 0;
  a.mode = MODE_DEVIATION;
  a.k_splits = 1;
  a.n_q_heads = d.n_q_heads;
  a.n_kv_heads = d.n_kv_heads;
  a.Vf = reinterpret_cast<const __nv_bfloat16*>(Vf);
  a.map = map;
  a.reqs = d_req;
  a.n_req = n_req;
  a.partial = partial;
  if (v_chunks) {
    a.chunks = v_chunks->d_chunks;
    a.n_chunks = v_chunks->n_chunks;
    a.kv_paged = v_chunks->kv_layout == FUSE_KV_PAGED;
    a.block_size = v_chunks->block_size > 0 ? v_chunks->block_size : 1;
    a.n_pool_blocks = v_chunks->n_pool_blocks;
  }
  a.err = err;
  return launch(mA, mB, mB, mB, a, s);
}

int deviation_tc_ctas(const fuse_layer_desc_t& d, int64_t n_rows) {
  const int64_t tiles = ((n_rows + BMP - 1) / BMP) * (d.n_kv_heads / 2);
  const int pairs =
      resident_pairs(reinterpret_cast<const void*>(gemm_tc_kernel<MODE_DEVIATION>));
  return 2 * (int)std::min<int64_t>(tiles, pairs);
}

cudaError_t launch_project_recompute_tc(const fuse_layer_desc_t& d, int64_t n_rows,
                                        const WorkRow* rows, const float2* rope, const void* H,
                                        const void* Wq, const void* Wk, const void* Wv, void* Q,
                                        void* Kf, void* Vf, void* Hs, uint32_t* err,
                                        cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  CUtensorMap mA, mQ, mK, mV;
  const int64_t kv = (int64_t)d.n_kv_heads * d.head_dim;
  if (!make_map(&mA, Hs, n_rows, d.hidden) ||
      !make_map(&mQ, Wq, (int64_t)d.n_q_heads * d.head_dim, d.hidden) ||
      !make_map(&mK, Wk, kv, d.hidden) || !make_map(&mV, Wv, kv, d.hidden))
    return cudaErrorInvalidValue;
  TcArgs a = {};
  a.M = (int)n_rows;
  a.K = d.hidden;
  a.m_tiles = (int)((n_rows + BMP - 1) / BMP);
  a.n_tiles = (d.n_q_heads + 2 * d.n_kv_heads) / 2;
  a.h0 = d.n_q_heads;
  a.h1 = d.n_kv_heads;
  a.mode = MODE_RECOMPUTE;
  a.k_splits = 1;
  a.n_q_heads = d.n_q_heads;
  a.n_kv_heads = d.n_kv_heads;
  a.rows = rows;
  a.rope = rope;
  a.Q = reinterpret_cast<__nv_bfloat16*>(Q);
  a.Kf = reinterpret_cast<__nv_bfloat16*>(Kf);
  a.Vout = reinterpret_cast<__nv_bfloat16*>(Vf);
  a.st32 = ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(Kf) |
             reinterpret_cast<uintptr_t>(Vf)) & 31u) == 0;
  a.err = err;
  return launch(mA, mQ, mK, mV, a, s);
}

namespace {

// Sum of the K splits in a fixed order, RoPE at each row's position, bf16 out:
// one block per (row, four heads), one thread per (head, rotation pair); the
// splits' loads are all issued before the sum.
constexpr int kMaxSplits = 8;
__global__ void __launch_bounds__(256) splitk_rope_kernel(const float* part, int k_splits, int M,
                                                          int n_heads, const float2* rope,
                                                          __nv_bfloat16* Q) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x;
  const int head = blockIdx.y * 4 + threadIdx.x / (BN / 2), j = threadIdx.x % (BN / 2);
  if (head >= n_heads) return;
  const int cols = n_heads * BN;
  float xs[kMaxSplits], ys[kMaxSplits];
#pragma unroll
  for (int ks = 0; ks < kMaxSplits; ++ks) {
    if (ks < k_splits) {
      const float* p = part + ((int64_t)ks * M + m) * cols + head * BN;
      xs[ks] = __ldg(p + j);
      ys[ks] = __ldg(p + j + BN / 2);
    }
  }
  float x = 0.f, y = 0.f;
#pragma unroll
  for (int ks = 0; ks < kMaxSplits; ++ks) {
    if (ks < k_splits) {
      x += xs[ks];
      y += ys[ks];
    }
  }
  const float2 c = rope[rope_index(j, m, M)];
  __nv_bfloat16* o = Q + ((int64_t)m * n_heads + head) * BN;
  o[j] = __float2bfloat16_rn(fmaf(x, c.x, -y * c.y));
  o[j + BN / 2] = __float2bfloat16_rn(fmaf(y, c.x, x * c.y));
}

}  // namespace

// Splits over K for a projection of n_rows rows onto n_heads heads: enough
// for the pair tiles to cover the resident pairs, at least four 64-deep
// steps each, at most 8.
int query_k_splits(const fuse_layer_desc_t& d, int64_t n_rows, int n_heads) {
  const int64_t tiles = ((n_rows + BMP - 1) / BMP) * (n_heads / 2);
  const int pairs = resident_pairs(reinterpret_cast<const void*>(gemm_tc_kernel<MODE_SPLITK>));
  int64_t ks = std::max<int64_t>(1, pairs / std::max<int64_t>(tiles, 1));
  ks = std::min<int64_t>(ks, std::max(1, d.hidden / BK / 4));
  return (int)std::min<int64_t>(ks, kMaxSplits);
}

// Q heads only (query-aware scoring): Q[m] = R^{pos} W_Q Hs[m]; no K/V scatter.
// With split_ws (room for max_splits * n_rows * Hq * 128 floats) and more
// than one split, the pair tiles split K and a second launch sums the splits
// in order and rotates; otherwise the recompute epilogue rotates.
cudaError_t launch_project_query_tc(const fuse_layer_desc_t& d, int64_t n_rows, const float2* rope,
                                    const void* Wq, void* Q, const void* Hs, uint32_t* err,
                                    cudaStream_t s, float* split_ws, int max_splits) {
  if (n_rows == 0) return cudaSuccess;
  CUtensorMap mA, mQ;
  if (!make_map(&mA, Hs, n_rows, d.hidden) ||
      !make_map(&mQ, Wq, (int64_t)d.n_q_heads * d.head_dim, d.hidden))
    return cudaErrorInvalidValue;
  TcArgs a = {};
  a.M = (int)n_rows;
  a.K = d.hidden;
  a.m_tiles = (int)((n_rows + BMP - 1) / BMP);
  a.n_tiles = d.n_q_heads / 2;
  a.h0 = d.n_q_heads;
  a.h1 = 0;
  a.mode = MODE_RECOMPUTE;
  a.k_splits = 1;
  a.n_q_heads = d.n_q_heads;
  a.n_kv_heads = d.n_kv_heads;
  a.rope = rope;
  a.Q = reinterpret_cast<__nv_bfloat16*>(Q);
  a.st32 = (reinterpret_cast<uintptr_t>(Q) & 31u) == 0;
  a.err = err;
  const int ks = split_ws ? std::min(max_splits, query_k_splits(d, n_rows, d.n_q_heads)) : 1;
  if (ks <= 1) return launch(mA, mQ, mQ, mQ, a, s);
  a.mode = MODE_SPLITK;
  a.k_splits = ks;
  a.split_out = split_ws;
  a.split_cols = d.n_q_heads * BN;
  cudaError_t e = launch(mA, mQ, mQ, mQ, a, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(splitk_rope_kernel, dim3((unsigned)n_rows, (d.n_q_heads + 3) / 4), dim3(256),
                    0, s, (const float*)split_ws, ks, (int)n_rows, d.n_q_heads, rope,
                    reinterpret_cast<__nv_bfloat16*>(Q));
}

}  // namespace fusekv
