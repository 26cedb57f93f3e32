// Stitch + RoPE re-rotation (+ KIVI int8 / int4 dequantisation, + paged gather).
//
// QCFuse (section 2.1.2, Eq. 4): chunk caches built alone at local positions
// are placed at their request positions; keys are remapped by the chunk's
// position offset o_i, values are copied in token order.  KVBoost (section
// 3.2): a key cached with R^r and reused at o_i + r needs the correction
// R^{o_i}.  KVBoost (section 4.5, Eq. 7): x = zero + q * scale, keys with
// per-channel statistics, values with per-token statistics.
//
// Memory-bound.  When the chunk caches have the layer's element type (no
// dequantisation), stitch_bulk_kernel streams them: persistent CTAs (two per
// SM), each working through a contiguous range of row tiles with a 3-stage
// shared-memory ring filled by 1-D bulk copies; the threads rotate the key
// tile in place and bulk stores write both tiles to the fused cache (values
// pass through untouched).  For int8 codes stitch_u8_kernel: tiles of a few
// rows of one chunk; each thread owns 16 key pairs and two groups of 16
// values, and every load of a tile (16-byte code loads, the values'
// per-token scales, the chunk's per-channel key scales into shared memory) is
// issued before the first use.  Otherwise (int4 codes, or a type change)
// stitch_kernel, the same scheme with 8-element groups.  Either way the chunk
// offset's (cos, sin) of the d/2 frequencies are computed once per CTA (and
// chunk) into shared memory.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace fusekv {

namespace {

constexpr int kStitchThreads = 256;
constexpr int kStitchItems = 2;      // V 16-byte groups per thread at most
constexpr int kStitchKItems = kStitchItems / 2;   // K pair groups: half as many as V groups

template <typename TS> struct Src8;

template <> struct Src8<float> {
  static __device__ __forceinline__ void load(const void* base, int64_t e, float (&x)[8]) {
    Vec8<float>::load(reinterpret_cast<const float*>(base) + e, x);
  }
};
template <> struct Src8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const void* base, int64_t e, float (&x)[8]) {
    Vec8<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16*>(base) + e, x);
  }
};
// Four-bit codes packed two per byte (element 2m in the low nibble of byte
// m): the tag type of the kernel's source argument.
struct Nibbles {
  uint8_t b;
};
// 8 four-bit codes from element e (a multiple of 8: 4 bytes at byte e / 2).
__device__ __forceinline__ void load_u4(const void* base, int64_t e, float (&x)[8]) {
  const uint32_t q = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(base) + e / 2));
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = (float)((q >> (4 * i)) & 0xFu);
}
// uint8 codes, dequantised with 8 per-element (scale, zero) pairs.
__device__ __forceinline__ void load_u8(const void* base, int64_t e, float (&x)[8]) {
  uint2 q = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(base) + e));
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = (float)((q.x >> (8 * i)) & 0xFFu);
#pragma unroll
  for (int i = 0; i < 4; ++i) x[4 + i] = (float)((q.y >> (8 * i)) & 0xFFu);
}
__device__ __forceinline__ void load_h8(const void* base, int64_t e, float (&x)[8]) {
  uint4 a = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(base) + e));
  const __half2* h = reinterpret_cast<const __half2*>(&a);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

template <typename TO> struct Dst8 {
  static __device__ __forceinline__ void store(void* base, int64_t e, const float (&x)[8]) {
    Vec8<TO>::store(reinterpret_cast<TO*>(base) + e, x);
  }
};

struct StitchArgs {
  int rows_per_cta;
  const fuse_chunk_t* chunks;
  void* Kf;
  void* Vf;
  uint32_t* err;
  int64_t n_pool_blocks;
  int32_t n_kv_heads;
  int32_t block_size;
  int32_t tiles_per_chunk;
  int32_t wait_first;         // int8 kernel: 0 = the previous kernel (which reads no
                              // output of this one) is waited for only at the end
  RopeFreqs freqs;
};

// Element offset of (local row r, head h, column j) of a chunk, or -1 if the
// paged block id is out of range.
template <bool PAGED, int D>
__device__ __forceinline__ int64_t chunk_elem(const fuse_chunk_t& c, int r, int h, int j,
                                              int Hkv, int bs, int64_t nblk, int64_t* tok_out) {
  int64_t tok;
  if (PAGED) {
    const int32_t b = __ldg(c.block_table + r / bs);
    if (b < 0 || b >= nblk) return -1;
    tok = (int64_t)b * bs + (r % bs);
  } else {
    tok = r;
  }
  *tok_out = tok;
  return (tok * Hkv + h) * D + j;
}

template <typename TS, typename TO, int D, bool PAGED>
__global__ void __launch_bounds__(kStitchThreads) stitch_kernel(const StitchArgs a) {
  constexpr int H2 = D / 2;
  constexpr int PG = H2 / 8;           // 8-pair groups per head (K)
  constexpr int VG = D / 8;            // 8-element groups per head (V)
  constexpr bool kU4 = std::is_same<TS, Nibbles>::value;
  constexpr bool kU8 = std::is_same<TS, uint8_t>::value || kU4;   // quantised codes
  constexpr bool kSame = sizeof(TS) == sizeof(TO) && !kU8;
  pdl_trigger();
  pdl_wait();
  const int chunk = blockIdx.x / a.tiles_per_chunk;
  const int tile = blockIdx.x % a.tiles_per_chunk;
  const fuse_chunk_t c = a.chunks[chunk];
  const int r0 = tile * a.rows_per_cta;
  if (r0 >= c.len) return;
  const int nrows = min(a.rows_per_cta, c.len - r0);
  const int Hkv = a.n_kv_heads;
  const int t = threadIdx.x;
  const int g = t % PG;                // this thread's pair group (fixed for all its K items)
  const int j0 = g * 8;
  const int k_items = nrows * Hkv * PG;
  const int v_items = nrows * Hkv * VG;

  // 1. issue every load of this thread first, so they are all in flight together
  float kx[kStitchKItems][8], ky[kStitchKItems][8], vx[kStitchItems][8];
  int64_t k_tok[kStitchKItems], v_tok[kStitchItems];
  bool k_ok[kStitchKItems], v_ok[kStitchItems];
#pragma unroll
  for (int q = 0; q < kStitchKItems; ++q) {
    const int it = t + q * kStitchThreads;
    k_ok[q] = false;
    if (it < k_items) {
      const int rh = it / PG;
      const int r = r0 + rh / Hkv;
      const int h = rh % Hkv;
      const int64_t e = chunk_elem<PAGED, D>(c, r, h, j0, Hkv, a.block_size, a.n_pool_blocks, &k_tok[q]);
      if (e < 0) {
        report_error(a.err, FUSE_ERR_DEVICE_BOUNDS, SITE_STITCH_BLOCK, chunk);
      } else {
        k_ok[q] = true;
        if constexpr (kU4) {
          load_u4(c.k, e, kx[q]);
          load_u4(c.k, e + H2, ky[q]);
        } else if constexpr (kU8) {
          load_u8(c.k, e, kx[q]);
          load_u8(c.k, e + H2, ky[q]);
        } else {
          Src8<TS>::load(c.k, e, kx[q]);
          Src8<TS>::load(c.k, e + H2, ky[q]);
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kStitchItems; ++q) {
    const int it = t + q * kStitchThreads;
    v_ok[q] = false;
    if (it < v_items) {
      const int gv = it % VG;
      const int rh = it / VG;
      const int r = r0 + rh / Hkv;
      const int h = rh % Hkv;
      const int64_t e = chunk_elem<PAGED, D>(c, r, h, gv * 8, Hkv, a.block_size, a.n_pool_blocks, &v_tok[q]);
      if (e < 0) {
        report_error(a.err, FUSE_ERR_DEVICE_BOUNDS, SITE_STITCH_BLOCK, chunk);
      } else {
        v_ok[q] = true;
        if constexpr (kU4)
          load_u4(c.v, e, vx[q]);
        else if constexpr (kU8)
          load_u8(c.v, e, vx[q]);
        else
          Src8<TS>::load(c.v, e, vx[q]);
      }
    }
  }

  // 2. the chunk offset's cos/sin of every frequency, once per CTA, while the
  //    loads fly
  __shared__ float s_cs[kMaxHalfDim], s_sn[kMaxHalfDim];
  const bool rotate = !(kSame && c.pos == 0);
  if (rotate && t < H2) rope_cos_sin(c.pos, a.freqs.hi[t], a.freqs.mid[t], a.freqs.lo[t], s_cs[t], s_sn[t]);
  __syncthreads();
  float cs[8], sn[8];
  if (rotate) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      cs[i] = s_cs[j0 + i];
      sn[i] = s_sn[j0 + i];
    }
  }

  // 3. keys: dequantise, rotate by R^{pos}, store
#pragma unroll
  for (int q = 0; q < kStitchKItems; ++q) {
    if (!k_ok[q]) continue;
    const int it = t + q * kStitchThreads;
    const int rh = it / PG;
    const int r = r0 + rh / Hkv;
    const int h = rh % Hkv;
    float* x = kx[q];
    float* y = ky[q];
    if constexpr (kU8) {
      float sx[8], zx[8], sy[8], zy[8];
      load_h8(c.k_scale, h * D + j0, sx);
      load_h8(c.k_zero, h * D + j0, zx);
      load_h8(c.k_scale, h * D + j0 + H2, sy);
      load_h8(c.k_zero, h * D + j0 + H2, zy);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[i] = fmaf(x[i], sx[i], zx[i]);
        y[i] = fmaf(y[i], sy[i], zy[i]);
      }
    }
    if (rotate) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float xr = fmaf(x[i], cs[i], -y[i] * sn[i]);
        const float yr = fmaf(y[i], cs[i], x[i] * sn[i]);
        x[i] = xr;
        y[i] = yr;
      }
    }
    const int64_t o = ((c.dst_row + r) * Hkv + h) * D + j0;
    Dst8<TO>::store(a.Kf, o, kx[q]);
    Dst8<TO>::store(a.Kf, o + H2, ky[q]);
  }

  // 4. values: dequantise, store
#pragma unroll
  for (int q = 0; q < kStitchItems; ++q) {
    if (!v_ok[q]) continue;
    const int it = t + q * kStitchThreads;
    const int gv = it % VG;
    const int rh = it / VG;
    const int r = r0 + rh / Hkv;
    const int h = rh % Hkv;
    if constexpr (kU8) {
      const int64_t sidx = v_tok[q] * Hkv + h;
      const float s = __half2float(reinterpret_cast<const __half*>(c.v_scale)[sidx]);
      const float z = __half2float(reinterpret_cast<const __half*>(c.v_zero)[sidx]);
#pragma unroll
      for (int i = 0; i < 8; ++i) vx[q][i] = fmaf(vx[q][i], s, z);
    }
    Dst8<TO>::store(a.Vf, ((c.dst_row + r) * Hkv + h) * D + gv * 8, vx[q]);
  }
}

// ---- int8 codes: 16-byte code loads, all loads of a tile issued first -------
// A CTA of 128 threads moves tiles of `rows_per_cta` rows of one chunk (the
// rows of a tile lie in one pool block when paged).  Thread t owns one key
// item -- 16 pairs (j, j + d/2) of one (row, head), two 16-byte code loads --
// and two value items of 16 codes each, with their per-token scale and zero.
// The chunk's per-channel key scales and zeros go to shared memory (16-byte
// loads), read back as 16-byte vectors.  Every global load of a tile is
// issued before the first use, so a tile takes one round trip to memory
// before it is computed and stored.  The kernel walks a contiguous range of
// tiles per CTA; it is launched with one CTA per tile.
constexpr int kU8Threads = 128;
constexpr int kU8MaxRowElems = 2048;                 // Hkv * d of one row (rows per CTA >= 2)

// Element i of 16 fp16 values held as two 16-byte words, as a float.
__device__ __forceinline__ float half16(const uint4 (&w)[2], int i) {
  const uint4 q = w[i >> 3];
  const uint32_t v[4] = {q.x, q.y, q.z, q.w};
  const uint32_t b = v[(i >> 1) & 3] >> (16 * (i & 1));
  return __half2float(__ushort_as_half((unsigned short)(b & 0xFFFFu)));
}

__device__ __forceinline__ void codes16(const uint4 q, float (&x)[16]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = (float)((w[i >> 2] >> (8 * (i & 3))) & 0xFFu);
}

template <typename TO, int D, bool PAGED>
__global__ void __launch_bounds__(kU8Threads, 8) stitch_u8_kernel(const StitchArgs a, int n_tiles) {
  constexpr int H2 = D / 2;
  constexpr int KG = H2 / 16;          // 16-pair key items per head
  constexpr int VG = D / 16;           // 16-code value items per head
  __shared__ __align__(16) __half s_ks[kU8MaxRowElems], s_kz[kU8MaxRowElems];
  __shared__ float s_cs[kMaxHalfDim], s_sn[kMaxHalfDim];
  pdl_trigger();
  if (a.wait_first) pdl_wait();
  const int Hkv = a.n_kv_heads;
  const int t = threadIdx.x;
  const int per = (n_tiles + gridDim.x - 1) / gridDim.x;
  const int t0 = blockIdx.x * per, t1 = min(n_tiles, t0 + per);
  int table_chunk = -1;                // chunk whose scales and cos/sin are in shared memory
  for (int tile = t0; tile < t1; ++tile) {
    const int chunk = tile / a.tiles_per_chunk;
    const fuse_chunk_t c = a.chunks[chunk];
    const int r0 = (tile % a.tiles_per_chunk) * a.rows_per_cta;
    if (r0 >= c.len) continue;         // CTA-uniform
    const int nrows = min(a.rows_per_cta, c.len - r0);
    int64_t tok0 = r0;                 // source row of r0 (pool row when paged)
    if (PAGED) {
      const int32_t b = __ldg(c.block_table + r0 / a.block_size);
      if (b < 0 || b >= a.n_pool_blocks) {               // CTA-uniform
        if (t == 0) report_error(a.err, FUSE_ERR_DEVICE_BOUNDS, SITE_STITCH_BLOCK, chunk);
        continue;
      }
      tok0 = (int64_t)b * a.block_size + r0 % a.block_size;
    }
    const uint8_t* kc = reinterpret_cast<const uint8_t*>(c.k);
    const uint8_t* vc = reinterpret_cast<const uint8_t*>(c.v);
    const int k_items = nrows * Hkv * KG, v_items = nrows * Hkv * VG;

    // 1. every load of the tile first
    uint4 kq0 = make_uint4(0, 0, 0, 0), kq1 = kq0, vq[2] = {kq0, kq0};
    float vs[2] = {0.f, 0.f}, vz[2] = {0.f, 0.f};
    if (t < k_items) {
      const int rh = t / KG;
      const int64_t e = ((tok0 + rh / Hkv) * Hkv + rh % Hkv) * D + (t % KG) * 16;
      kq0 = __ldg(reinterpret_cast<const uint4*>(kc + e));
      kq1 = __ldg(reinterpret_cast<const uint4*>(kc + e + H2));
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int it = t + q * kU8Threads;
      if (it < v_items) {
        const int rh = it / VG;
        const int64_t th = (tok0 + rh / Hkv) * Hkv + rh % Hkv;
        vq[q] = __ldg(reinterpret_cast<const uint4*>(vc + th * D + (it % VG) * 16));
        vs[q] = __half2float(reinterpret_cast<const __half*>(c.v_scale)[th]);
        vz[q] = __half2float(reinterpret_cast<const __half*>(c.v_zero)[th]);
      }
    }
    const bool rotate = c.pos != 0;
    if (chunk != table_chunk) {        // CTA-uniform
      __syncthreads();                 // the previous chunk's tables are read out
      for (int i = t * 8; i < Hkv * D; i += kU8Threads * 8) {
        *reinterpret_cast<uint4*>(s_ks + i) = __ldg(reinterpret_cast<const uint4*>(
            reinterpret_cast<const __half*>(c.k_scale) + i));
        *reinterpret_cast<uint4*>(s_kz + i) = __ldg(reinterpret_cast<const uint4*>(
            reinterpret_cast<const __half*>(c.k_zero) + i));
      }
      // 2. the chunk offset's cos/sin of every frequency, while the loads fly
      if (rotate && t < H2)
        rope_cos_sin(c.pos, a.freqs.hi[t], a.freqs.mid[t], a.freqs.lo[t], s_cs[t], s_sn[t]);
      __syncthreads();
      table_chunk = chunk;
    }

    // 3. keys: x = zero + q * scale per channel, rotated by R^{pos}
    if (t < k_items) {
      const int rh = t / KG;
      const int r = rh / Hkv, h = rh % Hkv;
      const int j0 = (t % KG) * 16;
      float x[16], y[16];
      codes16(kq0, x);
      codes16(kq1, y);
      const uint4* ks = reinterpret_cast<const uint4*>(s_ks + h * D + j0);
      const uint4* kz = reinterpret_cast<const uint4*>(s_kz + h * D + j0);
      const uint4 sx[2] = {ks[0], ks[1]}, zx[2] = {kz[0], kz[1]};
      const uint4 sy[2] = {ks[H2 / 8], ks[H2 / 8 + 1]}, zy[2] = {kz[H2 / 8], kz[H2 / 8 + 1]};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        x[i] = fmaf(x[i], half16(sx, i), half16(zx, i));
        y[i] = fmaf(y[i], half16(sy, i), half16(zy, i));
      }
      if (rotate) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float cs = s_cs[j0 + i], sn = s_sn[j0 + i];
          const float xr = fmaf(x[i], cs, -y[i] * sn);
          const float yr = fmaf(y[i], cs, x[i] * sn);
          x[i] = xr;
          y[i] = yr;
        }
      }
      TO* dst = reinterpret_cast<TO*>(a.Kf) + ((c.dst_row + r0 + r) * Hkv + h) * D + j0;
      Vec8<TO>::store(dst, *reinterpret_cast<float(*)[8]>(x));
      Vec8<TO>::store(dst + 8, *reinterpret_cast<float(*)[8]>(x + 8));
      Vec8<TO>::store(dst + H2, *reinterpret_cast<float(*)[8]>(y));
      Vec8<TO>::store(dst + H2 + 8, *reinterpret_cast<float(*)[8]>(y + 8));
    }
    // 4. values: x = zero + q * scale per token
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int it = t + q * kU8Threads;
      if (it < v_items) {
        const int rh = it / VG;
        float x[16];
        codes16(vq[q], x);
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = fmaf(x[i], vs[q], vz[q]);
        TO* dst = reinterpret_cast<TO*>(a.Vf) + ((c.dst_row + r0 + rh / Hkv) * Hkv + rh % Hkv) * D +
                  (it % VG) * 16;
        Vec8<TO>::store(dst, *reinterpret_cast<float(*)[8]>(x));
        Vec8<TO>::store(dst + 8, *reinterpret_cast<float(*)[8]>(x + 8));
      }
    }
  }
  // completing implies the previous kernel completed, for the kernels after
  if (!a.wait_first) pdl_wait();
}

// ---- streamed path (chunk storage type == layer type) ------------------------
constexpr int kBulkThreads = 256;
constexpr int kBulkStages = 3;
constexpr int kBulkTileBytes = 16384;              // K tile or V tile, at most
constexpr int kBulkSmem = kBulkStages * 2 * kBulkTileBytes;

struct BulkArgs {
  const fuse_chunk_t* chunks;
  void* Kf;
  void* Vf;
  uint32_t* err;
  int64_t n_pool_blocks;
  int32_t n_kv_heads;
  int32_t block_size;
  int32_t rt;                 // rows per tile; divides block_size when paged
  int32_t tiles_per_chunk;
  int32_t total_tiles;
  int32_t wait_first;         // 0: the previous kernel (which reads no output of
                              // this one) is waited for only at the end
  RopeFreqs freqs;
};

struct BulkTile {
  int chunk, r0, nrows;       // nrows 0: nothing to do
  int64_t src_row;            // first source row (pool row when paged)
};

template <bool PAGED>
__device__ __forceinline__ BulkTile bulk_tile(const BulkArgs& a, int tile, const fuse_chunk_t& c) {
  BulkTile x;
  x.chunk = tile / a.tiles_per_chunk;
  x.r0 = (tile % a.tiles_per_chunk) * a.rt;
  x.nrows = max(0, min(a.rt, c.len - x.r0));
  x.src_row = x.r0;
  if (PAGED && x.nrows > 0) {
    const int32_t b = __ldg(c.block_table + x.r0 / a.block_size);
    if (b < 0 || b >= a.n_pool_blocks) {
      x.nrows = 0;            // reported by the caller
      x.src_row = -1;
    } else {
      x.src_row = (int64_t)b * a.block_size + x.r0 % a.block_size;
    }
  }
  return x;
}

template <typename T, int D, bool PAGED>
__global__ void __launch_bounds__(kBulkThreads) stitch_bulk_kernel(const BulkArgs a) {
  constexpr int H2 = D / 2;
  constexpr int PG = H2 / 8;                         // 8-pair groups per head
  extern __shared__ __align__(128) uint8_t ring[];   // stage s: K tile, then V tile
  __shared__ __align__(8) uint64_t full[kBulkStages];
  __shared__ float s_cs[kMaxHalfDim], s_sn[kMaxHalfDim];
  __shared__ int s_abort;
  const int t = threadIdx.x;
  const int Hkv = a.n_kv_heads;
  const int64_t row_elems = (int64_t)Hkv * D;
  const uint32_t row_bytes = (uint32_t)(row_elems * sizeof(T));
  const int per = (a.total_tiles + gridDim.x - 1) / gridDim.x;
  const int t0 = blockIdx.x * per;
  const int t1 = min(a.total_tiles, t0 + per);
  pdl_trigger();
  if (t == 0) {
    for (int s = 0; s < kBulkStages; ++s) tc::mbar_init(&full[s], 1);
    s_abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (a.wait_first) pdl_wait();
  // thread 0 fills stage (i % 3) with tile t0 + i; a stage's barrier completes
  // one phase per non-empty tile, so both sides count phases per stage
  uint32_t issued[kBulkStages] = {0, 0, 0}, used[kBulkStages] = {0, 0, 0};
  auto fill = [&](int i) {
    const int tile = t0 + i;
    const fuse_chunk_t c = a.chunks[tile / a.tiles_per_chunk];
    const BulkTile x = bulk_tile<PAGED>(a, tile, c);
    if (x.src_row < 0) report_error(a.err, FUSE_ERR_DEVICE_BOUNDS, SITE_STITCH_BLOCK, x.chunk);
    if (x.nrows == 0) return;
    const int s = i % kBulkStages;
    const uint32_t bytes = (uint32_t)x.nrows * row_bytes;
    uint8_t* st = ring + s * 2 * kBulkTileBytes;
    ++issued[s];
    tc::mbar_arrive_expect_tx(&full[s], 2 * bytes);
    tc::bulk_g2s(st, reinterpret_cast<const T*>(c.k) + x.src_row * row_elems, bytes, &full[s]);
    tc::bulk_g2s(st + kBulkTileBytes, reinterpret_cast<const T*>(c.v) + x.src_row * row_elems, bytes,
                 &full[s]);
  };
  if (t == 0)
    for (int i = 0; i < kBulkStages && t0 + i < t1; ++i) fill(i);
  int table_chunk = -1;
  for (int i = 0; t0 + i < t1; ++i) {
    const int tile = t0 + i;
    const fuse_chunk_t c = a.chunks[tile / a.tiles_per_chunk];
    const BulkTile x = bulk_tile<PAGED>(a, tile, c);
    const int s = i % kBulkStages;
    uint8_t* st = ring + s * 2 * kBulkTileBytes;
    if (x.nrows > 0) {
      if (!tc::mbar_wait(&full[s], used[s] & 1, &s_abort)) {
        if (atomicExch(&s_abort, 1) == 0)
          report_error(a.err, FUSE_ERR_TIMEOUT, SITE_STITCH_TIMEOUT, blockIdx.x);
      }
      ++used[s];
      __syncthreads();
      if (s_abort) break;                               // block-uniform after the barrier
      if (c.pos != 0) {
        if (x.chunk != table_chunk) {                  // block-uniform
          if (t < H2) rope_cos_sin(c.pos, a.freqs.hi[t], a.freqs.mid[t], a.freqs.lo[t], s_cs[t], s_sn[t]);
          __syncthreads();
          table_chunk = x.chunk;
        }
        T* k = reinterpret_cast<T*>(st);
        const int items = x.nrows * Hkv * PG;
        for (int it = t; it < items; it += kBulkThreads) {
          const int g = it % PG;
          T* p = k + (int64_t)(it / PG) * D + g * 8;   // (row, head) base + pair group
          float xv[8], yv[8];
          Vec8<T>::load_shared(p, xv);
          Vec8<T>::load_shared(p + H2, yv);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float cs = s_cs[g * 8 + q], sn = s_sn[g * 8 + q];
            const float xr = fmaf(xv[q], cs, -yv[q] * sn);
            const float yr = fmaf(yv[q], cs, xv[q] * sn);
            xv[q] = xr;
            yv[q] = yr;
          }
          Vec8<T>::store(p, xv);
          Vec8<T>::store(p + H2, yv);
        }
        tc::fence_proxy_async_smem();
      }
      __syncthreads();                                  // the tile is final in shared memory
      if (t == 0) {
        const uint32_t bytes = (uint32_t)x.nrows * row_bytes;
        const int64_t dst = (c.dst_row + x.r0) * row_elems;
        tc::bulk_s2g(reinterpret_cast<T*>(a.Kf) + dst, st, bytes);
        tc::bulk_s2g(reinterpret_cast<T*>(a.Vf) + dst, st + kBulkTileBytes, bytes);
        tc::bulk_commit();
      }
    }
    if (t == 0 && t0 + i + kBulkStages < t1) {
      tc::bulk_wait_read_all();                         // stage s is read out
      fill(i + kBulkStages);
    }
  }
  if (t == 0) {
    tc::bulk_wait_all();
    // after an abort, let loads still in flight land before the CTA exits
    for (int s = 0; s < kBulkStages; ++s)
      if (issued[s] > 0) tc::mbar_wait(&full[s], (issued[s] - 1) & 1);
  }
  // completing implies the previous kernel completed, for the kernels after
  if (!a.wait_first) pdl_wait();
}

template <typename T, int D, bool PAGED>
cudaError_t launch_bulk_t(const BulkArgs& a, int free_sms, cudaStream_t s) {
  if (a.total_tiles == 0) return cudaSuccess;
  auto k = stitch_bulk_kernel<T, D, PAGED>;
  cudaError_t e = set_dyn_smem_once(reinterpret_cast<const void*>(k), kBulkSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // two CTAs per SM of the device, each through a short contiguous range of
  // tiles: beside a kernel that holds most SMs (free_sms >= 0), the CTAs past
  // the free SMs start as that kernel's CTAs finish and end soon after
  (void)free_sms;
  const int ctas = 2 * std::max(sms, 1);
  const int grid = std::min(a.total_tiles, ctas);
  return launch_pdl(k, dim3(grid), dim3(kBulkThreads), kBulkSmem, s, a);
}

template <typename TS, typename TO, int D, bool PAGED>
cudaError_t launch_t(const StitchArgs& a, int n_chunks, cudaStream_t s) {
  const int grid = n_chunks * a.tiles_per_chunk;
  if (grid == 0) return cudaSuccess;
  return launch_pdl(stitch_kernel<TS, TO, D, PAGED>, dim3(grid), dim3(kStitchThreads), 0, s, a);
}

template <typename TS, typename TO>
cudaError_t launch_d(const StitchArgs& a, int n_chunks, int D, bool paged, cudaStream_t s) {
  if (D == 128)
    return paged ? launch_t<TS, TO, 128, true>(a, n_chunks, s)
                 : launch_t<TS, TO, 128, false>(a, n_chunks, s);
  return paged ? launch_t<TS, TO, 64, true>(a, n_chunks, s)
               : launch_t<TS, TO, 64, false>(a, n_chunks, s);
}

}  // namespace

bool stitch_streamed(const fuse_layer_desc_t& desc, const fuse_chunks_t& chunks) {
  const int64_t row_bytes =
      (int64_t)desc.n_kv_heads * desc.head_dim * (desc.dtype == FUSE_F32 ? 4 : 2);
  return chunks.kv_storage == desc.dtype && row_bytes <= kBulkTileBytes;
}

cudaError_t launch_stitch(const fuse_layer_desc_t& desc, const fuse_chunks_t& chunks,
                          const RopeFreqs& freqs, int max_len, void* Kf, void* Vf, uint32_t* err,
                          cudaStream_t s, int free_sms) {
  const bool paged = chunks.kv_layout == FUSE_KV_PAGED;
  const int D = desc.head_dim;
  const bool same = chunks.kv_storage == desc.dtype;   // F32 / BF16 codes are the dtypes
  const int64_t row_bytes = (int64_t)desc.n_kv_heads * D * (desc.dtype == FUSE_F32 ? 4 : 2);
  if (same && row_bytes <= kBulkTileBytes) {
    BulkArgs b;
    b.chunks = chunks.d_chunks;
    b.Kf = Kf;
    b.Vf = Vf;
    b.err = err;
    b.n_pool_blocks = chunks.n_pool_blocks;
    b.n_kv_heads = desc.n_kv_heads;
    b.block_size = chunks.block_size > 0 ? chunks.block_size : 1;
    int rt = (int)(kBulkTileBytes / row_bytes);
    if (paged)
      while (b.block_size % rt != 0) --rt;     // a tile never leaves its page
    b.rt = rt;
    b.tiles_per_chunk = (max_len + rt - 1) / rt;
    b.total_tiles = chunks.n_chunks * b.tiles_per_chunk;
    b.wait_first = free_sms < 0;
    b.freqs = freqs;
    if (desc.dtype == FUSE_BF16)
      return D == 128 ? (paged ? launch_bulk_t<__nv_bfloat16, 128, true>(b, free_sms, s)
                               : launch_bulk_t<__nv_bfloat16, 128, false>(b, free_sms, s))
                      : (paged ? launch_bulk_t<__nv_bfloat16, 64, true>(b, free_sms, s)
                               : launch_bulk_t<__nv_bfloat16, 64, false>(b, free_sms, s));
    return D == 128 ? (paged ? launch_bulk_t<float, 128, true>(b, free_sms, s)
                             : launch_bulk_t<float, 128, false>(b, free_sms, s))
                    : (paged ? launch_bulk_t<float, 64, true>(b, free_sms, s)
                             : launch_bulk_t<float, 64, false>(b, free_sms, s));
  }
  StitchArgs a;
  a.chunks = chunks.d_chunks;
  a.Kf = Kf;
  a.Vf = Vf;
  a.err = err;
  a.n_pool_blocks = chunks.n_pool_blocks;
  a.n_kv_heads = desc.n_kv_heads;
  a.block_size = chunks.block_size > 0 ? chunks.block_size : 1;
  a.freqs = freqs;
  a.wait_first = free_sms < 0;
  if (chunks.kv_storage == FUSE_U8_ASYM && desc.n_kv_heads * D <= kU8MaxRowElems) {
    // one key item (16 pairs) per thread: rows_per_cta * Hkv * d / 32 = 128
    int rows = std::max(1, kU8Threads * 32 / (desc.n_kv_heads * D));
    if (paged)
      while (a.block_size % rows != 0) --rows;   // a tile never leaves its page
    a.rows_per_cta = rows;
    a.tiles_per_chunk = (max_len + rows - 1) / rows;
    const int n_tiles = chunks.n_chunks * a.tiles_per_chunk;
    if (n_tiles == 0) return cudaSuccess;
    const int grid = n_tiles;                  // one CTA per tile
    const bool bf = desc.dtype == FUSE_BF16;
#define FUSEKV_U8(TO, DD, PG) \
    return launch_pdl(stitch_u8_kernel<TO, DD, PG>, dim3(grid), dim3(kU8Threads), 0, s, a, n_tiles)
    if (D == 128) {
      if (bf) { if (paged) FUSEKV_U8(__nv_bfloat16, 128, true); FUSEKV_U8(__nv_bfloat16, 128, false); }
      if (paged) FUSEKV_U8(float, 128, true);
      FUSEKV_U8(float, 128, false);
    }
    if (bf) { if (paged) FUSEKV_U8(__nv_bfloat16, 64, true); FUSEKV_U8(__nv_bfloat16, 64, false); }
    if (paged) FUSEKV_U8(float, 64, true);
    FUSEKV_U8(float, 64, false);
#undef FUSEKV_U8
  }
  // rows per CTA: every thread gets at most kStitchItems V groups (D/8 per
  // head-row) and, as K groups are half as many, at most that many K groups
  a.rows_per_cta = std::max(1, (kStitchThreads * kStitchItems) / (desc.n_kv_heads * (desc.head_dim / 8)));
  a.tiles_per_chunk = (max_len + a.rows_per_cta - 1) / a.rows_per_cta;
  a.freqs = freqs;
  const bool out_bf16 = desc.dtype == FUSE_BF16;
  switch (chunks.kv_storage) {
    case FUSE_F32:
      return out_bf16 ? launch_d<float, __nv_bfloat16>(a, chunks.n_chunks, D, paged, s)
                      : launch_d<float, float>(a, chunks.n_chunks, D, paged, s);
    case FUSE_BF16:
      return out_bf16 ? launch_d<__nv_bfloat16, __nv_bfloat16>(a, chunks.n_chunks, D, paged, s)
                      : launch_d<__nv_bfloat16, float>(a, chunks.n_chunks, D, paged, s);
    case FUSE_U4_ASYM:
      return out_bf16 ? launch_d<Nibbles, __nv_bfloat16>(a, chunks.n_chunks, D, paged, s)
                      : launch_d<Nibbles, float>(a, chunks.n_chunks, D, paged, s);
    default:
      return out_bf16 ? launch_d<uint8_t, __nv_bfloat16>(a, chunks.n_chunks, D, paged, s)
                      : launch_d<uint8_t, float>(a, chunks.n_chunks, D, paged, s);
  }
}

}  // namespace fusekv
