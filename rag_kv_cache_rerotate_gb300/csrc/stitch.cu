// Stitch + RoPE re-rotation (+ KIVI int8 dequantisation, + paged gather).
//
// QCFuse (section 2.1.2, Eq. 4): chunk caches built alone at local positions
// are placed at their request positions; keys are remapped by the chunk's
// position offset o_i, values are copied in token order.  KVBoost (section
// 3.2): a key cached with R^r and reused at o_i + r needs the correction
// R^{o_i}.  KVBoost (section 4.5, Eq. 7): x = zero + q * scale, keys with
// per-channel statistics, values with per-token statistics.
//
// Memory-bound.  One CTA moves a few rows of one chunk; each thread owns one
// group of 8 key pairs and two groups of 8 values and issues all its 16-byte
// loads before anything else, so every thread keeps four loads in flight at
// low register use.  The chunk offset's (cos, sin) of the d/2 frequencies are
// computed once per CTA into shared memory while those loads are in flight.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

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
  constexpr bool kU8 = sizeof(TS) == 1;
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
        if constexpr (kU8) {
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
        if constexpr (kU8)
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

cudaError_t launch_stitch(const fuse_layer_desc_t& desc, const fuse_chunks_t& chunks,
                          const RopeFreqs& freqs, int max_len, void* Kf, void* Vf, uint32_t* err,
                          cudaStream_t s) {
  StitchArgs a;
  a.chunks = chunks.d_chunks;
  a.Kf = Kf;
  a.Vf = Vf;
  a.err = err;
  a.n_pool_blocks = chunks.n_pool_blocks;
  a.n_kv_heads = desc.n_kv_heads;
  a.block_size = chunks.block_size > 0 ? chunks.block_size : 1;
  // rows per CTA: every thread gets at most kStitchItems V groups (D/8 per
  // head-row) and, as K groups are half as many, at most that many K groups
  a.rows_per_cta = std::max(1, (kStitchThreads * kStitchItems) / (desc.n_kv_heads * (desc.head_dim / 8)));
  a.tiles_per_chunk = (max_len + a.rows_per_cta - 1) / a.rows_per_cta;
  a.freqs = freqs;
  const bool paged = chunks.kv_layout == FUSE_KV_PAGED;
  const int D = desc.head_dim;
  const bool out_bf16 = desc.dtype == FUSE_BF16;
  switch (chunks.kv_storage) {
    case FUSE_F32:
      return out_bf16 ? launch_d<float, __nv_bfloat16>(a, chunks.n_chunks, D, paged, s)
                      : launch_d<float, float>(a, chunks.n_chunks, D, paged, s);
    case FUSE_BF16:
      return out_bf16 ? launch_d<__nv_bfloat16, __nv_bfloat16>(a, chunks.n_chunks, D, paged, s)
                      : launch_d<__nv_bfloat16, float>(a, chunks.n_chunks, D, paged, s);
    default:
      return out_bf16 ? launch_d<uint8_t, __nv_bfloat16>(a, chunks.n_chunks, D, paged, s)
                      : launch_d<uint8_t, float>(a, chunks.n_chunks, D, paged, s);
  }
}

}  // namespace fusekv
