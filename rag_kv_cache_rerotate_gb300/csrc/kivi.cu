// KIVI asymmetric quantisation of chunk caches (KVBoost section 4.5, Eq. 7,
// with b = 8 or 4): input preparation for the int8 / int4 storage modes, not
// part of a layer-step.
//
// For b-bit codes with L = 2^b - 1 levels, a group of values x with minimum
// mn and maximum mx is stored as
//   q = rint((x - mn) / (mx - mn) * L),  scale = (mx - mn) / L,  zero = mn,
// scale and zero rounded to fp16; a constant group (mx == mn) gets q = 0 and
// scale 0.  Keys are grouped per (chunk, head, channel) over the chunk's
// tokens, values per (token, head) over the head dimension.  The codes are
// formed in fp64 (round to nearest even), so a code is the same on any
// machine that follows IEEE 754 for the one division and one multiplication.
#include "common.cuh"
#include "launch.h"

namespace fusekv {

namespace {

struct KiviArgs {
  const fuse_chunk_t* src;   // layer-type caches, CONTIGUOUS [len, Hkv, d]
  const fuse_chunk_t* dst;   // codes and fp16 scale / zero, CONTIGUOUS
  int32_t n_kv_heads;
  int32_t levels;            // 255 or 15
};

template <typename T> __device__ __forceinline__ double load_elem(const void* p, int64_t e) {
  if constexpr (sizeof(T) == 4)
    return (double)__ldg(reinterpret_cast<const float*>(p) + e);
  else
    return (double)__bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[e]);
}

__device__ __forceinline__ uint32_t kivi_code(double x, double mn, double span, double levels) {
  return span > 0.0 ? (uint32_t)rint((x - mn) / span * levels) : 0u;
}

// One CTA per (chunk, head), thread j = channel: the key statistics run over
// the chunk's tokens.  Codes of channels 2m, 2m + 1 share byte m for b = 4.
template <typename T, int D>
__global__ void __launch_bounds__(D) kivi_key_kernel(const KiviArgs a) {
  const fuse_chunk_t s = a.src[blockIdx.x];
  const fuse_chunk_t o = a.dst[blockIdx.x];
  const int h = blockIdx.y, j = threadIdx.x, Hkv = a.n_kv_heads;
  double mn = 0.0, mx = 0.0;
  for (int r = 0; r < s.len; ++r) {
    const double x = load_elem<T>(s.k, ((int64_t)r * Hkv + h) * D + j);
    mn = r == 0 ? x : fmin(mn, x);
    mx = r == 0 ? x : fmax(mx, x);
  }
  if (s.len == 0) return;
  const double span = mx - mn, L = (double)a.levels;
  reinterpret_cast<__half*>(const_cast<void*>(o.k_scale))[h * D + j] = __double2half(span / L);
  reinterpret_cast<__half*>(const_cast<void*>(o.k_zero))[h * D + j] = __double2half(mn);
  uint8_t* q = reinterpret_cast<uint8_t*>(const_cast<void*>(o.k));
  for (int r = 0; r < s.len; ++r) {
    const uint32_t c = kivi_code(load_elem<T>(s.k, ((int64_t)r * Hkv + h) * D + j), mn, span, L);
    const int64_t e = ((int64_t)r * Hkv + h) * D + j;
    if (a.levels == 255) {
      q[e] = (uint8_t)c;
    } else {
      const uint32_t hi = __shfl_down_sync(0xffffffffu, c, 1);   // channel j + 1
      if ((j & 1) == 0) q[e / 2] = (uint8_t)(c | (hi << 4));
    }
  }
}

// One warp per (token, head) of one chunk: the value statistics run over d.
template <typename T, int D>
__global__ void __launch_bounds__(256) kivi_value_kernel(const KiviArgs a, int max_len) {
  constexpr int E = D / 32;                     // elements per lane (consecutive)
  const int chunk = blockIdx.y;
  const fuse_chunk_t s = a.src[chunk];
  const fuse_chunk_t o = a.dst[chunk];
  const int Hkv = a.n_kv_heads;
  const int64_t w = (int64_t)blockIdx.x * 8 + threadIdx.x / 32;   // token * Hkv + head
  const int lane = threadIdx.x % 32;
  if (w >= (int64_t)s.len * Hkv) return;
  (void)max_len;
  double x[E];
  double mn, mx;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    x[i] = load_elem<T>(s.v, w * D + lane * E + i);
    mn = i == 0 ? x[i] : fmin(mn, x[i]);
    mx = i == 0 ? x[i] : fmax(mx, x[i]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mn = fmin(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  const double span = mx - mn, L = (double)a.levels;
  if (lane == 0) {
    reinterpret_cast<__half*>(const_cast<void*>(o.v_scale))[w] = __double2half(span / L);
    reinterpret_cast<__half*>(const_cast<void*>(o.v_zero))[w] = __double2half(mn);
  }
  uint8_t* q = reinterpret_cast<uint8_t*>(const_cast<void*>(o.v));
  if (a.levels == 255) {
#pragma unroll
    for (int i = 0; i < E; ++i) q[w * D + lane * E + i] = (uint8_t)kivi_code(x[i], mn, span, L);
  } else {
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const uint32_t lo = kivi_code(x[i], mn, span, L), hi = kivi_code(x[i + 1], mn, span, L);
      q[(w * D + lane * E + i) / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

template <typename T, int D>
cudaError_t launch_kivi_t(const KiviArgs& a, int n_chunks, int max_len, cudaStream_t s) {
  kivi_key_kernel<T, D><<<dim3(n_chunks, a.n_kv_heads), D, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t warps = (int64_t)max_len * a.n_kv_heads;
  const int gx = (int)((warps + 7) / 8);
  kivi_value_kernel<T, D><<<dim3(gx, n_chunks), 256, 0, s>>>(a, max_len);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kivi_quantize(const fuse_layer_desc_t& d, const fuse_chunks_t& src,
                                 const fuse_chunks_t& dst, int max_len, cudaStream_t s) {
  KiviArgs a;
  a.src = src.d_chunks;
  a.dst = dst.d_chunks;
  a.n_kv_heads = d.n_kv_heads;
  a.levels = dst.kv_storage == FUSE_U4_ASYM ? 15 : 255;
  if (src.n_chunks == 0 || max_len == 0) return cudaSuccess;
  if (d.dtype == FUSE_BF16)
    return d.head_dim == 128 ? launch_kivi_t<__nv_bfloat16, 128>(a, src.n_chunks, max_len, s)
                             : launch_kivi_t<__nv_bfloat16, 64>(a, src.n_chunks, max_len, s);
  return d.head_dim == 128 ? launch_kivi_t<float, 128>(a, src.n_chunks, max_len, s)
                           : launch_kivi_t<float, 64>(a, src.n_chunks, max_len, s);
}

}  // namespace fusekv
