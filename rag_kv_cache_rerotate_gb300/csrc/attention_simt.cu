// Causal GQA attention of the recomputed rows over the fused cache, on CUDA
// cores: the fp32 path, and the fallback for shapes the tensor-core kernel
// does not take.
//
// QCFuse (section 2.1.3, Eq. 6): a selected token at position p reads every
// prefix position j <= p of the partially fused cache.  KVBoost (section
// 3.1, Eq. 2): softmax(q K^T / sqrt(d)) V over j <= p.  One warp serves one
// (row, KV head) and all g = Hq/Hkv query heads that share it; the softmax is
// online (running max and sum), in base 2.
#include "common.cuh"
#include "launch.h"

namespace fusekv {

namespace {

struct AttnArgs {
  const WorkRow* rows;
  const void* Q;
  const void* Kf;
  const void* Vf;
  void* O;
  int64_t n_rows;
  int n_q_heads;
  int n_kv_heads;
  float qscale;   // log2(e) / sqrt(d)
};

template <typename T, int EL> struct LdEl;
template <> struct LdEl<float, 4> {
  static __device__ __forceinline__ void load(const float* p, float (&x)[4]) {
    float4 v = __ldg(reinterpret_cast<const float4*>(p));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&x)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
};
template <> struct LdEl<float, 2> {
  static __device__ __forceinline__ void load(const float* p, float (&x)[2]) {
    float2 v = __ldg(reinterpret_cast<const float2*>(p));
    x[0] = v.x; x[1] = v.y;
  }
  static __device__ __forceinline__ void store(float* p, const float (&x)[2]) {
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
  }
};
template <> struct LdEl<__nv_bfloat16, 4> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[4]) {
    uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&x)[4]) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
  }
};
template <> struct LdEl<__nv_bfloat16, 2> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[2]) {
    uint32_t v = __ldg(reinterpret_cast<const unsigned int*>(p));
    x[0] = bf16_lo(v); x[1] = bf16_hi(v);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&x)[2]) {
    *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(x[0], x[1]);
  }
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(128) attn_simt_kernel(const AttnArgs a) {
  constexpr int EL = D / 32;
  const int lane = threadIdx.x % 32;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int Hkv = a.n_kv_heads;
  const int Hq = a.n_q_heads;
  if (gw >= a.n_rows * Hkv) return;
  const int64_t m = gw / Hkv;
  const int kvh = (int)(gw % Hkv);
  const WorkRow w = a.rows[m];
  const int64_t row0 = w.dst_row - w.pos;
  const int p = w.pos;
  const T* Q = reinterpret_cast<const T*>(a.Q);
  const T* Kf = reinterpret_cast<const T*>(a.Kf);
  const T* Vf = reinterpret_cast<const T*>(a.Vf);

  float q[G][EL], acc[G][EL], mx[G], l[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    LdEl<T, EL>::load(Q + (m * Hq + kvh * G + h) * D + lane * EL, q[h]);
#pragma unroll
    for (int e = 0; e < EL; ++e) {
      q[h][e] *= a.qscale;
      acc[h][e] = 0.f;
    }
    mx[h] = -INFINITY;
    l[h] = 0.f;
  }
  for (int j = 0; j <= p; ++j) {
    const int64_t base = ((row0 + j) * Hkv + kvh) * D + lane * EL;
    float k[EL], v[EL];
    LdEl<T, EL>::load(Kf + base, k);
    LdEl<T, EL>::load(Vf + base, v);
    float sc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < EL; ++e) s = fmaf(q[h][e], k[e], s);
      sc[h] = s;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int h = 0; h < G; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], o);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mn = fmaxf(mx[h], sc[h]);
      const float corr = exp2f(mx[h] - mn);
      const float pe = exp2f(sc[h] - mn);
      l[h] = fmaf(l[h], corr, pe);
#pragma unroll
      for (int e = 0; e < EL; ++e) acc[h][e] = fmaf(acc[h][e], corr, pe * v[e]);
      mx[h] = mn;
    }
  }
  T* O = reinterpret_cast<T*>(a.O);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float inv = 1.0f / l[h];
    float o[EL];
#pragma unroll
    for (int e = 0; e < EL; ++e) o[e] = acc[h][e] * inv;
    LdEl<T, EL>::store(O + (m * Hq + kvh * G + h) * D + lane * EL, o);
  }
}

template <typename T, int D>
cudaError_t run_g(const AttnArgs& a, int g, cudaStream_t s) {
  const int64_t threads = a.n_rows * a.n_kv_heads * 32;
  const unsigned grid = (unsigned)((threads + 127) / 128);
  switch (g) {
    case 1: attn_simt_kernel<T, D, 1><<<grid, 128, 0, s>>>(a); break;
    case 2: attn_simt_kernel<T, D, 2><<<grid, 128, 0, s>>>(a); break;
    case 4: attn_simt_kernel<T, D, 4><<<grid, 128, 0, s>>>(a); break;
    case 8: attn_simt_kernel<T, D, 8><<<grid, 128, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_simt(const fuse_layer_desc_t& desc, int64_t n_rows, const WorkRow* rows,
                                  const void* Q, const void* Kf, const void* Vf, void* O,
                                  cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  AttnArgs a;
  a.rows = rows;
  a.Q = Q;
  a.Kf = Kf;
  a.Vf = Vf;
  a.O = O;
  a.n_rows = n_rows;
  a.n_q_heads = desc.n_q_heads;
  a.n_kv_heads = desc.n_kv_heads;
  a.qscale = 1.4426950408889634f / sqrtf((float)desc.head_dim);
  const int g = desc.n_q_heads / desc.n_kv_heads;
  if (desc.dtype == FUSE_BF16)
    return desc.head_dim == 128 ? run_g<__nv_bfloat16, 128>(a, g, s) : run_g<__nv_bfloat16, 64>(a, g, s);
  return desc.head_dim == 128 ? run_g<float, 128>(a, g, s) : run_g<float, 64>(a, g, s);
}

}  // namespace fusekv
