// CUDA-core (SIMT) projection GEMMs with fused epilogues: the fp32 path of
// the library, and the fallback for shapes the tensor-core kernel does not
// take.  C[m, n] = sum_k A[a_row(m), k] * W[n, k] with fp32 accumulation,
// one output tile spanning exactly one head (BN = head_dim), so that every
// epilogue sees whole heads:
//
//  * deviation (KVBoost Alg. 2 step 2, on V): per (token, KV head) cosine
//    between the fresh V tile and the cached V row -> partial[slot, h];
//  * recompute (QCFuse Eqs. 6-7; KVBoost Eqs. 1-3): RoPE at each row's
//    request position for Q and K heads, Q to a compact buffer, K and V
//    scattered into the fused cache at the row's position;
//  * PIC precompute (QCFuse Eq. 3): K (RoPE at the chunk-local position) and
//    V written into the chunk caches.
#include "common.cuh"
#include "launch.h"

namespace fusekv {

namespace {

constexpr int kBM = 64;
constexpr int kBK = 16;
constexpr int kThreads = 256;

enum EpiMode : int { EPI_DEVIATION = 0, EPI_RECOMPUTE = 1, EPI_PIC = 2 };

struct GemmArgs {
  int64_t M;                 // rows
  int K;                     // hidden
  const void* A;             // [*, K]
  const WorkRow* rows;       // nullable: identity rows
  const void* W0;            // weight blocks stacked along n, each [n_i, K]
  const void* W1;
  const void* W2;
  int n0, n1;                // column counts of W0, W1 (W2 takes the rest)
  int n_q_heads, n_kv_heads;
  int mode;
  // deviation
  const void* Vf;
  const int32_t* map;
  float* partial;
  // recompute / pic
  const float2* rope;
  void* Q;
  void* Kf;
  void* Vf_out;
  const fuse_chunk_t* chunks;
  int pic_max_len;           // PIC: GEMM row m is token m % max_len of chunk m / max_len
  uint32_t* err;
  RopeFreqs freqs;           // PIC: RoPE at the chunk-local position
};

template <typename T> struct Ld4;
template <> struct Ld4<float> {
  static __device__ __forceinline__ float4 load(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
  }
};
template <> struct Ld4<__nv_bfloat16> {
  static __device__ __forceinline__ float4 load(const __nv_bfloat16* p) {
    uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    return make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
  }
};

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

template <typename T, int BN>
__global__ void __launch_bounds__(kThreads) gemm_simt_kernel(const GemmArgs a) {
  constexpr int TN = BN / 16;
  constexpr int H2 = BN / 2;
  constexpr int kAS = kBK * (kBM + 4);
  constexpr int kBS = kBK * (BN + 4);
  constexpr int kCS = kBM * (BN + 1);
  constexpr int kSmem = (kAS + kBS) > kCS ? (kAS + kBS) : kCS;
  __shared__ __align__(16) float smem[kSmem];
  float* As = smem;
  float* Bs = smem + kAS;

  const int t = threadIdx.x;
  const int tx = t % 16;
  const int ty = t / 16;
  const int64_t m0 = (int64_t)blockIdx.y * kBM;
  const int n0 = blockIdx.x * BN;
  const T* A = reinterpret_cast<const T*>(a.A);

  // weight block and its first row for this column tile
  const T* W;
  int wn0;
  if (n0 < a.n0) {
    W = reinterpret_cast<const T*>(a.W0);
    wn0 = n0;
  } else if (n0 < a.n0 + a.n1) {
    W = reinterpret_cast<const T*>(a.W1);
    wn0 = n0 - a.n0;
  } else {
    W = reinterpret_cast<const T*>(a.W2);
    wn0 = n0 - a.n0 - a.n1;
  }

  // A row of this thread's loads
  const int arow = t >> 2;
  const int kq = (t & 3) * 4;
  int64_t src_row = -1;
  {
    const int64_t m = m0 + arow;
    if (m < a.M) {
      if (a.mode == EPI_PIC) {
        const fuse_chunk_t& c = a.chunks[m / a.pic_max_len];
        const int r = (int)(m % a.pic_max_len);
        src_row = r < c.len ? c.dst_row + r : -1;
      } else {
        src_row = a.rows ? a.rows[m].a_row : m;
      }
    }
  }

  float acc[4][TN];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < TN; ++c) acc[i][c] = 0.f;

  for (int k0 = 0; k0 < a.K; k0 += kBK) {
    float4 av = make_float4(0.f, 0.f, 0.f, 0.f);
    if (src_row >= 0) av = Ld4<T>::load(A + src_row * a.K + k0 + kq);
    As[(kq + 0) * (kBM + 4) + arow] = av.x;
    As[(kq + 1) * (kBM + 4) + arow] = av.y;
    As[(kq + 2) * (kBM + 4) + arow] = av.z;
    As[(kq + 3) * (kBM + 4) + arow] = av.w;
#pragma unroll
    for (int rr = arow; rr < BN; rr += kThreads / 4) {
      const float4 bv = Ld4<T>::load(W + (int64_t)(wn0 + rr) * a.K + k0 + kq);
      Bs[(kq + 0) * (BN + 4) + rr] = bv.x;
      Bs[(kq + 1) * (BN + 4) + rr] = bv.y;
      Bs[(kq + 2) * (BN + 4) + rr] = bv.z;
      Bs[(kq + 3) * (BN + 4) + rr] = bv.w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      const float4 av4 = *reinterpret_cast<const float4*>(&As[kk * (kBM + 4) + ty * 4]);
      const float ar[4] = {av4.x, av4.y, av4.z, av4.w};
      float br[TN];
#pragma unroll
      for (int c = 0; c < TN; ++c) br[c] = Bs[kk * (BN + 4) + tx + 16 * c];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < TN; ++c) acc[i][c] = fmaf(ar[i], br[c], acc[i][c]);
    }
    __syncthreads();
  }

  // stage the tile
  float* Cs = smem;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < TN; ++c) Cs[(ty * 4 + i) * (BN + 1) + tx + 16 * c] = acc[i][c];
  __syncthreads();

  const int Hq = a.n_q_heads;
  const int Hkv = a.n_kv_heads;
  const int head = n0 / BN;
  if (a.mode == EPI_DEVIATION) {
    const int warp = t / 32;
    const int lane = t % 32;
    const T* Vf = reinterpret_cast<const T*>(a.Vf);
    for (int i = warp; i < kBM; i += kThreads / 32) {
      const int64_t m = m0 + i;
      if (m >= a.M) break;
      const int32_t slot = a.map[m];
      if (slot < 0) continue;
      float dot = 0.f, na = 0.f, nb = 0.f;
      const T* vrow = Vf + (m * Hkv + head) * BN;
      for (int c = lane; c < BN; c += 32) {
        const float v = Cs[i * (BN + 1) + c];
        const float f = to_f<T>(vrow[c]);
        dot = fmaf(v, f, dot);
        na = fmaf(v, v, na);
        nb = fmaf(f, f, nb);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        dot += __shfl_xor_sync(0xffffffffu, dot, o);
        na += __shfl_xor_sync(0xffffffffu, na, o);
        nb += __shfl_xor_sync(0xffffffffu, nb, o);
      }
      if (lane == 0) a.partial[(int64_t)slot * Hkv + head] = dot / fmaxf(sqrtf(na) * sqrtf(nb), 1e-30f);
    }
    return;
  }

  // recompute / PIC: (row, pair) items
  for (int it = t; it < kBM * H2; it += kThreads) {
    const int i = it / H2;
    const int j = it % H2;
    const int64_t m = m0 + i;
    if (m >= a.M) break;
    float x = Cs[i * (BN + 1) + j];
    float y = Cs[i * (BN + 1) + j + H2];
    T* dst;
    bool rot;
    if (a.mode == EPI_RECOMPUTE) {
      const WorkRow w = a.rows[m];
      if (head < Hq) {
        dst = reinterpret_cast<T*>(a.Q) + (m * Hq + head) * BN;
        rot = true;
      } else if (head < Hq + Hkv) {
        dst = reinterpret_cast<T*>(a.Kf) + (w.dst_row * Hkv + (head - Hq)) * BN;
        rot = true;
      } else {
        dst = reinterpret_cast<T*>(a.Vf_out) + (w.dst_row * Hkv + (head - Hq - Hkv)) * BN;
        rot = false;
      }
      if (rot) {
        const float2 cs = a.rope[rope_index(j, m, a.M)];
        const float xr = fmaf(x, cs.x, -y * cs.y);
        const float yr = fmaf(y, cs.x, x * cs.y);
        x = xr;
        y = yr;
      }
    } else {
      const fuse_chunk_t& c = a.chunks[m / a.pic_max_len];
      const int r = (int)(m % a.pic_max_len);
      if (r >= c.len) continue;
      if (head < Hkv) {
        dst = const_cast<T*>(reinterpret_cast<const T*>(c.k)) + ((int64_t)r * Hkv + head) * BN;
        float cs, sn;
        rope_cos_sin(r, a.freqs.hi[j], a.freqs.mid[j], a.freqs.lo[j], cs, sn);
        const float xr = fmaf(x, cs, -y * sn);
        const float yr = fmaf(y, cs, x * sn);
        x = xr;
        y = yr;
      } else {
        dst = const_cast<T*>(reinterpret_cast<const T*>(c.v)) + ((int64_t)r * Hkv + (head - Hkv)) * BN;
      }
    }
    dst[j] = from_f<T>(x);
    dst[j + H2] = from_f<T>(y);
  }
}

template <typename T>
cudaError_t run(const GemmArgs& a, int n_total, int head_dim, cudaStream_t s) {
  if (a.M == 0) return cudaSuccess;
  dim3 grid(n_total / head_dim, (unsigned)((a.M + kBM - 1) / kBM));
  if (head_dim == 128)
    gemm_simt_kernel<T, 128><<<grid, kThreads, 0, s>>>(a);
  else
    gemm_simt_kernel<T, 64><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t dispatch(const fuse_layer_desc_t& desc, const GemmArgs& a, int n_total, cudaStream_t s) {
  if (desc.dtype == FUSE_BF16) return run<__nv_bfloat16>(a, n_total, desc.head_dim, s);
  return run<float>(a, n_total, desc.head_dim, s);
}

__global__ void deviation_reduce_kernel(int64_t n, int n_parts, int Hkv, const float* partial,
                                        float* score) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  score[i] = head_mean_score(partial + i * n_parts, n_parts, Hkv);
}

}  // namespace

cudaError_t launch_deviation_partials_simt(const fuse_layer_desc_t& desc, int64_t n_rows,
                                           const void* H, const void* Wv, const void* Vf,
                                           const int32_t* map, float* partial, uint32_t* err,
                                           cudaStream_t s) {
  GemmArgs a = {};
  a.M = n_rows;
  a.K = desc.hidden;
  a.A = H;
  a.W0 = Wv;
  a.n0 = desc.n_kv_heads * desc.head_dim;
  a.n1 = 0;
  a.n_q_heads = desc.n_q_heads;
  a.n_kv_heads = desc.n_kv_heads;
  a.mode = EPI_DEVIATION;
  a.Vf = Vf;
  a.map = map;
  a.partial = partial;
  a.err = err;
  return dispatch(desc, a, a.n0, s);
}

cudaError_t launch_deviation_reduce(int64_t n_ctx, int n_parts, int n_kv_heads,
                                    const float* partial, float* score, cudaStream_t s) {
  if (n_ctx == 0) return cudaSuccess;
  deviation_reduce_kernel<<<(unsigned)((n_ctx + 255) / 256), 256, 0, s>>>(n_ctx, n_parts,
                                                                          n_kv_heads, partial,
                                                                          score);
  return cudaGetLastError();
}

cudaError_t launch_project_recompute_simt(const fuse_layer_desc_t& desc, int64_t n_rows,
                                          const WorkRow* rows, const float2* rope, const void* H,
                                          const void* Wq, const void* Wk, const void* Wv, void* Q,
                                          void* Kf, void* Vf, uint32_t* err, cudaStream_t s) {
  GemmArgs a = {};
  a.M = n_rows;
  a.K = desc.hidden;
  a.A = H;
  a.rows = rows;
  a.W0 = Wq;
  a.W1 = Wk;
  a.W2 = Wv;
  a.n0 = desc.n_q_heads * desc.head_dim;
  a.n1 = desc.n_kv_heads * desc.head_dim;
  a.n_q_heads = desc.n_q_heads;
  a.n_kv_heads = desc.n_kv_heads;
  a.mode = EPI_RECOMPUTE;
  a.rope = rope;
  a.Q = Q;
  a.Kf = Kf;
  a.Vf_out = Vf;
  a.err = err;
  return dispatch(desc, a, a.n0 + 2 * a.n1, s);
}

cudaError_t launch_project_query_simt(const fuse_layer_desc_t& desc, int64_t n_rows,
                                      const WorkRow* rows, const float2* rope, const void* H,
                                      const void* Wq, void* Q, uint32_t* err, cudaStream_t s) {
  GemmArgs a = {};
  a.M = n_rows;
  a.K = desc.hidden;
  a.A = H;
  a.rows = rows;
  a.W0 = Wq;
  a.W1 = Wq;
  a.W2 = Wq;
  a.n0 = desc.n_q_heads * desc.head_dim;
  a.n1 = 0;
  a.n_q_heads = desc.n_q_heads;
  a.n_kv_heads = desc.n_kv_heads;
  a.mode = EPI_RECOMPUTE;
  a.rope = rope;
  a.Q = Q;
  a.err = err;
  return dispatch(desc, a, a.n0, s);     // Q heads only: no K/V columns, no scatter
}

cudaError_t launch_project_pic(const fuse_layer_desc_t& desc, int n_chunks, int max_len,
                               const RopeFreqs& freqs, const void* H, const void* Wk, const void* Wv,
                               const fuse_chunk_t* d_chunks, uint32_t* err, cudaStream_t s) {
  GemmArgs a = {};
  a.M = (int64_t)n_chunks * max_len;
  a.K = desc.hidden;
  a.A = H;
  a.pic_max_len = max_len > 0 ? max_len : 1;
  a.freqs = freqs;
  a.W0 = Wk;
  a.W1 = Wv;
  a.n0 = desc.n_kv_heads * desc.head_dim;
  a.n1 = desc.n_kv_heads * desc.head_dim;
  a.n_q_heads = desc.n_q_heads;
  a.n_kv_heads = desc.n_kv_heads;
  a.mode = EPI_PIC;
  a.chunks = d_chunks;
  a.err = err;
  return dispatch(desc, a, a.n0 + a.n1, s);
}

}  // namespace fusekv
