// Top-k selection per request: TopK(score, k) of QCFuse (Eq. 11) and step 3
// of KVBoost's CacheBlendRecompute (Alg. 2).
//
// Scores become order-preserving 32-bit keys (-0 folded onto +0, NaN below
// every number and reported).  A block-wide radix select finds the k-th
// largest key tau in four 8-bit rounds; then one pass in index order keeps
// every key above tau and the lowest-indexed keys equal to tau, so ties go
// to the lower index and the output is already ascending.  Exact integer
// work: the result is unique given the score array.
#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace fusekv {

namespace {

constexpr int kTopkThreads = 1024;
constexpr int kTopkSmemKeys = 40 * 1024;   // keys kept in shared memory (160 KB)
constexpr int kTopkBatch = 4;              // tokens per thread whose loads are in flight together
constexpr int kTopkClusterMin = 8192;      // larger requests go to the cluster kernel

__device__ __forceinline__ uint32_t float_key(float f, bool* is_nan) {
  uint32_t b = __float_as_uint(f);
  *is_nan = (b & 0x7FFFFFFFu) > 0x7F800000u;
  if (*is_nan) return 0u;
  if (b == 0x80000000u) b = 0u;                       // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// With partial != null the scores are first formed from the cosine partials
// (n_parts per token), score = 1 - (sum_p partial[p]) / Hkv summed in order
// (the same expression as deviation_reduce_kernel), and written to score[].
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const fuse_request_t* reqs,
                                                            const float* score, int32_t* idx,
                                                            uint32_t* keys_ws, uint32_t* err,
                                                            int keys_in_smem,
                                                            const float* partial = nullptr,
                                                            int n_parts = 0, int n_kv_heads = 0,
                                                            float* score_out = nullptr) {
  extern __shared__ uint32_t dyn[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_buf[32];
  __shared__ uint32_t sel_digit, sel_remaining;
  __shared__ uint2 pair_buf[32];
  __shared__ uint2 sel_scan[32];
  const int r = blockIdx.x;
  const fuse_request_t R = reqs[r];     // the caller's table: no kernel writes it
  pdl_trigger();
  pdl_wait();
  const int n = R.n_ctx;
  const int k = R.k;
  if (n <= 0) return;
  const int t = threadIdx.x;
  if (k <= 0) {                      // nothing to select; still form the scores
    if (partial) {
      for (int i = t; i < n; i += kTopkThreads)
        score_out[R.score0 + i] =
            head_mean_score(partial + (R.score0 + i) * n_parts, n_parts, n_kv_heads);
    }
    return;
  }
  uint32_t* keys = keys_in_smem ? dyn : keys_ws + R.score0;

  bool nan_seen = false;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  // kTopkBatch tokens per thread at a time: their loads are all issued before the
  // first store, so their latencies overlap
  for (int i0 = t; i0 < n; i0 += kTopkBatch * kTopkThreads) {
    float v[kTopkBatch];
    if (partial && n_parts == 4) {                 // one 16-byte load per token
      float4 pv[kTopkBatch];
#pragma unroll
      for (int q = 0; q < kTopkBatch; ++q) {
        const int i = i0 + q * kTopkThreads;
        if (i < n) pv[q] = __ldg(reinterpret_cast<const float4*>(partial) + (R.score0 + i));
      }
#pragma unroll
      for (int q = 0; q < kTopkBatch; ++q)
        if (i0 + q * kTopkThreads < n) v[q] = head_mean_score4(pv[q], n_kv_heads);
    } else {
#pragma unroll
      for (int q = 0; q < kTopkBatch; ++q) {
        const int i = i0 + q * kTopkThreads;
        if (i < n)
          v[q] = partial ? head_mean_score(partial + (R.score0 + i) * n_parts, n_parts, n_kv_heads)
                         : score[R.score0 + i];
      }
    }
#pragma unroll
    for (int q = 0; q < kTopkBatch; ++q) {
      const int i = i0 + q * kTopkThreads;
      if (i < n) {
        if (partial) score_out[R.score0 + i] = v[q];
        bool nn;
        const uint32_t key = float_key(v[q], &nn);
        keys[i] = key;
        kmin = min(kmin, key);
        kmax = max(kmax, key);
        nan_seen |= nn;
      }
    }
  }
  if (nan_seen) report_error(err, FUSE_ERR_DEVICE_BOUNDS, SITE_TOPK_NAN, r);
  // the keys' common leading bits decide nothing: start below them
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if ((t & 31) == 0) {
    warp_buf[t >> 5] = kmin;
    hist[t >> 5] = kmax;
  }
  __syncthreads();
  if (t < 32) {
    constexpr int kWarps = kTopkThreads / 32;
    uint32_t a = t < kWarps ? warp_buf[t] : 0xFFFFFFFFu, b = t < kWarps ? hist[t] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
      b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    if (t == 0) {
      sel_digit = a;
      sel_remaining = b;
    }
  }
  __syncthreads();
  kmin = sel_digit;
  kmax = sel_remaining;
  __syncthreads();
  int lo = 32 - __clz(kmin ^ kmax);      // bits [0, lo) still differ between keys
  uint32_t mask = lo >= 32 ? 0u : ~((1u << lo) - 1u);
  uint32_t prefix = kmin & mask;
  uint32_t remaining = (uint32_t)k;
  // radix rounds of at most 8 bits over the differing bits, highest first
  while (lo > 0) {
    const int w = min(8, lo);
    const int shift = lo - w;
    const uint32_t dmask = (1u << w) - 1u;
    for (int b = t; b < 256; b += kTopkThreads) hist[b] = 0u;
    __syncthreads();
    // Scores crowd into few bins, and same-address shared-memory atomics of a
    // warp serialise: the lanes whose key falls in lane 0's bin add their
    // count with one atomic, the others one each.
    for (int base = t - (t & 31); base < n; base += kTopkThreads) {   // warp-uniform
      const int i = base + (t & 31);
      const uint32_t key = i < n ? keys[i] : 0u;
      const bool act = i < n && (key & mask) == prefix;
      const uint32_t bin = act ? (key >> shift) & dmask : 0xFFFFFFFFu;
      const uint32_t lead = __shfl_sync(0xffffffffu, bin, 0);
      const uint32_t same = __ballot_sync(0xffffffffu, act && bin == lead);
      if ((t & 31) == 0 && same) atomicAdd(&hist[lead], (uint32_t)__popc(same));
      if (act && bin != lead) atomicAdd(&hist[bin], 1u);
    }
    __syncthreads();
    if (t < 32) {
      // warp 0: scan the 256 bins from the top, 8 bins per lane
      uint32_t c[8], lsum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        c[q] = hist[255 - (t * 8 + q)];
        lsum += c[q];
      }
      uint32_t incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (t >= o) incl += y;
      }
      uint32_t cum = incl - lsum;   // count in bins above this lane's first bin
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (cum < remaining && cum + c[q] >= remaining) {
          sel_digit = 255 - (t * 8 + q);
          sel_remaining = remaining - cum;
          warp_buf[0] = c[q];                      // keys in the chosen bin
        }
        cum += c[q];
      }
    }
    __syncthreads();
    prefix |= sel_digit << shift;
    mask |= dmask << shift;
    remaining = sel_remaining;
    const uint32_t in_bin = warp_buf[0];
    lo = shift;
    __syncthreads();
    if (in_bin == remaining) break;      // every key of the chosen bin is taken
  }
  // keys above the prefix are taken; of the keys equal to it under the mask,
  // the lowest-indexed `remaining` ones
  const uint32_t tau = prefix;
  const uint32_t need_eq = remaining;

  // compaction in index order: warp w owns the contiguous range [w0, w1),
  // walked 32 keys at a time (lane l takes key base + l: consecutive lanes
  // read consecutive words, no bank conflicts); ballots give each lane's
  // rank within a step
  const int lane = t & 31, warp = t >> 5;
  constexpr int kWarps = kTopkThreads / 32;
  const int per_w = (((n + kWarps - 1) / kWarps) + 31) & ~31;
  const int w0 = min(n, warp * per_w);
  const int w1 = min(n, w0 + per_w);
  uint32_t n_gt = 0, n_eq = 0;                     // warp-uniform
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w1 ? keys[i] & mask : 0u;
    n_gt += __popc(__ballot_sync(0xffffffffu, i < w1 && key > tau));
    n_eq += __popc(__ballot_sync(0xffffffffu, i < w1 && key == tau));
  }
  // outputs before this warp's range: every key above tau there, and of the
  // keys equal to it the first need_eq in index order (one scan over warps)
  if (lane == 0) pair_buf[warp] = make_uint2(n_gt, n_eq);
  __syncthreads();
  if (warp == 0) {
    uint2 v = lane < kWarps ? pair_buf[lane] : make_uint2(0u, 0u);
    uint32_t ga = v.x, ea = v.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t yg = __shfl_up_sync(0xffffffffu, ga, o);
      const uint32_t ye = __shfl_up_sync(0xffffffffu, ea, o);
      if (lane >= o) {
        ga += yg;
        ea += ye;
      }
    }
    if (lane < kWarps) sel_scan[lane] = make_uint2(ga - v.x, ea - v.y);   // exclusive
  }
  __syncthreads();
  const uint32_t gt_before = sel_scan[warp].x, eq_before = sel_scan[warp].y;
  uint32_t out_pos = gt_before + min(eq_before, need_eq);   // warp-uniform
  uint32_t eq_seen = eq_before;                              // warp-uniform
  int32_t* out = idx + R.sel0;
  const uint32_t below = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w1 ? keys[i] & mask : 0u;
    const bool gt = i < w1 && key > tau;
    const bool eq = i < w1 && key == tau;
    const uint32_t be = __ballot_sync(0xffffffffu, eq);
    const bool take = gt || (eq && eq_seen + __popc(be & below) < need_eq);
    const uint32_t bt = __ballot_sync(0xffffffffu, take);
    if (take) {
      const uint32_t o = out_pos + __popc(bt & below);
      if (o < (uint32_t)k) out[o] = i;
    }
    out_pos += __popc(bt);
    eq_seen += __popc(be);
  }
}

// ---- top-k of large requests on a cluster of CTAs --------------------------
// The same selection, with a request's keys spread over the kTopkCluster CTAs
// of one thread-block cluster: CTA c holds the contiguous index range
// [c * per, (c + 1) * per) of the keys in its shared memory.  Every radix
// round builds each CTA's histogram of its keys; after a cluster barrier
// every CTA sums all the CTAs' histograms through distributed shared memory
// (in CTA order, so all reach the same digit).  The compaction takes each
// CTA's counts the same way, so CTA c writes its selected indices after
// those of CTAs 0 .. c - 1, in index order.  Histograms are double-buffered:
// a round's buffer is rewritten only two rounds later, after a barrier that
// every CTA passes once it has read the buffer.
constexpr int kTopkCluster = 8;
constexpr int kTcThreads = 512;

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

__global__ void __launch_bounds__(kTcThreads) topk_cluster_kernel(
    const fuse_request_t* reqs, const float* score, int32_t* idx, uint32_t* err,
    const float* partial, int n_parts, int n_kv_heads, float* score_out) {
  extern __shared__ uint32_t keys[];                 // this CTA's slice
  __shared__ uint32_t hist[2][256];
  __shared__ uint32_t xmin, xmax, xgt, xeq;          // read by the other CTAs
  __shared__ uint32_t s_digit, s_remaining, s_inbin;
  __shared__ uint32_t warp_a[32], warp_b[32];
  __shared__ uint2 pair_buf[32], sel_scan[32];
  const uint32_t crank = tc::cluster_rank();
  const int r = blockIdx.x / kTopkCluster;
  const fuse_request_t R = reqs[r];     // the caller's table: no kernel writes it
  pdl_trigger();
  pdl_wait();
  const int n = R.n_ctx;
  const int k = R.k;
  if (n <= 0) return;                   // the same in every CTA of the cluster
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  constexpr int kWarps = kTcThreads / 32;
  const int per = (((n + kTopkCluster - 1) / kTopkCluster) + 31) & ~31;
  const int c0 = min(n, (int)crank * per), c1 = min(n, c0 + per);
  const int m = c1 - c0;
  if (k <= 0) {                         // nothing to select; still form the scores
    if (partial)
      for (int i = c0 + t; i < c1; i += kTcThreads)
        score_out[R.score0 + i] = head_mean_score(partial + (R.score0 + i) * n_parts, n_parts, n_kv_heads);
    return;
  }

  // 1. keys of the slice (scores formed from the partials first), min and max
  bool nan_seen = false;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int j0 = t; j0 < m; j0 += kTopkBatch * kTcThreads) {
    float v[kTopkBatch];
    if (partial && n_parts == 4) {
      float4 pv[kTopkBatch];
#pragma unroll
      for (int q = 0; q < kTopkBatch; ++q) {
        const int j = j0 + q * kTcThreads;
        if (j < m) pv[q] = __ldg(reinterpret_cast<const float4*>(partial) + (R.score0 + c0 + j));
      }
#pragma unroll
      for (int q = 0; q < kTopkBatch; ++q)
        if (j0 + q * kTcThreads < m) v[q] = head_mean_score4(pv[q], n_kv_heads);
    } else {
#pragma unroll
      for (int q = 0; q < kTopkBatch; ++q) {
        const int j = j0 + q * kTcThreads;
        if (j < m)
          v[q] = partial ? head_mean_score(partial + (R.score0 + c0 + j) * n_parts, n_parts, n_kv_heads)
                         : score[R.score0 + c0 + j];
      }
    }
#pragma unroll
    for (int q = 0; q < kTopkBatch; ++q) {
      const int j = j0 + q * kTcThreads;
      if (j < m) {
        if (partial) score_out[R.score0 + c0 + j] = v[q];
        bool nn;
        const uint32_t key = float_key(v[q], &nn);
        keys[j] = key;
        kmin = min(kmin, key);
        kmax = max(kmax, key);
        nan_seen |= nn;
      }
    }
  }
  if (nan_seen) report_error(err, FUSE_ERR_DEVICE_BOUNDS, SITE_TOPK_NAN, r);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    warp_a[warp] = kmin;
    warp_b[warp] = kmax;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t a = lane < kWarps ? warp_a[lane] : 0xFFFFFFFFu, b = lane < kWarps ? warp_b[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
      b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    if (lane == 0) {
      xmin = a;
      xmax = b;
    }
  }
  tc::cluster_sync_all();               // every CTA's keys, min and max are in place
  kmin = 0xFFFFFFFFu;
  kmax = 0u;
  for (int c = 0; c < kTopkCluster; ++c) {
    kmin = min(kmin, ld_cluster_u32(tc::peer_smem(&xmin, c)));
    kmax = max(kmax, ld_cluster_u32(tc::peer_smem(&xmax, c)));
  }
  int lo = 32 - __clz(kmin ^ kmax);      // bits [0, lo) still differ between keys
  uint32_t mask = lo >= 32 ? 0u : ~((1u << lo) - 1u);
  uint32_t prefix = kmin & mask;
  uint32_t remaining = (uint32_t)k;

  // 2. radix rounds over the differing bits, 8 at a time, highest first
  int b = 0;
  while (lo > 0) {
    const int w = min(8, lo);
    const int shift = lo - w;
    const uint32_t dmask = (1u << w) - 1u;
    for (int i = t; i < 256; i += kTcThreads) hist[b][i] = 0u;
    __syncthreads();
    for (int base = t - lane; base < m; base += kTcThreads) {   // warp-uniform
      const int j = base + lane;
      const uint32_t key = j < m ? keys[j] : 0u;
      const bool act = j < m && (key & mask) == prefix;
      const uint32_t bin = act ? (key >> shift) & dmask : 0xFFFFFFFFu;
      const uint32_t lead = __shfl_sync(0xffffffffu, bin, 0);
      const uint32_t same = __ballot_sync(0xffffffffu, act && bin == lead);
      if (lane == 0 && same) atomicAdd(&hist[b][lead], (uint32_t)__popc(same));
      if (act && bin != lead) atomicAdd(&hist[b][bin], 1u);
    }
    tc::cluster_sync_all();             // every CTA's histogram of this round is complete
    if (warp == 0) {
      // the cluster's histogram (CTAs summed in order), scanned from the top,
      // 8 bins per lane
      uint32_t cnt[8], lsum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int bin = 255 - (lane * 8 + q);
        uint32_t acc = 0;
        for (int c = 0; c < kTopkCluster; ++c) acc += ld_cluster_u32(tc::peer_smem(&hist[b][bin], c));
        cnt[q] = acc;
        lsum += acc;
      }
      uint32_t incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t cum = incl - lsum;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (cum < remaining && cum + cnt[q] >= remaining) {
          s_digit = 255 - (lane * 8 + q);
          s_remaining = remaining - cum;
          s_inbin = cnt[q];
        }
        cum += cnt[q];
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= dmask << shift;
    remaining = s_remaining;
    const uint32_t in_bin = s_inbin;
    lo = shift;
    b ^= 1;
    __syncthreads();
    if (in_bin == remaining) break;     // the same decision in every CTA
  }
  const uint32_t tau = prefix;
  const uint32_t need_eq = remaining;

  // 3. compaction in index order: warps own contiguous ranges of the slice,
  //    CTAs contiguous ranges of the request
  const int per_w = (((m + kWarps - 1) / kWarps) + 31) & ~31;
  const int w0 = min(m, warp * per_w), w1 = min(m, w0 + per_w);
  uint32_t n_gt = 0, n_eq = 0;
  for (int base = w0; base < w1; base += 32) {
    const int j = base + lane;
    const uint32_t key = j < w1 ? keys[j] & mask : 0u;
    n_gt += __popc(__ballot_sync(0xffffffffu, j < w1 && key > tau));
    n_eq += __popc(__ballot_sync(0xffffffffu, j < w1 && key == tau));
  }
  if (lane == 0) pair_buf[warp] = make_uint2(n_gt, n_eq);
  __syncthreads();
  if (warp == 0) {
    const uint2 v = lane < kWarps ? pair_buf[lane] : make_uint2(0u, 0u);
    uint32_t ga = v.x, ea = v.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t yg = __shfl_up_sync(0xffffffffu, ga, o);
      const uint32_t ye = __shfl_up_sync(0xffffffffu, ea, o);
      if (lane >= o) {
        ga += yg;
        ea += ye;
      }
    }
    if (lane < kWarps) sel_scan[lane] = make_uint2(ga - v.x, ea - v.y);
    if (lane == 31) {
      xgt = ga;                          // this CTA's totals
      xeq = ea;
    }
  }
  tc::cluster_sync_all();               // every CTA's totals are in place
  uint32_t gt_cta = 0, eq_cta = 0;      // keys of the CTAs before this one
  for (int c = 0; c < (int)crank; ++c) {
    gt_cta += ld_cluster_u32(tc::peer_smem(&xgt, c));
    eq_cta += ld_cluster_u32(tc::peer_smem(&xeq, c));
  }
  const uint32_t eq_before = eq_cta + sel_scan[warp].y;
  uint32_t out_pos = gt_cta + sel_scan[warp].x + min(eq_before, need_eq);
  uint32_t eq_seen = eq_before;
  int32_t* out = idx + R.sel0;
  const uint32_t below = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int j = base + lane;
    const uint32_t key = j < w1 ? keys[j] & mask : 0u;
    const bool gt = j < w1 && key > tau;
    const bool eq = j < w1 && key == tau;
    const uint32_t be = __ballot_sync(0xffffffffu, eq);
    const bool take = gt || (eq && eq_seen + __popc(be & below) < need_eq);
    const uint32_t bt = __ballot_sync(0xffffffffu, take);
    if (take) {
      const uint32_t o = out_pos + __popc(bt & below);
      if (o < (uint32_t)k) out[o] = c0 + j;
    }
    out_pos += __popc(bt);
    eq_seen += __popc(be);
  }
  tc::cluster_sync_all();               // no CTA leaves while another reads its memory
}

// Cluster launch of kTopkCluster CTAs per request, with programmatic
// stream serialisation.
template <typename... Args>
cudaError_t launch_topk_cluster(int n_req, size_t smem, cudaStream_t s, Args... args) {
  static const bool attr_ok = [] {
    return cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kTopkSmemKeys * (int)sizeof(uint32_t)) == cudaSuccess;
  }();
  if (!attr_ok) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_req * kTopkCluster);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kTopkCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel, args...);
}

// Requests large enough for the cluster kernel, and small enough for its
// shared memory.
bool topk_use_cluster(int max_ctx) {
  const int64_t per = (((int64_t)max_ctx + kTopkCluster - 1) / kTopkCluster + 31) & ~31;
  return max_ctx > kTopkClusterMin && per <= kTopkSmemKeys;
}

}  // namespace

cudaError_t launch_reduce_topk(const fuse_requests_t& reqs, int max_ctx, const float* partial,
                               int n_parts, int n_kv_heads, float* score, int32_t* idx,
                               uint32_t* keys_ws, uint32_t* err, cudaStream_t s) {
  if (reqs.n_req == 0) return cudaSuccess;
  if (topk_use_cluster(max_ctx)) {
    const size_t per = (((size_t)max_ctx + kTopkCluster - 1) / kTopkCluster + 31) & ~(size_t)31;
    return launch_topk_cluster(reqs.n_req, per * sizeof(uint32_t), s, reqs.d_req,
                               (const float*)nullptr, idx, err, partial, n_parts, n_kv_heads,
                               score);
  }
  const int in_smem = max_ctx <= kTopkSmemKeys;
  const size_t smem = in_smem ? (size_t)max_ctx * sizeof(uint32_t) : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTopkSmemKeys * (int)sizeof(uint32_t));
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(topk_kernel, dim3(reqs.n_req), dim3(kTopkThreads), smem, s, reqs.d_req,
                    (const float*)nullptr, idx, keys_ws, err, in_smem, partial, n_parts,
                    n_kv_heads, score);
}

cudaError_t launch_topk(const fuse_requests_t& reqs, int max_ctx, const float* score, int32_t* idx,
                        uint32_t* keys_ws, uint32_t* err, cudaStream_t s) {
  if (reqs.n_req == 0) return cudaSuccess;
  if (topk_use_cluster(max_ctx)) {
    const size_t per = (((size_t)max_ctx + kTopkCluster - 1) / kTopkCluster + 31) & ~(size_t)31;
    return launch_topk_cluster(reqs.n_req, per * sizeof(uint32_t), s, reqs.d_req, score, idx, err,
                               (const float*)nullptr, 0, 0, (float*)nullptr);
  }
  const int in_smem = max_ctx <= kTopkSmemKeys;
  const size_t smem = in_smem ? (size_t)max_ctx * sizeof(uint32_t) : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTopkSmemKeys * (int)sizeof(uint32_t));
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(topk_kernel, dim3(reqs.n_req), dim3(kTopkThreads), smem, s, reqs.d_req, score,
                    idx, keys_ws, err, in_smem, (const float*)nullptr, 0, 0, (float*)nullptr);
}

}  // namespace fusekv

// ----------------------------------------------------------------------------
// Top-k without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they select
// tokens: a serving loop that has handed every byte of HBM to its KV-cache
// pool, or code running inside a framework callback that must not touch the
// allocator.  For them the key scratch of the top-k lives in this file-scope
// device array instead of a workspace.  It is created when the library is
// loaded and held on every GPU that loads the library until the process
// exits.
// ----------------------------------------------------------------------------
#include <mutex>

namespace fusekv {
namespace {

constexpr int kNoallocHeaderWords = 64;          // word 0: device error code (written, never read)
constexpr int kNoallocMaxDevices = 64;

static __device__ __align__(256) uint32_t g_topk_scratch[kNoallocHeaderWords + FUSE_TOPK_NOALLOC_MAX_KEYS];

std::mutex g_noalloc_mu;
uint32_t* g_noalloc_addr[kNoallocMaxDevices] = {};

// Device address of g_topk_scratch on the current device; looked up once
// per device (host code cannot use the symbol itself as an address).
cudaError_t noalloc_scratch(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_noalloc_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace fusekv

extern "C" fuse_status_t fuse_select_topk_noalloc(const fuse_requests_t* reqs, const float* score,
                                                  int32_t* idx, fuse_stream_t stream) {
  using namespace fusekv;
  if (!reqs || reqs->n_req < 0) return FUSE_ERR_INVALID_ARG;
  if (reqs->n_req > 65535) return FUSE_ERR_UNSUPPORTED;   // the request-table limit of every call
  if (reqs->n_req == 0) return FUSE_OK;
  if (!reqs->h_req || !reqs->d_req) return FUSE_ERR_INVALID_ARG;
  int64_t n_ctx = 0, n_sel = 0;
  int max_ctx = 0;
  for (int i = 0; i < reqs->n_req; ++i) {
    const fuse_request_t& q = reqs->h_req[i];
    if (q.n_ctx < 0 || q.n_query < 0 || q.k < 0 || q.k > q.n_ctx || q.reserved != 0 ||
        q.score0 < 0 || q.sel0 < 0)
      return FUSE_ERR_INVALID_ARG;
    n_ctx = std::max<int64_t>(n_ctx, q.score0 + q.n_ctx);
    n_sel = std::max<int64_t>(n_sel, q.sel0 + q.k);
    max_ctx = std::max(max_ctx, q.n_ctx);
  }
  if (n_ctx > FUSE_TOPK_NOALLOC_MAX_KEYS) return FUSE_ERR_WORKSPACE;
  if (n_sel == 0) return FUSE_OK;
  if (!score || !idx) return FUSE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(score) | reinterpret_cast<uintptr_t>(idx)) & 15u)
    return FUSE_ERR_MISALIGNED;
  uint32_t* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return FUSE_ERR_CUDA;
  // The kernel records a NaN score in the scratch's error word, which nothing
  // reads (this variant does not report NaN), so the word is never cleared.
  // cudaLaunchKernelEx returns this launch's own error, not one left pending
  // by earlier work.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(reqs->n_req);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = (cudaStream_t)stream;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, topk_kernel, reqs->d_req, score, idx, scratch + kNoallocHeaderWords,
                         scratch, /*keys_in_smem=*/0, (const float*)nullptr, 0, 0, (float*)nullptr);
  (void)max_ctx;
  return e == cudaSuccess ? FUSE_OK : FUSE_ERR_CUDA;
}
