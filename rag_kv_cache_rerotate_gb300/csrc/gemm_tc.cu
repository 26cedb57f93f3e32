// Tensor-core (tcgen05 / TMEM / TMA) projection GEMMs: bf16 operands, fp32
// accumulators in tensor memory.
#include "common.cuh"
#include "launch.h"

namespace fusekv {

bool tc_gemm_supported(const fuse_layer_desc_t&) { return false; }

cudaError_t launch_deviation_partials_tc(const fuse_layer_desc_t&, int64_t, const void*, const void*,
                                         const void*, const int32_t*, float*, uint32_t*,
                                         cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t launch_project_recompute_tc(const fuse_layer_desc_t&, int64_t, const WorkRow*,
                                        const float2*, const void*, const void*, const void*,
                                        const void*, void*, void*, void*, void*, uint32_t*,
                                        cudaStream_t) {
  return cudaErrorNotSupported;
}

bool tc_attention_supported(const fuse_layer_desc_t&) { return false; }

cudaError_t launch_attention_tc(const fuse_layer_desc_t&, int64_t, int, const fuse_request_t*,
                                const WorkRow*, const void*, const void*, const void*, void*,
                                uint32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace fusekv
