// Self-test of the device-side failure detection: a bounded mbarrier wait on
// a barrier that nothing arrives on gives up and is reported through the
// workspace's error word, with no fault and no endless wait.
#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace fusekv {
namespace {

// Site of the self-test's report (err_detail's top byte; outside ErrSite).
constexpr uint32_t kSiteSelfTest = 0xEE;

__global__ void selftest_wait_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0))
    report_error(err, FUSE_ERR_TIMEOUT, kSiteSelfTest, 0);
}

}  // namespace

cudaError_t launch_selftest_wait(uint32_t* err, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(err);
  return cudaGetLastError();
}

}  // namespace fusekv
