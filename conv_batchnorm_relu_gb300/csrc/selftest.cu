// Failure-detection self-test: one warp waits, with the bounded mbarrier wait every library
// kernel uses, on a barrier that nothing will complete.  When the limit runs out it records
// the timeout in the device error word and exits, exactly as a library kernel that gives up
// on a wait does, so the host-side detection (cbr_stream_status) can be exercised without a
// fault, a trap or a hang.
#include "cbr_internal.h"
#include "common.cuh"

namespace cbr {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // one arrival expected; none is ever made
    fence_mbarrier_init();
  }
  __syncwarp();
  const bool done = mbar_wait(b, 0, limit_ns);
  if (threadIdx.x == 0 && !done) report_error(err, kErrWaitOperand);
}

}  // namespace

int launch_selftest_wait(uint32_t* err, uint64_t limit_ns, cudaStream_t st) {
  bounded_wait_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

}  // namespace cbr
