// Self-test of the failure path every pipelined kernel relies on: a barrier wait
// whose partner never arrives must give up within its budget, record
// BSA_ERR_TIMEOUT in the caller's status word and return, leaving the CUDA
// context usable.  The wait here is the kernels' own bounded mbar_wait, with a
// budget of about ten milliseconds instead of seconds.
#include "common.cuh"
#include "kernels.h"

namespace bsa {
namespace {

constexpr long long kSelftestCycles = 20000000LL;

__global__ void wait_timeout_selftest_kernel(int32_t *status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival expected; none is ever made
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    (void)mbar_wait<kSelftestCycles>(smem_u32(&bar), 0, &abort_flag, status);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int32_t *dev_status, cudaStream_t st) {
  wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(dev_status);
  return cudaGetLastError();
}

}  // namespace bsa
