// Self-test of the device-side failure path: a bounded mbarrier wait that runs out.
//
// Every kernel of the library bounds its mbarrier waits by %globaltimer and, on giving up,
// sets a bit in the context's status word instead of trapping, so that the CUDA context
// stays usable and oscar_check_status reports the failure.  This kernel takes that path on
// purpose: one thread waits on a barrier that nothing arrives on (a flag that nothing
// sets) until the caller's limit, then sets the timeout bit and returns.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

__global__ void wait_selftest_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // expects one arrival; none comes
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&bar, 0)) {
      if (globaltimer_ns() - t0 > limit_ns) {
        flag_error(status, kDevTimeout);
        break;
      }
    }
  }
}

}  // namespace

int launch_wait_selftest(int* status, long long limit_ns, void* stream) {
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, (unsigned long long)limit_ns);
  return (int)cudaGetLastError();
}

}  // namespace oscar
