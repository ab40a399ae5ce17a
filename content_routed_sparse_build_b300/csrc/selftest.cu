// selftest.cu -- exercises the bounded wait every kernel of the library uses.
//
// One thread waits, with the given limit, on an mbarrier that nothing
// arrives at, then records SSA_DEVERR_WAIT_TIMEOUT in the workspace's error
// record and returns: the same give-up path as the attend and router kernels,
// with no bulk copy and no tensor memory involved, so that a test can run it
// out on a real device and check that the status comes back and the
// context stays usable.
#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(uint32_t* __restrict__ err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, limit_ns)) flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace ssa
