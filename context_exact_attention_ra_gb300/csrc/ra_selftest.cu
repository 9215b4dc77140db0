// Self-test of the device-timeout path: one block waits, through the same
// bounded wait the attention kernels use, on an mbarrier that nothing ever
// arrives on.  The wait must give up after the given limit, set its bit in the
// device error word and let the kernel finish, so that the host sees
// RA_ERR_TIMEOUT and the device stays usable.  Nothing here faults or hangs:
// the only thing that runs out is the wait.

#include <cuda_runtime.h>

#include <cstdint>

#include "ra_internal.h"
#include "ra_wait.cuh"
#include "sm103_ptx.cuh"

namespace ra {
namespace {

__global__ void unsatisfied_wait_kernel(unsigned int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t barrier;
  __shared__ int abort_flag;
  const uint32_t bar = ptx::smem_u32(&barrier);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Abort ab{&abort_flag, err};
    wait_bar(bar, 0, ab, kErrSelfTest, limit_ns);   // no arrival will come
  }
}

}  // namespace

int launch_selftest_timeout(unsigned int* err, uint64_t limit_ns, void* stream) {
  launch_stage() = "self-test kernel launch";
  unsatisfied_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, limit_ns);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace ra
