// Self-test of the GEMMs' failure detection: the bounded pipeline wait.
//
// Every wait of the grouped-GEMM pipeline gives up after a time limit, sets
// LIGER_MOE_DEVERR_WAIT_TIMEOUT in the device error flag and lets the kernel return, so a
// stalled pipeline is reported instead of hanging the GPU.  This kernel makes that path run on
// purpose: one thread waits, through the same wait primitive, on an mbarrier phase that nothing
// ever completes, with a short limit, and records the timeout in the flag exactly as a GEMM role
// would.  Nothing faults and nothing waits past the limit.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace lmoe {
namespace {

__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, int* err) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival completes phase 0; none is ever made
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int never = 0;
    if (!mbar_wait(smem_u32(&bar), 0u, &never, limit_ns)) atomicOr(err, LIGER_MOE_DEVERR_WAIT_TIMEOUT);
  }
}

}  // namespace

int launch_bounded_wait_selftest(uint64_t limit_ns, const DeviceInfo& dev, cudaStream_t s) {
  {
    KernelScope trace("bounded_wait_selftest", s);
    launch_kernel(bounded_wait_selftest_kernel, dim3(1), dim3(32), 0, s, "bounded_wait_selftest", 1, limit_ns,
                  dev.err_flag);
  }
  return check_launch("bounded_wait_selftest");
}

}  // namespace lmoe
