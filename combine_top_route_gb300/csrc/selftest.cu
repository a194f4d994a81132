// Self-test of the library's failure detection: the bounded mbarrier wait that
// every pipelined kernel uses gives up after its time limit, latches
// OCCULT_ERR_DEVICE_TIMEOUT into the device error word and lets the kernel
// return, so the context stays usable.  The test kernel waits on a barrier that
// nothing completes (or, as a control, one it completes itself); it touches no
// memory but its own shared memory and the error word.
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

__global__ void __launch_bounds__(32)
selftest_wait_kernel(int complete, uint64_t limit_ns, int* dev_err) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    if (complete) mbar_arrive(&bar);
    if (!mbar_wait(&bar, 0, &abort_flag, limit_ns)) latch_error(dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
  }
}

}  // namespace

int launch_selftest_wait(const LaunchCtx& ctx, int complete, uint64_t limit_ns) {
  launch_pdl(selftest_wait_kernel, 1, 32, 0, ctx.stream, complete, limit_ns, ctx.dev_err);
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
