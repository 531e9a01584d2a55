// Self-test of the bounded waits (a library diagnostic with no counterpart in the pages).
// One CTA waits, through the bounded wait every kernel of the library uses, on an mbarrier
// phase that nothing completes.  When the wait limit passes, the wait records kDevTimeout in
// the device status word and returns, and the kernel exits: the context stays usable.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace gcs {
namespace {

__global__ void __launch_bounds__(32, 1) bounded_wait_selftest_kernel(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  const Abort ab{&abort_flag, status};
  // phase 0 never completes: nothing arrives on the barrier and no copy targets it
  if (!wait_bar(&bar, 0, ab)) return;
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int* status, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(status);
  return cudaGetLastError();
}

}  // namespace gcs
