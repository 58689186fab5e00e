// selftest.cu: exercises the bounded-wait failure path without any fault.
// One CTA waits on an mbarrier phase that nothing completes; the wait must
// expire after limit_ns, record its site in the device status word and let the
// kernel return normally.
#include "internal.h"

namespace dg {
namespace {

__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // expects one arrival; none ever comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl wc{limit_ns, status, &abort_flag};
    if (!wait_bounded(smem_u32(&bar), 0, wc, kSiteSelfTest)) return;
  }
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, int* status, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace dg
