// selftest.cu -- exercises the failure path every kernel shares: a bounded mbarrier wait
// that runs out records kDevTimeout in the device status word and returns, so the kernel
// ends and the context stays usable.  The kernel waits on a barrier that nothing arrives on.
#include "internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

__global__ void selftest_wait_kernel(uint64_t limit_ns, uint32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  // phase 0 needs one arrival; none comes, so the wait gives up after limit_ns
  mbar_wait(b, 0, status, limit_ns);
}

}  // namespace

cudaError_t launch_selftest_wait(uint64_t limit_ns, uint32_t* status, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace fa
