// Failure-detection self-test: one thread waits, through the same bounded wait
// every kernel of the library uses, on an mbarrier that nothing ever arrives on.
// The wait gives up after the given limit, records the failure in the device
// error record and returns, so the kernel ends and the context stays usable;
// fa_check_device_status then reports it like any real timeout.
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

__global__ void fa_selftest_wait_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    mbar_wait_for(b, 0, err, kErrSelfTest, false, limit_ns);  // no arrival: gives up
  }
}

}  // namespace

cudaError_t launch_selftest_wait(uint32_t* err, uint64_t limit_ns, cudaStream_t stream) {
  fa_selftest_wait_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace fa
