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

#ifdef FA_DEBUG
// FA_DEBUG builds: one thread hands the device-side checks a value that breaks the
// rule of check `kind` (the kinds of ptx.cuh's kDbg* codes), the way the kernels
// call them before every copy, tensor-memory access and at CTA exit.  Nothing is
// copied or accessed: the clamped values the checks return are discarded, so the
// only effect is the record the failed check leaves.
__global__ void fa_selftest_check_kernel(uint32_t* err, int kind) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  dbg_tmem_base = 0;
  dbg_err_ptr = err;
  const Extent3 ext{128, 300, 4};  // a [4, 300, 128] tensor
  int c0 = 0, c1 = 0, c2 = 0;
  long long first = 0;
  volatile uint32_t sink = 0;
  switch (kind) {
    case kDbgTmaCol: c0 = 72; check_box(c0, c1, c2, ext, err); break;     // not a multiple of 64
    case kDbgTmaRow: c1 = 512; check_box(c0, c1, c2, ext, err); break;    // rows 300 -> 512 is past the end
    case kDbgTmaPlane: c2 = 4; check_box(c0, c1, c2, ext, err); break;    // planes 0..3
    case kDbgTmemCol: sink = tm(480, 64); break;                          // columns 480..543 of 512
    case kDbgTmemLane: sink = tm(16u << 16, 32); break;                   // lane 16: not a warp's quarter
    case kDbgBulk: first = 1020; check_rows(first, 512, 1024, err); break;  // 128 floats from 1020 of 1024
    case kDbgPhase: {                                                     // 0 phases completed, 1 expected
      const uint32_t b = smem_u32(&bar);
      mbar_init(b, 1);
      fence_mbar_init();
      check_phase(b, 1, err, 0);
      break;
    }
    default: break;
  }
  (void)sink;
}
#endif

}  // namespace

#ifdef FA_DEBUG
cudaError_t launch_selftest_check(uint32_t* err, int kind, cudaStream_t stream) {
  fa_selftest_check_kernel<<<1, 32, 0, stream>>>(err, kind);
  return cudaGetLastError();
}
#endif

cudaError_t launch_selftest_wait(uint32_t* err, uint64_t limit_ns, cudaStream_t stream) {
  fa_selftest_wait_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace fa
