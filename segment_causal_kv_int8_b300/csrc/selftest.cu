// selftest.cu - kernels that exercise the library's two device-side error
// paths without any fault: the bounded wait and (checked build) the range
// check.
//
// Every wait of the library's kernels on an mbarrier gives up after a time
// limit, records NOMAS_ERR_DEVICE_TIMEOUT in the device error word and
// returns, so a lost arrival never hangs the GPU.  This kernel waits, with the
// caller's limit, on a barrier that nothing ever arrives on, which takes that
// path on purpose without any fault: the wait ends by the clock, the error word
// is set, and the kernel exits normally.
#include <cuda_runtime.h>
#include <stdint.h>

#include "checks.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace nomas {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ AbortState ab;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival that never comes
    ab.flag = 0;
    fence_mbarrier_init();
  }
  __syncwarp();
  warp_wait_limit(&bar, 0, &ab, err, limit_ns);
}

// Checked build: one range check of index 4 against a buffer declared to
// hold 4 elements, which fails, records NOMAS_ERR_INVALID_ARG and skips the
// store.  (Launched only in the checked build; the array has a fifth element
// so the store would stay in bounds even without the check.)
__global__ void __launch_bounds__(32) bounds_check_kernel(uint32_t* err) {
  __shared__ volatile uint32_t buf[5];
  if (threadIdx.x == 0 && in_bounds(4, 1, 4, err)) buf[4] = 1u;
}

}  // namespace

bool bounds_checked_build() { return kBoundsChecked; }

cudaError_t launch_bounds_check_selftest(uint32_t* err, cudaStream_t stream) {
  if (!kBoundsChecked) return cudaErrorNotSupported;
  bounds_check_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace nomas
