// Self-tests of the device status path.
//   k_status_selftest  One CTA waits, with the bounded mbarrier wait the Newton-Schulz
//                      kernels use, on a barrier that nothing completes.  When the limit
//                      runs out it records a timeout in the device status word, as a
//                      stalled chain kernel would, and returns; the context stays usable.
//                      nsm_device_status then reports it, and nsm_device_status_detail
//                      names this kernel and its barrier (role 0).
//   k_bounds_selftest  One thread runs the bounds test the kernels use on an index one
//                      past the end of a one-element range and makes no access.  The
//                      checked build records the failure; the regular build compiles the
//                      test out and records nothing.
#include <cuda_runtime.h>

#include "nsm_internal.h"
#include "ptx.cuh"

namespace nsm {
namespace {

__global__ void k_status_selftest(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int never;
  if (threadIdx.x == 0) {
    never = 0;
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // no thread ever arrives: phase 0 of the barrier does not complete
    if (!ptx::mbar_wait_bounded(ptx::smem_u32(&bar), 0u, &never, limit_ns)) {
      record_timeout(status, NSM_KERNEL_SELFTEST, 0, NSM_SITE_SELFTEST);
    }
  }
}

__global__ void k_bounds_selftest(int* status, int len) {
  const int i = static_cast<int>(threadIdx.x) + len;  // one past the end
  (void)bounds_ok(i >= 0 && i < len, status, NSM_KERNEL_SELFTEST, 0, NSM_SITE_SELFTEST_BOUNDS);
}

}  // namespace

cudaError_t launch_bounds_selftest(cudaStream_t stream) {
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  k_bounds_selftest<<<1, 1, 0, stream>>>(status, 1);
  return cudaGetLastError();
}

cudaError_t launch_status_selftest(uint64_t limit_ns, cudaStream_t stream) {
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  k_status_selftest<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace nsm
