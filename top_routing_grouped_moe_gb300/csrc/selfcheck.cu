// Failure detection, checked without a fault: a kernel waits on an mbarrier
// phase that nothing completes, through the same bounded wait the GEMMs use,
// with a short limit.  The wait gives up, the kernel records MOE_ERR_TIMEOUT
// in the device status word and returns; the context stays usable.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(unsigned long long limit_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);  // one expected arrival, which never comes
    volatile int never = 0;
    if (!ptx::mbar_wait_bounded(&bar, 0, &never, limit_ns)) record_status(status, MOE_ERR_TIMEOUT);
  }
}

}  // namespace
}  // namespace moe

extern "C" MOE_API int moe_selftest_wait_timeout(int limit_us, void* stream) {
  using namespace moe;
  if (limit_us < 1 || (unsigned long long)limit_us * 1000ull > kWaitLimitNs) return MOE_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((unsigned long long)limit_us * 1000ull,
                                                                       device_status_ptr());
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
