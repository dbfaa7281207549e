// A check of the failure path every kernel of the library shares: a wait on
// an mbarrier that nothing will ever complete. The bounded wait (the same
// mbar_wait the GEMMs and routers use) gives up after kWaitLimitNs of
// %globaltimer, records the timeout bit in the device status word and
// returns, so the context stays usable; no fault, no trap, no hang.
#include "mm.h"
#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncwarp();
  // Phase 0 needs one arrival, and none is ever made.
  if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0)) atomicOr(err, kDevErrTimeout);
}

}  // namespace
}  // namespace mm

extern "C" int mm_selftest_wait_timeout(void* stream) {
  unsigned* status = nullptr;
  const int rc = mm::current_status_word(&status);
  if (rc != MM_OK) return rc;
  mm::wait_timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
  return cudaGetLastError() == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}
