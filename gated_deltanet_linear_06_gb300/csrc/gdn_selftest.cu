// gdn_selftest.cu -- a self-test of the device-side failure path.
//
// Every wait of the tensor-core kernels is bounded: tc::mbar_wait gives up
// after a budget of clock cycles, the kernel records GDN_ERR_DEVICE_TIMEOUT in
// its status word and exits, and the context stays usable.  A real kernel only
// takes that path when a copy or a product never completes, which cannot be
// provoked safely.  This kernel takes it on purpose, on the same helpers: one
// CTA waits on a shared-memory mbarrier that nothing ever arrives on (a flag
// nothing sets), with a short budget, and reports the time-out.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_trace.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

__global__ void wait_timeout_kernel(int32_t* status, long long budget) {
  __shared__ __align__(8) uint64_t mbar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&mbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // phase 0 of a barrier expecting one arrival that never comes
  const bool landed = tc::mbar_wait(&mbar, 0, budget);
  if (!__syncthreads_or(landed ? 1 : 0) && threadIdx.x == 0)
    record_status(status, GDN_ERR_DEVICE_TIMEOUT);
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_selftest_wait_timeout(int32_t* device_status, long long budget_cycles,
                                                void* stream) {
  gdn::TraceRange trace_range("gdn_selftest_wait_timeout");
  if (!device_status || (reinterpret_cast<uintptr_t>(device_status) & 3u) || budget_cycles < 1 ||
      budget_cycles > (1LL << 31))
    return GDN_ERR_INVALID_ARG;
  gdn::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(device_status,
                                                                           budget_cycles);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
