// Self-test of the failure path of the kernels' pipeline waits.
//
// Every wait of the compressor kernels on a shared-memory mbarrier goes
// through mbar_wait_bounded_for: it gives up after a limit of SM clock cycles,
// the kernel records KVC_ERR_TIMEOUT in the device error word and returns
// instead of hanging.  This kernel makes that path run on purpose, without a
// fault: one thread waits on a barrier that nothing will ever complete, with
// a short limit chosen by the caller, then records the timeout.  The context
// stays usable, which the tests check by running the compressor afterwards.

#include <cuda_runtime.h>

#include "kvc_device.cuh"

namespace kvc {
namespace {

using namespace dev;

__global__ void kvc_selftest_wait_kernel(long long limit, uint32_t* error) {
  __shared__ unsigned long long bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);  // one arrival expected; none will come
  fence_mbar_init();
  if (!mbar_wait_bounded_for(&bar, 0u, limit)) record_error(error, kErrTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(long long limit_cycles, uint32_t* err, cudaStream_t stream) {
  kvc_selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_cycles, err);
  return cudaGetLastError();
}

}  // namespace kvc
