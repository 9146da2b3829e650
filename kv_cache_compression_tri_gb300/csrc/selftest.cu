// selftest.cu -- a check of the failure path every kernel shares: a bounded
// mbarrier wait that runs out records TRI_DEV_TIMEOUT in the caller's status
// word and returns, leaving the context usable. The wait here is on an
// mbarrier that nothing arrives on, so it always runs out; the kernels use the
// same wait (mbar_wait_limit) with a limit of about two seconds.
#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

__global__ void wait_timeout_kernel(int32_t* dev_status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  mbar_init_fence();
  if (!mbar_wait_limit(&bar, 0u, limit_ns)) set_status(dev_status, TRI_DEV_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int32_t* dev_status, uint64_t limit_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(dev_status, limit_ns);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tri
