// Self-test of the failure path.  One block waits on a barrier that nothing
// arrives at, gives up after a short limit and records CP_ERR_TIMEOUT in the
// status word, exactly as a scan kernel does when one of its bounded waits
// runs out; the context stays usable.  Callers (and the tests) read the
// status back with causal_product_status.
#include "cp_internal.h"
#include "sm103_ptx.cuh"

namespace cp {
namespace {

__global__ void selftest_timeout_kernel(int* status, uint64_t wait_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !ptx::mbar_wait_timeout(&bar, 0, wait_ns))
    atomicCAS(status, 0, (int)CP_ERR_TIMEOUT);
}

}  // namespace

cudaError_t selftest_timeout_launch(int* status, uint64_t wait_ns, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(status, wait_ns);
  return cudaGetLastError();
}

}  // namespace cp
