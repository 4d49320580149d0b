// Self-test of the failure path every kernel of the library shares: a bounded mbarrier wait
// that nothing completes gives up after its time limit, records QG_ERR_TIMEOUT in the
// workspace status word and returns, leaving the CUDA context usable.  It faults nothing:
// the wait simply runs out.
#include <cuda_runtime.h>

#include "qg_internal.h"
#include "qg_sync.cuh"

namespace qg {

__global__ void selftest_wait_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, status);  // no arrival will ever come
}

}  // namespace qg

extern "C" qg_status qg_selftest_wait_timeout(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return QG_ERR_INVALID_ARG;
  if (workspace_bytes < sizeof(int)) return QG_ERR_WORKSPACE_TOO_SMALL;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return QG_ERR_MISALIGNED;
  qg::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<int*>(workspace));
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}
