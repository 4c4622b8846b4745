// k_selftest.cu -- exercises the failure path of the bounded waits.
//
// Every barrier wait of the Newton-Schulz kernels gives up after a time
// limit, records MUON_ERR_TIMEOUT in the handle's device flag and lets the
// kernel return, so that a lost arrival never hangs the GPU.  This kernel
// waits on a barrier that nothing will ever complete, through the same
// wait routine, with a short limit: the wait must expire, the flag must be
// set, and the kernel must return normally.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace muon {
namespace {

__global__ void bounded_wait_selftest_kernel(int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);  // one arrival expected; none will come
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns)) atomicOr(err, kDevErrTimeout);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace muon
