// debug.cu - a kernel whose wait is made to run out, so that the bounded-wait
// and status-word path can be exercised end to end without hanging a GPU.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_kernels.h"
#include "mx_ptx.cuh"

namespace mx {

namespace {

// One thread initialises an mbarrier that expects one arrival and never gets
// it, then waits on it with the same bounded loop the GEMM uses (but with the
// caller's limit).  On expiry it sets the status word and returns.
__global__ void expire_wait_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(&bar, 0)) {
    if (globaltimer() - t0 > limit_ns) {
      atomicOr(&g_status, kStatusTimeout);
      return;
    }
  }
}

}  // namespace

cudaError_t launch_expire_wait(uint64_t timeout_ns, cudaStream_t stream) {
  expire_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns);
  return cudaGetLastError();
}

cudaError_t take_status_debug(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace mx
