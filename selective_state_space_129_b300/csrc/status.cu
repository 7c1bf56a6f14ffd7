// Device-side flag of expired bounded waits, one word per device.
//
// Kernels whose warps wait on mbarriers bound every wait by an iteration
// limit. When a limit is reached the kernel ORs a code into this word, winds
// down without trapping, and the host learns of it through
// m3_device_status(). The word is a file-scope __device__ variable, so every
// device that loads the library holds its own copy.
#include "launch.h"
#include "ptx.cuh"

namespace m3 {

__device__ unsigned int g_wait_status = 0u;

cudaError_t status_word(unsigned int** ptr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_wait_status);
}

cudaError_t read_clear_status(unsigned int* value, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(value, g_wait_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0u;
  return cudaMemcpyToSymbol(g_wait_status, &zero, sizeof(unsigned int));
}

namespace {

// One mbarrier that nothing arrives at, waited on with the kernels' bounded
// wait: the wait runs out after limit_ns and the expiry is recorded in the
// status word exactly as a kernel's would be.
__global__ void expired_wait_kernel(unsigned int* status, uint64_t limit_ns) {
  __shared__ uint64_t never;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&never, 1);
    ptx::fence_mbar_init();
    if (!ptx::mbar_wait(&never, 0u, limit_ns)) atomicOr(status, 2u);
  }
}

}  // namespace

cudaError_t launch_expired_wait(uint64_t limit_ns, cudaStream_t s) {
  unsigned int* status = nullptr;
  cudaError_t e = status_word(&status);
  if (e != cudaSuccess) return e;
  expired_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace m3
