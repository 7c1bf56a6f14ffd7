// Device-side flag of expired bounded waits, one word per device.
//
// Kernels whose warps wait on mbarriers bound every wait by an iteration
// limit. When a limit is reached the kernel ORs a code into this word, winds
// down without trapping, and the host learns of it through
// m3_device_status(). The word is a file-scope __device__ variable, so every
// device that loads the library holds its own copy.
#include "launch.h"

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

}  // namespace m3
