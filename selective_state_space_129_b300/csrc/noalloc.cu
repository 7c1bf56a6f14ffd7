// Prefill that allocates no device memory.
//
// Some callers cannot have a library allocate device memory on their behalf:
// a framework or inference server whose allocator owns all of the GPU's memory
// and hands it out itself, or a latency-critical caller for which a device
// allocation (it may block, and it may fail under memory pressure) is not
// acceptable. m3_scan_fwd needs scratch for segmented long sequences and,
// when the caller gives none, allocates it. m3_scan_fwd_noalloc runs the same
// computation with that scratch in a fixed array of this library instead.
//
// The array lives in device memory for as long as the library is loaded, on
// every GPU that loads it. Its host-side name is only a stand-in for the
// symbol, not a device address, so every call looks up the current device's
// address of the array (cudaGetSymbolAddress, a host-side query that
// allocates nothing; the first call on a device also loads the library's
// device code there) and passes it on as the workspace pointer. Looking it up
// each time, rather than remembering it per device, keeps the address right
// if the device's context is destroyed and created again (cudaDeviceReset),
// after which the array may sit elsewhere.
#include <cuda_runtime.h>
#include <stdint.h>

#include "m3scan.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the current device's copy of the scratch array.
m3_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return M3_ERR_CUDA;
  }
  *out = p;
  return M3_OK;
}

}  // namespace

extern "C" {

m3_status m3_scan_fwd_noalloc(const void* x, const float* dt, const float* A, const float* lambda,
                              const void* B, const void* C, const float* theta,
                              const m3_dims* dims, int R, int chunk, void* out,
                              float* final_state, void* stream) {
  if (dims == nullptr) return M3_ERR_INVALID_ARG;
  const size_t need = m3_scan_workspace_bytes(dims, R, chunk);
  if (need == (size_t)-1) return M3_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return M3_ERR_UNSUPPORTED;  // beyond the fixed scratch
  m3_dims d = *dims;
  d.workspace = nullptr;
  d.workspace_bytes = 0;
  if (need > 0) {
    // Every call shares the array; the scan writes all of the scratch it reads,
    // so nothing needs clearing between calls.
    void* p = nullptr;
    const m3_status st = scratch_address(&p);
    if (st != M3_OK) return st;
    d.workspace = p;
    d.workspace_bytes = kStaticScratchBytes;
  }
  return m3_scan_fwd(x, dt, A, lambda, B, C, theta, &d, R, chunk, out, final_state, stream);
}

}  // extern "C"
