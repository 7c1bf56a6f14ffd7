// Tensor-core (tcgen05) chunked prefill: not yet enabled in this build.
#include "launch.h"

namespace m3 {

bool scan_tc_supported(int64_t, int64_t, int, int) { return false; }

cudaError_t launch_scan_tc(const ScanArgs&, unsigned int*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace m3
