// prefill_tc.cu -- tensor-core chunked prefill (placeholder until the tcgen05
// kernel lands: every request goes to the CUDA-core path).
#include "la_internal.h"

namespace la {

bool prefill_tc_supported(const PrefillArgs&) { return false; }

size_t prefill_tc_workspace_bytes(int, int, int, int, int) { return 0; }

cudaError_t launch_prefill_tc(const PrefillArgs&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace la
