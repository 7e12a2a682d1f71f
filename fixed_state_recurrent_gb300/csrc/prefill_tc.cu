// prefill_tc.cu -- choice of the tensor-core prefill (bf16 inputs, dk = dv in
// {64, 128}), both in the chunked form of the page "线性注意力与SSM",
// section 3.  dk = 64: the two launches of prefill_prefix64.cu while what
// they read twice fits in L2, else the three launches of prefill_chunked64.cu
// (a running state per block of chunks); dk = 128: the three launches of
// prefill_chunked128.cu.
#include "prefill_tc_common.cuh"

namespace la {

bool prefill_tc_supported(const PrefillArgs& a) {
  return a.bf16 && a.dk == a.dv && (a.dk == 64 || a.dk == 128) && a.chunk == tcp::C && a.N > 0 &&
         tcp::get_encode() != nullptr;
}

size_t prefill_tc_workspace_bytes(int B, int H, int N, int d, int /*chunk*/) {
  if (d == 64)
    return prefill_prefix64_chosen(B, H, N) ? prefill_prefix64_workspace_bytes(B, H, N)
                                            : prefill_chunked64_workspace_bytes(B, H, N);
  return prefill_chunked128_workspace_bytes(B, H, N);
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream) {
  if (a.dk == 64)
    return prefill_prefix64_chosen(a.B, a.H, a.N) ? launch_prefill_prefix64(a, stream)
                                                  : launch_prefill_chunked64(a, stream);
  return launch_prefill_chunked128(a, stream);
}

}  // namespace la
