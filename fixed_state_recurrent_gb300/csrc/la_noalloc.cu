// la_noalloc.cu -- la_prefill_noalloc: la_prefill for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or any allocator: code running while a
// CUDA graph is being captured, plugins of inference servers that only hand
// out input and output buffers, or hosts whose memory pools are owned by
// another runtime.  la_prefill needs a caller-provided workspace; this entry
// point instead uses one fixed scratch array that lives in this library's own
// device image (every GPU that loads the library holds it until the process
// exits).  Inputs and outputs are still the caller's.
#include "la.h"
#include "la_internal.h"

namespace {

// 16 MiB of scratch per device: enough for la_prefill's workspace at
// dk = dv = 64 up to e.g. 8 heads of 4096 tokens, at dk = dv = 128 up to e.g.
// 4 heads of 2048 tokens.
constexpr size_t kScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_la_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];  // device address of g_la_scratch, per device

// One-time set-up on the current device: look up the device address of the
// scratch array (its host-side name is only a stand-in) and zero it, since
// la_prefill expects a zero-filled workspace on first use.
la_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LA_ERR_UNSUPPORTED;
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_la_scratch) != cudaSuccess || !ptr) return LA_ERR_CUDA;
    if (cudaMemset(ptr, 0, kScratchBytes) != cudaSuccess) return LA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return LA_OK;
}

}  // namespace

extern "C" la_status la_prefill_noalloc(const void* q, const void* k, const void* v,
                                        la_dtype in_dtype, int B, int H, int N, int dk, int dv,
                                        float eps, const float* S0, const float* z0, float* o,
                                        float* S_N, float* z_N, int chunk, cudaStream_t stream) {
  const size_t need = la_prefill_workspace_bytes(B, H, N, dk, dv, in_dtype, chunk);
  if (need == 0 || need > kScratchBytes) return LA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const la_status st = scratch_for_current_device(&scratch);
  if (st != LA_OK) return st;
  return la_prefill(q, k, v, in_dtype, B, H, N, dk, dv, eps, S0, z0, o, S_N, z_N, chunk,
                    scratch, kScratchBytes, stream);
}
