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

#include <atomic>
#include <mutex>

namespace {

// 16 MiB of scratch per device: enough for la_prefill's workspace at
// dk = dv = 64 up to e.g. 16 heads of 4096 tokens (and, past 2048 chunks of
// 128 tokens, where only each piece's state is kept, for a few hundred heads
// of any length), at dk = dv = 128 up to e.g. 4 heads of 2048 tokens.
constexpr size_t kScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_la_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// Per device: the device address of g_la_scratch (its host-side name is only
// a stand-in) and of the library status word, looked up once with that device
// current.  Published with release order after both are known, so a thread
// that sees the scratch address also sees the status address.
std::atomic<void*> g_scratch_ptr[kMaxDevices];
unsigned* g_status_ptr[kMaxDevices];
std::mutex g_setup_mutex;

// The scratch needs no initialisation: the kernels write every part of it
// before reading it, and their error bits go to the library status word, not
// into the scratch.  So the set-up issues no device work at all.
la_status scratch_for_current_device(void** scratch, unsigned** status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LA_ERR_UNSUPPORTED;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
      unsigned* st = nullptr;
      if (cudaGetSymbolAddress(&p, g_la_scratch) != cudaSuccess || !p) return LA_ERR_CUDA;
      if (la::library_status_word(&st) != cudaSuccess || !st) return LA_ERR_CUDA;
      g_status_ptr[dev] = st;
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *scratch = p;
  *status = g_status_ptr[dev];
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
  unsigned* status = nullptr;
  const la_status st = scratch_for_current_device(&scratch, &status);
  if (st != LA_OK) return st;
  return la::prefill_entry(q, k, v, in_dtype, B, H, N, dk, dv, eps, S0, z0, o, S_N, z_N, chunk,
                           scratch, kScratchBytes, status, stream);
}
