// la_internal.h -- declarations shared by the translation units of libla.so.
// Not part of the public ABI (that is include/la.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "la.h"

namespace la {

// Workspace header: the first 256 bytes of every prefill workspace.
//   status  sticky error bits set by kernels (kStatusTimeout); it must be zero
//           before the workspace's first use, and la_read_device_status
//           clears it.  Nothing else in a workspace is read before the call
//           that uses it has written it.
struct WsHeader {
  unsigned status;
  unsigned reserved[63];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusLayout = 2u;  // a kernel found its shared window misaligned and stopped

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  bool bf16;
  int B, H, N, dk, dv;
  float eps;
  const float* S0;
  const float* z0;
  float* o;
  float* S_N;
  float* z_N;
  int chunk;
  void* workspace;
  size_t ws_bytes;
  unsigned* status;  // where the tensor-core kernels record errors; NULL = the workspace header's word
  bool strict;       // read before write: token t reads the state before its own write (keys s < t)
};

// la_prefill's argument checks, path choice and launches, with the status
// word of the tensor-core kernels given explicitly (NULL: the workspace
// header's word, as la_prefill does).
la_status prefill_entry(const void* q, const void* k, const void* v, la_dtype in_dtype, int B,
                        int H, int N, int dk, int dv, float eps, const float* S0, const float* z0,
                        float* o, float* S_N, float* z_N, int chunk, void* workspace,
                        size_t ws_bytes, unsigned* status, cudaStream_t stream);

// CUDA-core prefill (any dk, dv <= 128; fp32 or bf16 inputs).  With a
// workspace of at least prefill_simt_workspace_bytes (nonzero when the heads'
// sequences are worth cutting into chunks) the chunks run in parallel (three
// launches); without one, one block walks each head.
size_t prefill_simt_workspace_bytes(int B, int H, int N, int dk, int dv);
cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream);
// The CUDA-core kernel's variants: alpha = per-token decay of (S, z) or NULL;
// mode 0 write-then-read, 1 read-then-write (strictly past), 2 non-causal
// (alpha must be NULL).
cudaError_t launch_prefill_variant_simt(const PrefillArgs& a, const float* alpha, int mode,
                                        cudaStream_t stream);

// Gradient of the causal prefill (backward_simt.cu): dq, dk, dv (and dS0, dz0
// if not NULL) given dO and dS_N, dz_N (NULL = zero); with p.workspace of at
// least backward_simt_workspace_bytes (no header) the heads' chunks run in
// parallel, else one block per head.
size_t backward_simt_workspace_bytes(int B, int H, int N, int dk, int dv);
cudaError_t launch_prefill_backward(const PrefillArgs& p, const float* dO, const float* dS_N,
                                    const float* dz_N, float* dq, float* dk, float* dv,
                                    float* dS0, float* dz0, cudaStream_t stream);
// The CUDA-core prefill's chunking (prefill_simt.cu) for about `blocks`
// blocks: the number of chunks per head (1: whole heads) and their length *L
// (a multiple of the 8-token stage); and its first two launches over NC
// chunks of L tokens, the state before every chunk into slots
// ([B H][NC][dk dv + dk], S row-major then z), S_N and z_N into the given
// buffers.
int simt_chunking(int BH, int N, int blocks, int* L);
cudaError_t launch_simt_entry_states(const PrefillArgs& a, int NC, int L, float* slots, float* S_N,
                                     float* z_N, cudaStream_t stream);
// The same gradient on the tensor cores for bf16 inputs at dk = dv = 64
// (backward_tc64.cu): a forward and a reverse sweep over 128-token chunks (it
// parks bf16 data in dv until the reverse sweep overwrites it); bounded-wait
// failures go to the library status word.
// With a.workspace of at least backward_tc64_workspace_bytes the pieces of the
// d = 64 split run over every SM (the prefill's aggregate and scan for the
// entry states, forward sweeps, a reverse scan of the gradient state, reverse
// sweeps); without one, one block per head.
bool backward_tc64_supported(const PrefillArgs& a);
size_t backward_tc64_workspace_bytes(int B, int H, int N);
cudaError_t launch_backward_tc64(const PrefillArgs& a, const float* dO, const float* dS_N,
                                 const float* dz_N, float* dq, float* dk, float* dv, float* dS0,
                                 float* dz0, cudaStream_t stream);

// Tensor-core chunked prefill for dk = dv = 64: aggregate, scan and output
// launches (prefill_chunked64.cu).  The workspace size depends on the SM count
// of the current device.
size_t prefill_chunked64_workspace_bytes(int B, int H, int N);
cudaError_t launch_prefill_chunked64(const PrefillArgs& a, cudaStream_t stream);
// The decayed write-then-read form of the same products (bf16, dk = dv = 64),
// one block per head; alpha: [B][H][N] per-token decay.  Needs no workspace.
// With a.workspace of at least prefill_decay64_workspace_bytes the heads are
// split over every SM (aggregate, scan, output), otherwise one block per head.
bool prefill_decay64_supported(const PrefillArgs& a);
// The entry state of every piece of the d = 64 split (the split of
// prefill_tc_common.cuh's make_split over the current device's SMs) into E,
// slot layout [BH * MPH][64 * 64 + 64]; agg (the same size), S_N and z_N
// (B * H states) are scratch.
cudaError_t launch_prefill_entry_states64(const PrefillArgs& a, float* agg, float* E, float* S_N,
                                          float* z_N, unsigned* status, cudaStream_t stream);
size_t prefill_decay64_workspace_bytes(int B, int H, int N);
cudaError_t launch_prefill_decay64(const PrefillArgs& a, const float* alpha, cudaStream_t stream);

// Two-launch form for dk = dv = 64 (prefill_prefix64.cu): per-chunk prefix
// tiles and piece totals, then the outputs.  Chosen by the tensor-core
// dispatch for calls small enough that what the second launch reads again
// stays in L2.
bool prefill_prefix64_chosen(int B, int H, int N);
size_t prefill_prefix64_workspace_bytes(int B, int H, int N);
cudaError_t launch_prefill_prefix64(const PrefillArgs& a, cudaStream_t stream);
// The same two launches with every buffer given: R piece totals ([BH * MPH]
// slots of 64 * 64 + 64 floats, MPH of prefill_tc_common.cuh's make_split over
// the current device's SMs), P prefix tiles ([BH * ceil(N / 128)][66][64]
// bf16), phik ([BH][N][64] bf16), o ([BH][N][64]: fp32, or bf16 when den is
// given), den (NULL, or [BH][N] fp32: den_t = phi(q_t)^T z_t + eps), E (with
// den: [G][66][64] bf16, G the split's block count: the entry-state tile of
// each block whose first piece has one, in the prefix tiles' format), S_N and
// z_N (B * H final states), status (where bounded waits that give up are
// recorded); force_wait: the test hook of the output kernel.  q, k, v, S0,
// z0, N, eps come from a.
struct Prefix64Buffers {
  float* R;
  uint8_t* P;
  __nv_bfloat16* phik;
  void* o;
  float* den;
  uint8_t* E;
  float* S_N;
  float* z_N;
  unsigned* status;
  int force_wait;
  int strict;  // read before write (keys s < t inside a chunk); not with den
};
cudaError_t launch_prefix64_pair(const PrefillArgs& a, const Prefix64Buffers& b, cudaStream_t stream);
// Read-before-write order (la_prefill_variant's LA_MODE_READ_BEFORE_WRITE, no
// decay) in the same two launches, for the calls prefill_prefix64_chosen
// takes; a.workspace of at least prefill_prefix64_workspace_bytes (no header;
// bounded-wait failures go to the library status word).
cudaError_t launch_prefill_rbw64(const PrefillArgs& a, cudaStream_t stream);
// The first of those launches alone, for its piece totals R only (with S0 in
// a piece that starts its head; neither P nor phik is written, but their maps
// are still made over the buffers given).
cudaError_t launch_prefix64_totals(const PrefillArgs& a, const Prefix64Buffers& b, cudaStream_t stream);
// Non-causal order (la_prefill_variant's LA_MODE_NONCAUSAL) at bf16,
// dk = dv = 64, for the calls prefill_prefix64_chosen takes: the piece totals,
// then every query reads its head's final state (prefill_noncausal.cu).
// a.workspace of at least prefill_nc64_workspace_bytes (no header);
// bounded-wait failures go to the library status word.
size_t prefill_nc64_workspace_bytes(int B, int H, int N);
cudaError_t launch_prefill_nc64(const PrefillArgs& a, cudaStream_t stream);
// The same order at bf16, dk = dv = 64 or 128, for calls of any length: the
// totals from the aggregate kernel of the three-launch prefill, then the
// reads.  a.workspace of at least prefill_nc_workspace_bytes (no header);
// bounded-wait failures go to the library status word.
size_t prefill_nc_workspace_bytes(int B, int H, int N, int d);
cudaError_t launch_prefill_nc(const PrefillArgs& a, cudaStream_t stream);
// The aggregate launch of the three-launch prefill alone: each piece's total
// (without S0) into agg, in slots of make_split(B H, N, SMs); bounded-wait
// failures go to `status`.  A programmatic dependent of what precedes it.
size_t aggregate64_totals_bytes(int B, int H, int N);
cudaError_t launch_aggregate64_totals(const PrefillArgs& a, float* agg, unsigned* status, cudaStream_t stream);
size_t aggregate128_totals_bytes(int B, int H, int N);
// The decayed write-then-read form at bf16, dk = dv = 128 (alpha: [B][H][N]):
// the three launches of prefill_chunked128.cu with decay weights (decayed
// piece totals and decays, the scan E' = Gamma E + R, the outputs).
// a.workspace of at least prefill_decay128_workspace_bytes (no header);
// bounded-wait failures go to the library status word.
size_t prefill_decay128_workspace_bytes(int B, int H, int N);
cudaError_t launch_prefill_decay128(const PrefillArgs& a, const float* alpha, cudaStream_t stream);
cudaError_t launch_aggregate128_totals(const PrefillArgs& a, float* agg, unsigned* status, cudaStream_t stream);
// The decayed write-then-read form (alpha: [B][H][N]) in the same two launches,
// for the calls prefill_prefix64_chosen takes: a.workspace of at least
// prefill_prefix64_decay_workspace_bytes (no header); bounded-wait failures go
// to the library status word.
size_t prefill_prefix64_decay_workspace_bytes(int B, int H, int N);
cudaError_t launch_prefill_prefix64_decay(const PrefillArgs& a, const float* alpha, cudaStream_t stream);

// The gradient of the prefill for bf16 at dk = dv = 64, chunk-parallel in four
// launches (backward_prefix64.cu): the two launches above (o and den into the
// workspace), the gradient-state tiles, then dq, dk, dv.  For the calls that
// prefill_prefix64_chosen takes; bounded-wait failures go to the library
// status word.
size_t backward_prefix64_workspace_bytes(int B, int H, int N);
cudaError_t launch_backward_prefix64(const PrefillArgs& a, const float* dO, const float* dS_N,
                                     const float* dz_N, float* dq, float* dk, float* dv, float* dS0,
                                     float* dz0, cudaStream_t stream);

// The same three launches for dk = dv = 128 (prefill_chunked128.cu).
size_t prefill_chunked128_workspace_bytes(int B, int H, int N);
cudaError_t launch_prefill_chunked128(const PrefillArgs& a, cudaStream_t stream);

// Tensor-core chunked prefill (bf16, dk = dv in {64, 128}).
bool prefill_tc_supported(const PrefillArgs& a);
size_t prefill_tc_workspace_bytes(int B, int H, int N, int d, int chunk);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream);

cudaError_t launch_decode_step(const void* q, const void* k, const void* v,
                               bool bf16, int B, int H, int dk, int dv,
                               float eps, float* S, float* z, float* o,
                               cudaStream_t stream);

// Tensor-core chunked delta rule (bf16, dk = dv = 64, 96 or 128;
// delta_chunked128.cu).
bool delta_chunked_supported(bool bf16, int dk, int dv);
// alpha: per-token forgetting of the gated form, or NULL; d = dk = dv.
cudaError_t launch_delta_chunked(const void* k, const void* v, const float* beta, const float* alpha,
                                 int B, int H, int N, int d, const float* S0, float* reads, float* S_N,
                                 cudaStream_t stream);
// The status word of the kernels whose calls take no workspace (the chunked
// delta kernels, the decayed tensor-core prefill): its device address, and
// reading it (returns and clears it; current device).
cudaError_t library_status_word(unsigned** out);
cudaError_t delta_status_take(unsigned* out);

// alpha: per-token forgetting of the gated delta rule, or NULL (plain rule).
cudaError_t launch_delta_prefill(const void* k, const void* v, bool bf16,
                                 const float* beta, const float* alpha, int B, int H, int N,
                                 int dk, int dv, const float* S0, float* reads,
                                 float* S_N, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Device helpers shared by the CUDA-core kernels.

// ELU+1 feature map, full-precision expf.  Page "AIGC 基本功|线性、循环与记忆
// 架构-LinearMem", section 03: phi(u) = u + 1 for u > 0, exp(u) otherwise.
__device__ __forceinline__ float phi_f32(float u) {
  return u > 0.f ? u + 1.f : expf(u);
}

// Element e of an input tensor stored as fp32 or bf16, widened to fp32.
__device__ __forceinline__ float load_in(const void* p, size_t e, bool bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[e]);
  return reinterpret_cast<const float*>(p)[e];
}

}  // namespace la
