// delta.cu -- the delta-rule fast-weight memory, token by token in fp32.
//
// Page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03 "从累加改成纠错",
// and page "sequence-models" practice notes, "Delta-rule fast weight": for each
// token the memory is first read with the key, read_t = k_t^T S_{t-1}, and
// then corrected, S_t = S_{t-1} + beta_t k_t (v_t - read_t)^T.
//
// Column j of S only ever meets column j (read_j = sum_i k_i S_ij, and the
// update of S_ij uses only read_j), so the columns are independent
// recurrences.  One block per head; column j is owned by P lanes of one warp,
// lane p holding rows [p*rows, (p+1)*rows) in registers.  Per token a lane
// loads its slice of k_t from shared memory (128-bit loads; the slices of the
// P lanes sit in different banks), forms its partial dot product, the P lanes
// combine it with xor shuffles, and every lane applies the rank-1 correction
// to its rows.  Keys, values and beta are staged TB tokens at a time; the next
// stage's global loads are issued before the current stage is consumed.  The
// work is 4 dk dv flops per token of fp32 FMA: this path is bound by the FP32
// pipe, not by HBM.
//
// Gated form (same page, section 03, the forgetting factor alpha_t, and its
// appendix delta_step): the old state decays first, D = alpha_t S_{t-1}; the read is
// the prediction from D, k_t^T D = alpha_t (k_t^T S_{t-1}); the correction is
// written on top of D: S_t = D + beta_t k_t (v_t - k_t^T D)^T.  alpha = NULL
// is the plain rule above.
#include "la_internal.h"

namespace la {
namespace {

constexpr int kTB = 16;      // tokens staged per round
constexpr int kMaxD = 128;
constexpr int kPad = 36;     // words per lane slice (32 rows + 4 words of bank skew)
constexpr int kRP = 32;      // max rows per lane
constexpr int kThreads = 512;  // dv * P <= 512; lanes past dv * P only stage

template <int P, bool GATED>
__global__ void __launch_bounds__(kThreads)
delta_kernel(const void* __restrict__ kin, const void* __restrict__ vin,
             bool bf16, const float* __restrict__ beta, const float* __restrict__ alpha,
             int N, int dk, int dv, const float* __restrict__ S0, float* __restrict__ reads,
             float* __restrict__ S_N) {
  __shared__ __align__(16) float ks[kTB][4 * kPad];
  __shared__ float vs[kTB][kMaxD];
  __shared__ float bs[kTB];
  __shared__ float as[kTB];

  const int tid = threadIdx.x;
  const int j = tid / P;      // column
  const int p = tid % P;      // slice of the rows
  const size_t head = blockIdx.x;
  const int rows = (dk + P - 1) / P;
  const int r0 = p * rows;
  const bool active = j < dv;

  float S[kRP];
#pragma unroll
  for (int r = 0; r < kRP; ++r) S[r] = 0.f;
  if (active && S0) {
#pragma unroll
    for (int r = 0; r < kRP; ++r)
      if (r < rows && r0 + r < dk) S[r] = S0[(head * dk + r0 + r) * dv + j];
  }

  // Staging: element e of a stage is token e / kMaxD, feature e % kMaxD; each
  // thread owns elements tid + u * kThreads in every stage.
  constexpr int kPer = kTB * kMaxD / kThreads;
  float kreg[kPer], vreg[kPer];
  auto fetch = [&](int t0) {
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = tid + u * kThreads;
      const int t = e / kMaxD, i = e % kMaxD;
      const int tok = t0 + t;
      kreg[u] = (tok < N && i < dk) ? load_in(kin, (head * N + tok) * dk + i, bf16) : 0.f;
      vreg[u] = (tok < N && i < dv) ? load_in(vin, (head * N + tok) * dv + i, bf16) : 0.f;
    }
  };
  float breg = 0.f, areg = 1.f;
  if (N > 0) {
    fetch(0);
    if (tid < kTB) breg = tid < N ? beta[head * N + tid] : 0.f;
    if (GATED && tid < kTB) areg = tid < N ? alpha[head * N + tid] : 1.f;
  }
  // words of the key slices that no feature maps to stay zero
  for (int e = tid; e < kTB * 4 * kPad; e += kThreads) {
    const int t = e / (4 * kPad), w = e % (4 * kPad);
    const int q = w / kPad, r = w % kPad;
    if (r >= rows || q * rows + r >= dk) ks[t][w] = 0.f;
  }

  for (int t0 = 0; t0 < N; t0 += kTB) {
    __syncthreads();  // the previous stage has been consumed
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = tid + u * kThreads;
      const int t = e / kMaxD, i = e % kMaxD;
      vs[t][i] = vreg[u];
      // feature i belongs to lane slice i / rows, at position i % rows
      if (i < dk) ks[t][(i / rows) * kPad + (i % rows)] = kreg[u];
    }
    if (tid < kTB) bs[tid] = breg;
    if (GATED && tid < kTB) as[tid] = areg;
    __syncthreads();
    // prefetch the next stage while this one is consumed
    if (t0 + kTB < N) {
      fetch(t0 + kTB);
      if (tid < kTB) breg = (t0 + kTB + tid < N) ? beta[head * N + t0 + kTB + tid] : 0.f;
      if (GATED && tid < kTB) areg = (t0 + kTB + tid < N) ? alpha[head * N + t0 + kTB + tid] : 1.f;
    }

    const int nt = min(kTB, N - t0);
    for (int t = 0; t < nt; ++t) {
      float kr[kRP];
      const float4* ksrc = reinterpret_cast<const float4*>(&ks[t][p * kPad]);
#pragma unroll
      for (int r = 0; r < kRP; r += 4) {
        const float4 x = ksrc[r / 4];
        kr[r] = x.x; kr[r + 1] = x.y; kr[r + 2] = x.z; kr[r + 3] = x.w;
      }
      // read before write
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int r = 0; r < kRP; r += 4) {
        a0 += kr[r] * S[r];
        a1 += kr[r + 1] * S[r + 1];
        a2 += kr[r + 2] * S[r + 2];
        a3 += kr[r + 3] * S[r + 3];
      }
      float part = (a0 + a1) + (a2 + a3);
#pragma unroll
      for (int off = 1; off < P; off <<= 1)
        part += __shfl_xor_sync(0xffffffffu, part, off);
      if (active) {
        if (GATED) {
          const float at = as[t];
          part *= at;  // the prediction from the decayed state
          if (p == 0) reads[(head * N + t0 + t) * dv + j] = part;
          const float e = bs[t] * (vs[t][j] - part);
#pragma unroll
          for (int r = 0; r < kRP; ++r) S[r] = fmaf(at, S[r], kr[r] * e);
        } else {
          if (p == 0) reads[(head * N + t0 + t) * dv + j] = part;
          const float e = bs[t] * (vs[t][j] - part);
#pragma unroll
          for (int r = 0; r < kRP; ++r) S[r] += kr[r] * e;
        }
      }
    }
  }

  if (active) {
#pragma unroll
    for (int r = 0; r < kRP; ++r)
      if (r < rows && r0 + r < dk) S_N[(head * dk + r0 + r) * dv + j] = S[r];
  }
}

}  // namespace

cudaError_t launch_delta_prefill(const void* k, const void* v, bool bf16,
                                 const float* beta, const float* alpha, int B, int H, int N,
                                 int dk, int dv, const float* S0, float* reads,
                                 float* S_N, cudaStream_t stream) {
  // bf16 keys and values at dk = dv = 128, gated or not: the chunkwise
  // tensor-core form (delta_chunked128.cu); everything else runs token by
  // token here.
  if (delta_chunked_supported(bf16, dk, dv))
    return launch_delta_chunked(k, v, beta, alpha, B, H, N, dk, S0, reads, S_N, stream);
  const unsigned blocks = (unsigned)((size_t)B * H);
  // P lanes per column (a power of two, at most 4): enough that a lane holds
  // at most 32 rows.  rows = ceil(dk / P) <= 32 and P * kPad <= 4 * kPad, so
  // every shared-memory index is in range; a lane's unused words are zero.
  int P = 1;
  while (P * 32 < dk) P <<= 1;
  const int threads = kThreads;
#define LA_DELTA_LAUNCH(PP, G)                                                              \
  delta_kernel<PP, G><<<blocks, threads, 0, stream>>>(k, v, bf16, beta, alpha, N, dk, dv, S0, \
                                                     reads, S_N)
  if (alpha) {
    switch (P) {
      case 1: LA_DELTA_LAUNCH(1, true); break;
      case 2: LA_DELTA_LAUNCH(2, true); break;
      default: LA_DELTA_LAUNCH(4, true); break;
    }
  } else {
    switch (P) {
      case 1: LA_DELTA_LAUNCH(1, false); break;
      case 2: LA_DELTA_LAUNCH(2, false); break;
      default: LA_DELTA_LAUNCH(4, false); break;
    }
  }
#undef LA_DELTA_LAUNCH
  return cudaGetLastError();
}

}  // namespace la
