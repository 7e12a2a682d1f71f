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
// each holding dk/P rows in registers.  Per token a lane forms its partial dot
// product, the P lanes combine it with xor shuffles, and every lane applies
// the rank-1 correction to its rows.  Keys, values and beta are staged TB
// tokens at a time in shared memory; the reads go out as one coalesced row per
// token.  The work is 4 dk dv flops per token of dependent fp32 FMA, so this
// path is bound by the FP32 pipe, not by HBM.
#include "la_internal.h"

namespace la {
namespace {

constexpr int kTB = 16;      // tokens staged per round
constexpr int kMaxD = 128;

template <int P>
__global__ void __launch_bounds__(512)
delta_kernel(const void* __restrict__ kin, const void* __restrict__ vin,
             bool bf16, const float* __restrict__ beta, int N, int dk, int dv,
             const float* __restrict__ S0, float* __restrict__ reads,
             float* __restrict__ S_N) {
  constexpr int RP = 32;  // max rows per lane: P is chosen so that ceil(dk / P) <= 32
  __shared__ float ks[kTB][kMaxD];
  __shared__ float vs[kTB][kMaxD];
  __shared__ float bs[kTB];

  const int tid = threadIdx.x;
  const int j = tid / P;      // column
  const int p = tid % P;      // part of the rows
  const size_t head = blockIdx.x;
  const int rows = (dk + P - 1) / P;
  const int r0 = p * rows;
  const bool active = j < dv;

  float S[RP];
#pragma unroll
  for (int r = 0; r < RP; ++r) S[r] = 0.f;
  if (active && S0) {
#pragma unroll
    for (int r = 0; r < RP; ++r)
      if (r < rows && r0 + r < dk) S[r] = S0[(head * dk + r0 + r) * dv + j];
  }

  for (int t0 = 0; t0 < N; t0 += kTB) {
    __syncthreads();  // previous round's readers are done with the stage
    for (int e = tid; e < kTB * kMaxD; e += blockDim.x) {
      const int t = e / kMaxD, i = e % kMaxD;
      const int tok = t0 + t;
      const bool in = tok < N;
      ks[t][i] = (in && i < dk) ? load_in(kin, (head * N + tok) * dk + i, bf16) : 0.f;
      vs[t][i] = (in && i < dv) ? load_in(vin, (head * N + tok) * dv + i, bf16) : 0.f;
    }
    if (tid < kTB) bs[tid] = (t0 + tid < N) ? beta[head * N + t0 + tid] : 0.f;
    __syncthreads();

    const int nt = min(kTB, N - t0);
    for (int t = 0; t < nt; ++t) {
      // read before write
      float part = 0.f;
#pragma unroll
      for (int r = 0; r < RP; ++r)
        if (r < rows) part += ks[t][r0 + r] * S[r];
#pragma unroll
      for (int off = 1; off < P; off <<= 1)
        part += __shfl_xor_sync(0xffffffffu, part, off);
      if (active) {
        if (p == 0) reads[(head * N + t0 + t) * dv + j] = part;
        const float e = bs[t] * (vs[t][j] - part);
#pragma unroll
        for (int r = 0; r < RP; ++r)
          if (r < rows) S[r] += ks[t][r0 + r] * e;
      }
    }
  }

  if (active) {
#pragma unroll
    for (int r = 0; r < RP; ++r)
      if (r < rows && r0 + r < dk) S_N[(head * dk + r0 + r) * dv + j] = S[r];
  }
}

}  // namespace

cudaError_t launch_delta_prefill(const void* k, const void* v, bool bf16,
                                 const float* beta, int B, int H, int N,
                                 int dk, int dv, const float* S0, float* reads,
                                 float* S_N, cudaStream_t stream) {
  const unsigned blocks = (unsigned)((size_t)B * H);
  // P lanes per column: enough that a lane holds at most 32 rows.
  int P = 1;
  while (P * 32 < dk) P <<= 1;
  const int threads = ((dv * P + 31) / 32) * 32;
  // A lane's rows are [p * rows, (p + 1) * rows) with rows = ceil(dk / P) <= 32;
  // since P is a power of two <= 4 that divides 128, P * rows <= 128, so every
  // shared-memory index stays below kMaxD.  Rows past dk read staged zeros and
  // are never stored.
  switch (P) {
    case 1: delta_kernel<1><<<blocks, threads, 0, stream>>>(k, v, bf16, beta, N, dk, dv, S0, reads, S_N); break;
    case 2: delta_kernel<2><<<blocks, threads, 0, stream>>>(k, v, bf16, beta, N, dk, dv, S0, reads, S_N); break;
    default: delta_kernel<4><<<blocks, threads, 0, stream>>>(k, v, bf16, beta, N, dk, dv, S0, reads, S_N); break;
  }
  return cudaGetLastError();
}

}  // namespace la
