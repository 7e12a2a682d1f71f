// prefill_simt.cu -- CUDA-core causal prefill for any dk, dv <= 128 and for
// fp32 inputs (where bf16 tensor-core operands would miss a 1e-5 tolerance).
//
// Computes, per (batch, head), the recurrence of page "AIGC 基本功|线性、循环
// 与记忆架构-LinearMem", section 03, token by token in fp32:
//   S += phi(k_t) v_t^T;  z += phi(k_t);  o_t = phi(q_t)^T S / (phi(q_t)^T z + eps)
//
// One block per head.  The fp32 state lives in registers: the dv columns are
// split into groups of 4 and the dk rows over the remaining threads, so each
// thread owns a (rows x 4) slice of S and updates it with no communication.
// Tokens are staged TB at a time in shared memory (phi applied on the way in);
// per token each thread writes its partial numerators (over its rows) and, for
// column group 0, its partial denominators; one reduction per TB tokens then
// forms o.  Three block barriers per TB tokens.
//
// Variants (la_prefill_variant), same state machinery:
//   decay: S_t = alpha_t S_{t-1} + phi(k_t) v_t^T, z_t = alpha_t z_{t-1} + phi(k_t)
//     (the linear-attention recurrence with one scalar on the old state: page
//     "线性注意力与SSM", sections 3-4; the normalizer decays with the state);
//   read before write: o_t from S_{t-1}, z_{t-1} (LinearMem sections 03 and 09:
//     strictly past, the first read is 0);
//   non-causal: the state over all N tokens first, then every query reads it
//     (the linear-attention explainer, section 线性化核心).
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kTB = 8;         // tokens staged per round
constexpr int kMaxD = 128;
constexpr int kMaxRows = 16;   // rows of S per thread (dk <= 128, >= 8 row groups)

struct SimtShape {
  int G;  // column groups of 4
  int R;  // row groups
  int dvp;  // dv rounded up to a multiple of 4
};

__host__ __device__ inline SimtShape simt_shape(int dk, int dv) {
  SimtShape s;
  s.dvp = (dv + 3) & ~3;
  s.G = s.dvp / 4;
  s.R = kThreads / s.G;
  if (s.R > dk) s.R = dk;
  return s;
}

// MODE: 0 write then read, 1 read then write, 2 non-causal.  DECAY: alpha != NULL.
template <int MODE, bool DECAY>
__global__ void __launch_bounds__(kThreads)
prefill_simt_kernel(const void* __restrict__ q, const void* __restrict__ k,
                    const void* __restrict__ v, bool bf16, int N, int dk, int dv,
                    float eps, const float* __restrict__ alpha, const float* __restrict__ S0,
                    const float* __restrict__ z0, float* __restrict__ o,
                    float* __restrict__ S_N, float* __restrict__ z_N) {
  extern __shared__ float smem[];
  const SimtShape sh = simt_shape(dk, dv);
  float* fq = smem;                        // [kTB][kMaxD]
  float* fk = fq + kTB * kMaxD;            // [kTB][kMaxD]
  float* fv = fk + kTB * kMaxD;            // [kTB][kMaxD]
  float* part = fv + kTB * kMaxD;          // [kTB][R][dvp]
  float* dpart = part + kTB * sh.R * sh.dvp;  // [kTB][R]
  float* fa = dpart + kTB * sh.R;          // [kTB] decay of each staged token

  const int tid = threadIdx.x;
  const int g = tid % sh.G;        // column group
  const int rg = tid / sh.G;       // row group
  const bool active = rg < sh.R;
  const int col0 = 4 * g;
  const size_t head = blockIdx.x;

  // rows owned: rg, rg + R, rg + 2R, ...
  float S[kMaxRows][4];
  float z[kMaxRows];
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) {
    z[r] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) S[r][c] = 0.f;
  }
  if (active) {
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      const int i = rg + r * sh.R;
      if (i < dk) {
        if (S0) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (col0 + c < dv) S[r][c] = S0[(head * dk + i) * dv + col0 + c];
        }
        if (z0 && g == 0) z[r] = z0[head * dk + i];
      }
    }
  }

  if (MODE == 2) {
    // ---- non-causal: the state over all tokens first
    for (int t0 = 0; t0 < N; t0 += kTB) {
      for (int e = tid; e < kTB * kMaxD; e += kThreads) {
        const int t = e / kMaxD, i = e % kMaxD;
        const int tok = t0 + t;
        const bool in = tok < N;
        fk[e] = (in && i < dk) ? phi_f32(load_in(k, (head * N + tok) * dk + i, bf16)) : 0.f;
        fv[e] = (in && i < dv) ? load_in(v, (head * N + tok) * dv + i, bf16) : 0.f;
      }
      __syncthreads();
      if (active) {
        for (int t = 0; t < kTB; ++t) {
          const float4 vv = *reinterpret_cast<const float4*>(&fv[t * kMaxD + col0]);
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r) {
            const int i = rg + r * sh.R;
            if (i < dk) {
              const float a = fk[t * kMaxD + i];
              S[r][0] += a * vv.x;
              S[r][1] += a * vv.y;
              S[r][2] += a * vv.z;
              S[r][3] += a * vv.w;
              z[r] += a;
            }
          }
        }
      }
      __syncthreads();
    }
  }

  for (int t0 = 0; t0 < N; t0 += kTB) {
    // ---- stage kTB tokens, phi applied; rows past N are zero (no effect)
    if (DECAY && tid < kTB) fa[tid] = (t0 + tid < N) ? alpha[head * N + t0 + tid] : 1.f;
    for (int e = tid; e < kTB * kMaxD; e += kThreads) {
      const int t = e / kMaxD, i = e % kMaxD;
      const int tok = t0 + t;
      const bool in = tok < N;
      fq[e] = (in && i < dk) ? phi_f32(load_in(q, (head * N + tok) * dk + i, bf16)) : 0.f;
      fk[e] = (in && i < dk) ? phi_f32(load_in(k, (head * N + tok) * dk + i, bf16)) : 0.f;
      fv[e] = (in && i < dv) ? load_in(v, (head * N + tok) * dv + i, bf16) : 0.f;
    }
    __syncthreads();

    // ---- per thread: write, then read, token by token (or read, then
    // write; or, non-causal, read the full state)
    if (active) {
      for (int t = 0; t < kTB; ++t) {
        const float4 vv = *reinterpret_cast<const float4*>(&fv[t * kMaxD + col0]);
        const float at = DECAY ? fa[t] : 1.f;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        float dacc = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
          const int i = rg + r * sh.R;
          if (i < dk) {
            const float a = fk[t * kMaxD + i];
            const float b = fq[t * kMaxD + i];
            if (MODE == 1 || MODE == 2) {
              acc[0] += b * S[r][0];
              acc[1] += b * S[r][1];
              acc[2] += b * S[r][2];
              acc[3] += b * S[r][3];
              dacc += b * z[r];
            }
            if (MODE != 2) {
              if (DECAY) {
                S[r][0] = fmaf(at, S[r][0], a * vv.x);
                S[r][1] = fmaf(at, S[r][1], a * vv.y);
                S[r][2] = fmaf(at, S[r][2], a * vv.z);
                S[r][3] = fmaf(at, S[r][3], a * vv.w);
                z[r] = fmaf(at, z[r], a);
              } else {
                S[r][0] += a * vv.x;
                S[r][1] += a * vv.y;
                S[r][2] += a * vv.z;
                S[r][3] += a * vv.w;
                z[r] += a;
              }
            }
            if (MODE == 0) {
              acc[0] += b * S[r][0];
              acc[1] += b * S[r][1];
              acc[2] += b * S[r][2];
              acc[3] += b * S[r][3];
              dacc += b * z[r];
            }
          }
        }
        float* pp = &part[(t * sh.R + rg) * sh.dvp + col0];
        pp[0] = acc[0];
        pp[1] = acc[1];
        pp[2] = acc[2];
        pp[3] = acc[3];
        if (g == 0) dpart[t * sh.R + rg] = dacc;
      }
    }
    __syncthreads();

    // ---- reduce over row groups and normalize
    for (int e = tid; e < kTB * dv; e += kThreads) {
      const int t = e / dv, j = e % dv;
      const int tok = t0 + t;
      if (tok < N) {
        float num = 0.f, den = 0.f;
        for (int r = 0; r < sh.R; ++r) {
          num += part[(t * sh.R + r) * sh.dvp + j];
          den += dpart[t * sh.R + r];
        }
        o[(head * N + tok) * dv + j] = num / (den + eps);
      }
    }
    __syncthreads();
  }

  // ---- final state
  if (active) {
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      const int i = rg + r * sh.R;
      if (i < dk) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (col0 + c < dv) S_N[(head * dk + i) * dv + col0 + c] = S[r][c];
        if (g == 0) z_N[head * dk + i] = z[r];
      }
    }
  }
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream) {
  return launch_prefill_variant_simt(a, nullptr, 0, stream);
}

cudaError_t launch_prefill_variant_simt(const PrefillArgs& a, const float* alpha, int mode,
                                        cudaStream_t stream) {
  const SimtShape sh = simt_shape(a.dk, a.dv);
  // Every thread must own at most kMaxRows rows.
  if ((a.dk + sh.R - 1) / sh.R > kMaxRows) return cudaErrorInvalidValue;
  if (mode < 0 || mode > 2 || (mode == 2 && alpha)) return cudaErrorInvalidValue;
  const size_t smem =
      sizeof(float) * (3 * kTB * kMaxD + kTB * sh.R * sh.dvp + kTB * sh.R + kTB);
  const unsigned blocks = (unsigned)((size_t)a.B * a.H);
  auto go = [&](auto kern) -> cudaError_t {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    kern<<<blocks, kThreads, smem, stream>>>(a.q, a.k, a.v, a.bf16, a.N, a.dk, a.dv, a.eps, alpha,
                                             a.S0, a.z0, a.o, a.S_N, a.z_N);
    return cudaGetLastError();
  };
  if (mode == 2) return go(prefill_simt_kernel<2, false>);
  if (mode == 1) return alpha ? go(prefill_simt_kernel<1, true>) : go(prefill_simt_kernel<1, false>);
  return alpha ? go(prefill_simt_kernel<0, true>) : go(prefill_simt_kernel<0, false>);
}

}  // namespace la
