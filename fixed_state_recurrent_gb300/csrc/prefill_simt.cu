// prefill_simt.cu -- CUDA-core causal prefill for any dk, dv <= 128 and for
// fp32 inputs (where bf16 tensor-core operands would miss a 1e-5 tolerance).
//
// Computes, per (batch, head), the recurrence of page "AIGC 基本功|线性、循环
// 与记忆架构-LinearMem", section 03, token by token in fp32:
//   S += phi(k_t) v_t^T;  z += phi(k_t);  o_t = phi(q_t)^T S / (phi(q_t)^T z + eps)
//
// One block walks a run of tokens of one head.  The fp32 state lives in
// registers: the dv columns are split into groups of 4 and the dk rows over
// the remaining threads, so each thread owns a (rows x 4) slice of S and
// updates it with no communication.  Tokens are staged TB at a time in shared
// memory (phi applied on the way in); per token each thread writes its partial
// numerators (over its rows) and, for column group 0, its partial
// denominators; one reduction per TB tokens then forms o.  Three block
// barriers per TB tokens.
//
// With a workspace the heads' sequences are cut into NC chunks (chunkwise
// evaluation, page "线性注意力与SSM", section 3: chunks hand over only the
// state) and three launches run them in parallel:
//   PASS 1: each chunk's increment from a zero state (with a decay, the
//     increment weighted by the decay to the chunk's end, and the chunk's
//     total decay);
//   scan: per head and state element, the state before every chunk (left
//     fold from S0, in chunk order), in place of the increments, and S_N, z_N;
//   PASS 2: each chunk's outputs, the walk above started from the state
//     before the chunk (non-causal: from the final state, read only).
// Without one (or for one chunk), PASS 0 walks each whole head in one block.
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

// The chunking of the three-launch form: NC chunks of L tokens per head, and
// per (head, chunk) a slot of dk dv + dk floats (S row-major, then z) plus the
// chunk's total decay.
struct SimtChunks {
  int NC, L;
  float* slots;  // [BH][NC][dk dv + dk]
  float* gam;    // [BH][NC]
};

// MODE: 0 write then read, 1 read then write, 2 non-causal.  DECAY: alpha != NULL.
// PASS: 0 whole heads, 1 chunk increments, 2 chunk outputs.
template <int MODE, bool DECAY, int PASS>
__global__ void __launch_bounds__(kThreads)
prefill_simt_kernel(const void* __restrict__ q, const void* __restrict__ k,
                    const void* __restrict__ v, bool bf16, int N, int dk, int dv,
                    float eps, const float* __restrict__ alpha, const float* __restrict__ S0,
                    const float* __restrict__ z0, float* __restrict__ o,
                    float* __restrict__ S_N, float* __restrict__ z_N, const SimtChunks ck) {
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
  const size_t head = PASS == 0 ? blockIdx.x : blockIdx.y;
  const int chunk = PASS == 0 ? 0 : blockIdx.x;
  const int tb = PASS == 0 ? 0 : chunk * ck.L;                     // this block's tokens: [tb, te)
  const int te = PASS == 0 ? N : min(N, tb + ck.L);
  const size_t sz = (size_t)dk * dv + dk;
  float* slot = PASS == 0 ? nullptr : ck.slots + (head * ck.NC + chunk) * sz;

  // rows owned: rg, rg + R, rg + 2R, ...  The walk starts from S0, z0 (whole
  // heads), zero (increments), or the state before the chunk (outputs; the
  // final state for the non-causal read)
  const float* Si = PASS == 0 ? S0 : PASS == 1 ? nullptr : (MODE == 2 ? S_N + head * dk * dv : slot);
  const float* zi = PASS == 0 ? z0 : PASS == 1 ? nullptr : (MODE == 2 ? z_N + head * dk : slot + dk * dv);
  const size_t sh0 = PASS == 2 ? 0 : head * dk * dv, zh0 = PASS == 2 ? 0 : head * dk;
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
        if (Si) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (col0 + c < dv) S[r][c] = Si[sh0 + (size_t)i * dv + col0 + c];
        }
        if (zi && g == 0) z[r] = zi[zh0 + i];
      }
    }
  }

  if (MODE == 2 && PASS == 0) {
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

  float gam = 1.f;  // increments: the chunk's total decay (thread 0)
  for (int t0 = tb; t0 < te; t0 += kTB) {
    // ---- stage kTB tokens, phi applied; rows past the run are zero (no
    // effect); all loads of a thread first
    if (DECAY && tid < kTB) fa[tid] = (t0 + tid < te) ? alpha[head * N + t0 + tid] : 1.f;
    constexpr int kPer = kTB * kMaxD / kThreads;
    float lq[kPer], lk[kPer], lv[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = tid + u * kThreads, t = e / kMaxD, i = e % kMaxD;
      const int tok = t0 + t;
      const bool in = tok < te;
      lq[u] = (PASS != 1 && in && i < dk) ? load_in(q, (head * N + tok) * dk + i, bf16) : 0.f;
      lk[u] = (in && i < dk) ? load_in(k, (head * N + tok) * dk + i, bf16) : 0.f;
      lv[u] = (in && i < dv) ? load_in(v, (head * N + tok) * dv + i, bf16) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = tid + u * kThreads, t = e / kMaxD, i = e % kMaxD;
      const bool in = t0 + t < te;
      fq[e] = (PASS != 1 && in && i < dk) ? phi_f32(lq[u]) : 0.f;
      fk[e] = (in && i < dk) ? phi_f32(lk[u]) : 0.f;
      fv[e] = lv[u];
    }
    __syncthreads();
    if (PASS == 1) {
      // ---- increments: the state updates alone
      if (active) {
        for (int t = 0; t < kTB; ++t) {
          const float4 vv = *reinterpret_cast<const float4*>(&fv[t * kMaxD + col0]);
          const float at = DECAY ? fa[t] : 1.f;
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r) {
            const int i = rg + r * sh.R;
            if (i < dk) {
              const float a = fk[t * kMaxD + i];
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
          }
        }
      }
      if (DECAY && tid == 0)
        for (int t = 0; t < kTB; ++t) gam *= fa[t];
      __syncthreads();
      continue;
    }

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
      if (tok < te) {
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

  // ---- final state (whole heads) or the chunk's increment (chunks)
  if (PASS != 2 && active) {
    float* Sd = PASS == 0 ? S_N + head * dk * dv : slot;
    float* zd = PASS == 0 ? z_N + head * dk : slot + dk * dv;
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      const int i = rg + r * sh.R;
      if (i < dk) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (col0 + c < dv) Sd[(size_t)i * dv + col0 + c] = S[r][c];
        if (g == 0) zd[i] = z[r];
      }
    }
  }
  if (PASS == 1 && DECAY && tid == 0) ck.gam[head * ck.NC + chunk] = gam;
}

// Per head and state element (S row-major, then z): the state before every
// chunk, in place of the chunk's increment, as the left fold from S0, z0 in
// chunk order (E' = gamma E + increment with a decay), and the final state.
template <bool DECAY>
__global__ void __launch_bounds__(kThreads)
simt_scan_kernel(int dk, int dv, const float* __restrict__ S0, const float* __restrict__ z0,
                 float* __restrict__ S_N, float* __restrict__ z_N, const SimtChunks ck) {
  const size_t head = blockIdx.y;
  const int e = blockIdx.x * kThreads + threadIdx.x;
  const int nS = dk * dv;
  if (e >= nS + dk) return;
  float acc = e < nS ? (S0 ? S0[head * nS + e] : 0.f) : (z0 ? z0[head * dk + e - nS] : 0.f);
  const size_t sz = (size_t)nS + dk;
  float* col = ck.slots + head * ck.NC * sz + e;
  for (int c = 0; c < ck.NC; ++c) {
    const float d = col[c * sz];
    col[c * sz] = acc;
    acc = DECAY ? fmaf(ck.gam[head * ck.NC + c], acc, d) : acc + d;
  }
  if (e < nS) S_N[head * nS + e] = acc;
  else z_N[head * dk + e - nS] = acc;
}

// Chunks per head of the three-launch form: enough blocks for about two per
// SM of a 152-SM GPU, at least kTB tokens per chunk, at most 64 chunks; 1 =
// whole heads.
int simt_chunks(int BH, int N) {
  const int by_len = (N + kTB - 1) / kTB;
  const int by_sm = (2 * 152 + BH - 1) / BH;
  int nc = by_len < by_sm ? by_len : by_sm;
  return nc < 64 ? nc : 64;
}

}  // namespace

size_t prefill_simt_workspace_bytes(int B, int H, int N, int dk, int dv) {
  const long long BH = (long long)B * H;
  const int nc = simt_chunks((int)BH, N);
  if (nc < 2) return 0;
  return (size_t)BH * nc * ((size_t)dk * dv + dk + 1) * sizeof(float);
}

int simt_chunking(int BH, int N, int blocks, int* L) {
  // as simt_chunks, with a target block count of the caller's
  const int by_len = (N + kTB - 1) / kTB;
  const int by_sm = (blocks + BH - 1) / BH;
  const int nc = by_len < by_sm ? by_len : by_sm;
  if (nc < 2) return 1;
  *L = ((N + nc - 1) / nc + kTB - 1) / kTB * kTB;
  return (N + *L - 1) / *L;
}

cudaError_t launch_simt_entry_states(const PrefillArgs& a, int NC, int L, float* slots, float* S_N,
                                     float* z_N, cudaStream_t stream) {
  const SimtShape sh = simt_shape(a.dk, a.dv);
  if ((a.dk + sh.R - 1) / sh.R > kMaxRows) return cudaErrorInvalidValue;
  const int BH = a.B * a.H;
  SimtChunks ck = {};
  ck.NC = NC;
  ck.L = L;
  if (NC < 2 || L % kTB != 0 || (long long)NC * L < a.N || (long long)(NC - 1) * L >= a.N)
    return cudaErrorInvalidValue;
  ck.slots = slots;
  const size_t smem = sizeof(float) * (3 * kTB * kMaxD + kTB * sh.R * sh.dvp + kTB * sh.R + kTB);
  auto kern = prefill_simt_kernel<0, false, 1>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<dim3((unsigned)ck.NC, (unsigned)BH), kThreads, smem, stream>>>(
      a.q, a.k, a.v, a.bf16, a.N, a.dk, a.dv, a.eps, nullptr, a.S0, a.z0, nullptr, S_N, z_N, ck);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 sgrid((unsigned)((a.dk * a.dv + a.dk + kThreads - 1) / kThreads), (unsigned)BH);
  simt_scan_kernel<false><<<sgrid, kThreads, 0, stream>>>(a.dk, a.dv, a.S0, a.z0, S_N, z_N, ck);
  return cudaGetLastError();
}

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
  const int BH = a.B * a.H;
  SimtChunks ck = {};
  ck.NC = simt_chunks(BH, a.N);
  const size_t need = prefill_simt_workspace_bytes(a.B, a.H, a.N, a.dk, a.dv);
  const bool chunked = ck.NC >= 2 && a.workspace && a.ws_bytes >= need && need > 0;
  if (chunked) {
    ck.L = ((a.N + ck.NC - 1) / ck.NC + kTB - 1) / kTB * kTB;
    ck.NC = (a.N + ck.L - 1) / ck.L;
    ck.slots = static_cast<float*>(a.workspace);
    ck.gam = ck.slots + (size_t)BH * ck.NC * ((size_t)a.dk * a.dv + a.dk);
  }
  auto go = [&](auto kern, dim3 grid) -> cudaError_t {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    kern<<<grid, kThreads, smem, stream>>>(a.q, a.k, a.v, a.bf16, a.N, a.dk, a.dv, a.eps, alpha,
                                           a.S0, a.z0, a.o, a.S_N, a.z_N, ck);
    return cudaGetLastError();
  };
  if (!chunked) {
    const dim3 grid((unsigned)BH);
    if (mode == 2) return go(prefill_simt_kernel<2, false, 0>, grid);
    if (mode == 1)
      return alpha ? go(prefill_simt_kernel<1, true, 0>, grid) : go(prefill_simt_kernel<1, false, 0>, grid);
    return alpha ? go(prefill_simt_kernel<0, true, 0>, grid) : go(prefill_simt_kernel<0, false, 0>, grid);
  }
  const dim3 cgrid((unsigned)ck.NC, (unsigned)BH);
  cudaError_t e = alpha ? go(prefill_simt_kernel<0, true, 1>, cgrid) : go(prefill_simt_kernel<0, false, 1>, cgrid);
  if (e != cudaSuccess) return e;
  const dim3 sgrid((unsigned)((a.dk * a.dv + a.dk + kThreads - 1) / kThreads), (unsigned)BH);
  if (alpha) simt_scan_kernel<true><<<sgrid, kThreads, 0, stream>>>(a.dk, a.dv, a.S0, a.z0, a.S_N, a.z_N, ck);
  else simt_scan_kernel<false><<<sgrid, kThreads, 0, stream>>>(a.dk, a.dv, a.S0, a.z0, a.S_N, a.z_N, ck);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (mode == 2) return go(prefill_simt_kernel<2, false, 2>, cgrid);
  if (mode == 1)
    return alpha ? go(prefill_simt_kernel<1, true, 2>, cgrid) : go(prefill_simt_kernel<1, false, 2>, cgrid);
  return alpha ? go(prefill_simt_kernel<0, true, 2>, cgrid) : go(prefill_simt_kernel<0, false, 2>, cgrid);
}

}  // namespace la
