// backward_simt.cu -- gradient of the causal prefill, on the CUDA cores.
//
// The map of la_prefill (page "AIGC 基本功|线性、循环与记忆架构-LinearMem",
// section 03): S_t = S_{t-1} + phi(k_t) v_t^T, z_t = z_{t-1} + phi(k_t),
// o_t = num_t / den_t with num_t = S_t^T phi(q_t), den_t = phi(q_t).z_t + eps.
// The page gives no backward pass; it notes that training must not keep every
// state and that recomputation solves it.  Given dO (and dS_N, dz_N, NULL =
// zero) the exact gradient is, with the states recomputed:
//   dnum_t = dO_t / den_t,  dden_t = -(dO_t . o_t) / den_t,
//   dphi(q_t) = S_t dnum_t + dden_t z_t                            (forward sweep)
//   G_t = dS_N + sum_{tau >= t} phi(q_tau) dnum_tau^T,
//   g_t = dz_N + sum_{tau >= t} dden_tau phi(q_tau),
//   dphi(k_t) = G_t v_t + g_t,  dv_t = G_t^T phi(k_t)              (reverse sweep)
//   dS0 = G_0, dz0 = g_0,  dq = dphi(q) phi'(q), dk = dphi(k) phi'(k)
// with phi'(u) = 1 for u > 0 and exp(u) for u <= 0.
//
// One block per head, fp32.  As in the CUDA-core prefill, thread (row group,
// column group) owns a (rows x 4) slice of S -- and in the reverse sweep the
// same slice of G.  Per token the block reduces num and den over row groups,
// dden over columns and dphi(q) over column groups through shared memory;
// the forward sweep parks dnum_t in dv's row t and dden_t in dk's row t
// (element 0), and the reverse sweep reads them back before overwriting those
// rows with the gradients.  Tokens are staged TB at a time.  This is the
// plain form of the backward pass (a token-serial chain per head); it is not
// a tensor-core kernel.
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kTB = 8;
constexpr int kMaxD = 128;
constexpr int kMaxRows = 16;

struct Shape {
  int G, R, dvp;
};

__host__ __device__ inline Shape bshape(int dk, int dv) {
  Shape s;
  s.dvp = (dv + 3) & ~3;
  s.G = s.dvp / 4;
  s.R = kThreads / s.G;
  if (s.R > dk) s.R = dk;
  return s;
}

__device__ __forceinline__ float dphi_f32(float u) { return u > 0.f ? 1.f : expf(u); }

struct BwdArgs {
  const void *q, *k, *v;
  bool bf16;
  int N, dk, dv;
  float eps;
  const float *S0, *z0, *dO, *dS_N, *dz_N;
  float *dq, *dk_out, *dv_out, *dS0, *dz0;
};

__global__ void __launch_bounds__(kThreads) backward_simt_kernel(const BwdArgs a) {
  extern __shared__ float sm[];
  const Shape sh = bshape(a.dk, a.dv);
  const int N = a.N, dk = a.dk, dv = a.dv;
  float* fq = sm;                        // [kTB][kMaxD] phi(q)
  float* fk = fq + kTB * kMaxD;          // [kTB][kMaxD] phi(k)
  float* fv = fk + kTB * kMaxD;          // [kTB][kMaxD] v
  float* gv = fv + kTB * kMaxD;          // [kTB][kMaxD] dO (forward) / dnum (reverse)
  float* dpq = gv + kTB * kMaxD;         // [kTB][kMaxD] phi'(q) (forward) / phi'(k) (reverse)
  float* sden = dpq + kTB * kMaxD;       // [kTB] dden (reverse)
  float* part = sden + kTB;              // [R][dvp]  partial sums over rows
  float* rpart = part + sh.R * sh.dvp;   // [kMaxD][G] partial sums over columns
  float* tmp = rpart + kMaxD * sh.G;     // [kMaxD] dnum of the current token
  float* scal = tmp + kMaxD;             // [4] den, dden

  const int tid = threadIdx.x;
  const int g = tid % sh.G, rg = tid / sh.G;
  const bool active = rg < sh.R;
  const int col0 = 4 * g;
  const size_t head = blockIdx.x;

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
        if (a.S0) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (col0 + c < dv) S[r][c] = a.S0[(head * dk + i) * dv + col0 + c];
        }
        if (a.z0) z[r] = a.z0[head * dk + i];
      }
    }
  }

  // ---------------------------------------------------------------- forward
  for (int t0 = 0; t0 < N; t0 += kTB) {
    for (int e = tid; e < kTB * kMaxD; e += kThreads) {
      const int t = e / kMaxD, i = e % kMaxD;
      const int tok = t0 + t;
      const bool in = tok < N;
      float qv = 0.f;
      if (in && i < dk) qv = load_in(a.q, (head * N + tok) * dk + i, a.bf16);
      fq[e] = (in && i < dk) ? phi_f32(qv) : 0.f;
      dpq[e] = (in && i < dk) ? dphi_f32(qv) : 0.f;
      fk[e] = (in && i < dk) ? phi_f32(load_in(a.k, (head * N + tok) * dk + i, a.bf16)) : 0.f;
      fv[e] = (in && i < dv) ? load_in(a.v, (head * N + tok) * dv + i, a.bf16) : 0.f;
      gv[e] = (in && i < dv) ? a.dO[(head * N + tok) * dv + i] : 0.f;
    }
    __syncthreads();
    const int nt = min(kTB, N - t0);
    for (int t = 0; t < nt; ++t) {
      const size_t tok = head * N + t0 + t;
      // write, then the partial read over this thread's rows
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, dacc = 0.f;
      if (active) {
        const float4 vv = *reinterpret_cast<const float4*>(&fv[t * kMaxD + col0]);
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
          const int i = rg + r * sh.R;
          if (i < dk) {
            const float kk = fk[t * kMaxD + i], qq = fq[t * kMaxD + i];
            S[r][0] += kk * vv.x;
            S[r][1] += kk * vv.y;
            S[r][2] += kk * vv.z;
            S[r][3] += kk * vv.w;
            z[r] += kk;
            acc[0] += qq * S[r][0];
            acc[1] += qq * S[r][1];
            acc[2] += qq * S[r][2];
            acc[3] += qq * S[r][3];
            dacc += qq * z[r];
          }
        }
        float* pp = &part[rg * sh.dvp + col0];
        pp[0] = acc[0];
        pp[1] = acc[1];
        pp[2] = acc[2];
        pp[3] = acc[3];
        if (g == 0) rpart[rg] = dacc;  // den partials (column 0 of rpart)
      }
      __syncthreads();
      // den, o, dnum, and the products dO . o
      if (tid == 0) {
        float den = a.eps;
        for (int r = 0; r < sh.R; ++r) den += rpart[r];
        scal[0] = den;
      }
      __syncthreads();
      const float den = scal[0];
      float prod = 0.f;
      if (tid < dv) {
        float num = 0.f;
        for (int r = 0; r < sh.R; ++r) num += part[r * sh.dvp + tid];
        const float o = num / den;
        const float go = gv[t * kMaxD + tid];
        tmp[tid] = go / den;
        prod = go * o;
        a.dv_out[tok * dv + tid] = go / den;  // park dnum_t for the reverse sweep
      } else if (tid < sh.dvp) {
        tmp[tid] = 0.f;  // the padding columns are read as float4 below
      }
      // dden = -sum_j dO_j o_j / den, over the first four warps (dv <= 128)
      if (tid < 128) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) prod += __shfl_xor_sync(0xFFFFFFFFu, prod, off);
        if ((tid & 31) == 0) scal[1 + tid / 32] = prod;  // scal[1..4]
      }
      __syncthreads();
      const float dden = -(scal[1] + scal[2] + scal[3] + scal[4]) / den;
      // dphi(q)_i = sum_j S_ij dnum_j + dden z_i, partial over this thread's columns
      if (active) {
        const float4 dn = *reinterpret_cast<const float4*>(&tmp[col0]);
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
          const int i = rg + r * sh.R;
          if (i < dk) {
            float s = S[r][0] * dn.x + S[r][1] * dn.y + S[r][2] * dn.z + S[r][3] * dn.w;
            if (g == 0) s += dden * z[r];
            rpart[i * sh.G + g] = s;
          }
        }
      }
      __syncthreads();
      if (tid < dk) {
        float s = 0.f;
        for (int c = 0; c < sh.G; ++c) s += rpart[tid * sh.G + c];
        a.dq[tok * dk + tid] = s * dpq[t * kMaxD + tid];
      }
      if (tid == 0) a.dk_out[tok * dk] = dden;  // park dden_t for the reverse sweep
      __syncthreads();
    }
  }

  // ---------------------------------------------------------------- reverse
  // S and z become G and g
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
        if (a.dS_N) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (col0 + c < dv) S[r][c] = a.dS_N[(head * dk + i) * dv + col0 + c];
        }
        if (a.dz_N) z[r] = a.dz_N[head * dk + i];
      }
    }
  }
  const int nstage = (N + kTB - 1) / kTB;
  for (int sidx = nstage - 1; sidx >= 0; --sidx) {
    const int t0 = sidx * kTB;
    const int nt = min(kTB, N - t0);
    __syncthreads();  // the previous stage's reads of the staging arrays are done
    for (int e = tid; e < kTB * kMaxD; e += kThreads) {
      const int t = e / kMaxD, i = e % kMaxD;
      const int tok = t0 + t;
      const bool in = t < nt;
      float kv = 0.f;
      if (in && i < dk) kv = load_in(a.k, (head * N + tok) * dk + i, a.bf16);
      fq[e] = (in && i < dk) ? phi_f32(load_in(a.q, (head * N + tok) * dk + i, a.bf16)) : 0.f;
      fk[e] = (in && i < dk) ? phi_f32(kv) : 0.f;
      dpq[e] = (in && i < dk) ? dphi_f32(kv) : 0.f;
      fv[e] = (in && i < dv) ? load_in(a.v, (head * N + tok) * dv + i, a.bf16) : 0.f;
      gv[e] = (in && i < dv) ? a.dv_out[(head * N + tok) * dv + i] : 0.f;  // dnum_t
    }
    if (tid < kTB) sden[tid] = tid < nt ? a.dk_out[(head * N + t0 + tid) * dk] : 0.f;  // dden_t
    __syncthreads();
    for (int t = nt - 1; t >= 0; --t) {
      const size_t tok = head * N + t0 + t;
      const float dd = sden[t];
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (active) {
        const float4 dn = *reinterpret_cast<const float4*>(&gv[t * kMaxD + col0]);
        const float4 vv = *reinterpret_cast<const float4*>(&fv[t * kMaxD + col0]);
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
          const int i = rg + r * sh.R;
          if (i < dk) {
            const float qq = fq[t * kMaxD + i], kk = fk[t * kMaxD + i];
            S[r][0] += qq * dn.x;
            S[r][1] += qq * dn.y;
            S[r][2] += qq * dn.z;
            S[r][3] += qq * dn.w;
            z[r] += dd * qq;
            // dv partials over this thread's rows, dphi(k) partials over its columns
            acc[0] += S[r][0] * kk;
            acc[1] += S[r][1] * kk;
            acc[2] += S[r][2] * kk;
            acc[3] += S[r][3] * kk;
            float s = S[r][0] * vv.x + S[r][1] * vv.y + S[r][2] * vv.z + S[r][3] * vv.w;
            if (g == 0) s += z[r];
            rpart[i * sh.G + g] = s;
          }
        }
        float* pp = &part[rg * sh.dvp + col0];
        pp[0] = acc[0];
        pp[1] = acc[1];
        pp[2] = acc[2];
        pp[3] = acc[3];
      }
      __syncthreads();
      if (tid < dk) {
        float s = 0.f;
        for (int c = 0; c < sh.G; ++c) s += rpart[tid * sh.G + c];
        a.dk_out[tok * dk + tid] = s * dpq[t * kMaxD + tid];
      }
      if (tid < dv) {
        float s = 0.f;
        for (int r = 0; r < sh.R; ++r) s += part[r * sh.dvp + tid];
        a.dv_out[tok * dv + tid] = s;
      }
      __syncthreads();
    }
  }
  if (active) {
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      const int i = rg + r * sh.R;
      if (i < dk) {
        if (a.dS0) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (col0 + c < dv) a.dS0[(head * dk + i) * dv + col0 + c] = S[r][c];
        }
        if (a.dz0 && g == 0) a.dz0[head * dk + i] = z[r];
      }
    }
  }
}

}  // namespace

cudaError_t launch_prefill_backward(const PrefillArgs& p, const float* dO, const float* dS_N,
                                    const float* dz_N, float* dq, float* dk, float* dv,
                                    float* dS0, float* dz0, cudaStream_t stream) {
  const Shape sh = bshape(p.dk, p.dv);
  if ((p.dk + sh.R - 1) / sh.R > kMaxRows) return cudaErrorInvalidValue;
  BwdArgs a;
  a.q = p.q; a.k = p.k; a.v = p.v; a.bf16 = p.bf16;
  a.N = p.N; a.dk = p.dk; a.dv = p.dv; a.eps = p.eps;
  a.S0 = p.S0; a.z0 = p.z0; a.dO = dO; a.dS_N = dS_N; a.dz_N = dz_N;
  a.dq = dq; a.dk_out = dk; a.dv_out = dv; a.dS0 = dS0; a.dz0 = dz0;
  const size_t smem = sizeof(float) * (5 * kTB * kMaxD + kTB + sh.R * sh.dvp + kMaxD * sh.G +
                                       kMaxD + 8);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(backward_simt_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const unsigned blocks = (unsigned)((size_t)p.B * p.H);
  backward_simt_kernel<<<blocks, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace la
