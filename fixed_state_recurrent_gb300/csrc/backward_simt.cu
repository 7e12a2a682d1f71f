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
// fp32.  As in the CUDA-core prefill, thread (row group, column group) owns a
// (rows x 4) slice of S -- and in the reverse sweep the same slice of G.  Per
// token the block reduces num and den over row groups, dden over columns and
// dphi(q) over column groups through shared memory; the forward sweep parks
// dnum_t in dv's row t and dden_t in dk's row t (element 0), and the reverse
// sweep reads them back before overwriting those rows with the gradients.
// Tokens are staged TB at a time.  Not a tensor-core kernel.
//
// Without a workspace one block walks a whole head, both sweeps (PASS 0).
// With one the heads are cut into the CUDA-core prefill's chunks and five
// launches run them in parallel:
//   1-2. the prefill's chunk increments and scan: the state before every
//        chunk (prefill_simt.cu);
//   3. PASS 1, per chunk: the forward sweep from the state before the chunk
//      (dq; dnum and dden parked);
//   4. per chunk, its gradient-state increment from the parked rows,
//      dG_c = sum_{t in c} phi(q_t) dnum_t^T, dg_c = sum_{t in c} dden_t phi(q_t)
//      (a product over the chunk's tokens, no per-token reductions);
//   5. per head, the gradient state after every chunk as the right fold
//      dS_N + dG_{c+1} + dG_{c+2} + ... (always in this order), and dS0, dz0;
//   6. PASS 2, per chunk: the reverse sweep from the gradient state after the
//      chunk.
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
  // chunked form: NC chunks of L tokens per head; per (head, chunk) a slot of
  // dk dv + dk floats (row-major [i][j], then the dk vector)
  int NC, L;
  const float* E;  // the state before every chunk
  float* Gs;       // PASS 1: the gradient-state increments; PASS 2: the gradient state after every chunk
};

// PASS 0: a whole head, both sweeps; 1: one chunk's forward sweep; 2: one
// chunk's reverse sweep (see the top of the file).
template <int PASS>
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
  const size_t head = PASS == 0 ? blockIdx.x : blockIdx.y;
  const int chunk = PASS == 0 ? 0 : blockIdx.x;
  const int tb = PASS == 0 ? 0 : chunk * a.L;             // this block's tokens [tb, te)
  const int te = PASS == 0 ? N : min(N, tb + a.L);
  const size_t slot_sz = (size_t)dk * dv + dk;
  const size_t slot = (head * a.NC + chunk) * slot_sz;

  float S[kMaxRows][4];
  float z[kMaxRows];
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) {
    z[r] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) S[r][c] = 0.f;
  }
  if (PASS != 2 && active) {  // the state before the block's first token
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      const int i = rg + r * sh.R;
      if (i < dk) {
        const float* Si = PASS == 0 ? (a.S0 ? a.S0 + (head * dk + i) * dv : nullptr) : a.E + slot + (size_t)i * dv;
        const float* zi = PASS == 0 ? (a.z0 ? a.z0 + head * dk + i : nullptr) : a.E + slot + (size_t)dk * dv + i;
        if (Si) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (col0 + c < dv) S[r][c] = Si[col0 + c];
        }
        if (zi) z[r] = *zi;
      }
    }
  }

  // ---------------------------------------------------------------- forward
  for (int t0 = tb; PASS != 2 && t0 < te; t0 += kTB) {
    for (int e = tid; e < kTB * kMaxD; e += kThreads) {
      const int t = e / kMaxD, i = e % kMaxD;
      const int tok = t0 + t;
      const bool in = tok < te;
      float qv = 0.f;
      if (in && i < dk) qv = load_in(a.q, (head * N + tok) * dk + i, a.bf16);
      fq[e] = (in && i < dk) ? phi_f32(qv) : 0.f;
      dpq[e] = (in && i < dk) ? dphi_f32(qv) : 0.f;
      fk[e] = (in && i < dk) ? phi_f32(load_in(a.k, (head * N + tok) * dk + i, a.bf16)) : 0.f;
      fv[e] = (in && i < dv) ? load_in(a.v, (head * N + tok) * dv + i, a.bf16) : 0.f;
      gv[e] = (in && i < dv) ? a.dO[(head * N + tok) * dv + i] : 0.f;
    }
    __syncthreads();
    const int nt = min(kTB, te - t0);
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

  if (PASS == 1) return;  // (the reverse sweep below is then unreachable)

  // ---------------------------------------------------------------- reverse
  // S and z become G and g
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) {
    z[r] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) S[r][c] = 0.f;
  }
  if (active) {  // the gradient state after the block's last token
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      const int i = rg + r * sh.R;
      if (i < dk) {
        const float* Gi = PASS == 0 ? (a.dS_N ? a.dS_N + (head * dk + i) * dv : nullptr) : a.Gs + slot + (size_t)i * dv;
        const float* gi = PASS == 0 ? (a.dz_N ? a.dz_N + head * dk + i : nullptr) : a.Gs + slot + (size_t)dk * dv + i;
        if (Gi) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (col0 + c < dv) S[r][c] = Gi[col0 + c];
        }
        if (gi) z[r] = *gi;
      }
    }
  }
  const int nstage = (te - tb + kTB - 1) / kTB;
  for (int sidx = nstage - 1; sidx >= 0; --sidx) {
    const int t0 = tb + sidx * kTB;
    const int nt = min(kTB, te - t0);
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
  if (PASS == 0 && active) {
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

// Per chunk (blockIdx.x) of head blockIdx.y: dG_c = sum_t phi(q_t) dnum_t^T
// and dg_c = sum_t dden_t phi(q_t) over the chunk's tokens, from the rows the
// forward sweep parked in dv_out (dnum) and dk_out (dden, element 0), into
// the chunk's slot of Gs.  Thread (row group, column group) owns the same
// (rows x 4) slice as in the sweeps.
__global__ void __launch_bounds__(kThreads) bwd_increment_kernel(const BwdArgs a) {
  extern __shared__ float sm[];
  const Shape sh = bshape(a.dk, a.dv);
  const int N = a.N, dk = a.dk, dv = a.dv;
  float* fq = sm;                  // [kTB][kMaxD] phi(q)
  float* dn = fq + kTB * kMaxD;    // [kTB][kMaxD] dnum
  float* dd = dn + kTB * kMaxD;    // [kTB] dden
  const int tid = threadIdx.x;
  const int g = tid % sh.G, rg = tid / sh.G;
  const bool active = rg < sh.R;
  const int col0 = 4 * g;
  const size_t head = blockIdx.y;
  const int chunk = blockIdx.x;
  const int tb = chunk * a.L, te = min(N, tb + a.L);
  const size_t slot = (head * a.NC + chunk) * ((size_t)dk * dv + dk);
  float G[kMaxRows][4], gz[kMaxRows];
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) {
    gz[r] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) G[r][c] = 0.f;
  }
  for (int t0 = tb; t0 < te; t0 += kTB) {
    const int nt = min(kTB, te - t0);
    __syncthreads();  // the previous stage has been read
    for (int e = tid; e < kTB * kMaxD; e += kThreads) {
      const int t = e / kMaxD, i = e % kMaxD;
      const bool in = t < nt;
      fq[e] = (in && i < dk) ? phi_f32(load_in(a.q, (head * N + t0 + t) * dk + i, a.bf16)) : 0.f;
      dn[e] = (in && i < dv) ? a.dv_out[(head * N + t0 + t) * dv + i] : 0.f;
    }
    if (tid < kTB) dd[tid] = tid < nt ? a.dk_out[(head * N + t0 + tid) * dk] : 0.f;
    __syncthreads();
    if (active) {
      for (int t = 0; t < nt; ++t) {
        const float4 d4 = *reinterpret_cast<const float4*>(&dn[t * kMaxD + col0]);
        const float de = dd[t];
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
          const int i = rg + r * sh.R;
          if (i < dk) {
            const float qq = fq[t * kMaxD + i];
            G[r][0] += qq * d4.x;
            G[r][1] += qq * d4.y;
            G[r][2] += qq * d4.z;
            G[r][3] += qq * d4.w;
            gz[r] += de * qq;
          }
        }
      }
    }
  }
  if (active) {
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      const int i = rg + r * sh.R;
      if (i < dk) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (col0 + c < dv) a.Gs[slot + (size_t)i * dv + col0 + c] = G[r][c];
        if (g == 0) a.Gs[slot + (size_t)dk * dv + i] = gz[r];
      }
    }
  }
}

// Per head and state element: the gradient state after every chunk, in
// place of the chunk's increment, as the right fold from dS_N (dz_N) taken
// from the last chunk back to the first, and dS0, dz0.
__global__ void __launch_bounds__(kThreads) bwd_gscan_kernel(const BwdArgs a) {
  const size_t head = blockIdx.y;
  const int e = blockIdx.x * kThreads + threadIdx.x;
  const int nS = a.dk * a.dv;
  if (e >= nS + a.dk) return;
  float acc = e < nS ? (a.dS_N ? a.dS_N[head * nS + e] : 0.f) : (a.dz_N ? a.dz_N[head * a.dk + e - nS] : 0.f);
  const size_t sz = (size_t)nS + a.dk;
  float* col = a.Gs + head * a.NC * sz + e;
  for (int c = a.NC - 1; c >= 0; --c) {
    const float d = col[c * sz];
    col[c * sz] = acc;
    acc += d;
  }
  if (e < nS) {
    if (a.dS0) a.dS0[head * nS + e] = acc;
  } else if (a.dz0) {
    a.dz0[head * a.dk + e - nS] = acc;
  }
}

}  // namespace

// Chunks of the chunked form: about four blocks per SM of a 152-SM GPU (the
// sweeps hold two blocks per SM), so that they run in whole waves.
constexpr int kBwdBlocks = 4 * 152;

// the chunked form: the state before every chunk, the gradient states, and
// S_N, z_N of the prefill's scan (unused)
size_t backward_simt_workspace_bytes(int B, int H, int N, int dk, int dv) {
  int L = 0;
  const int nc = simt_chunking(B * H, N, kBwdBlocks, &L);
  if (nc < 2) return 0;
  return (size_t)B * H * (2 * (size_t)nc + 1) * ((size_t)dk * dv + dk) * sizeof(float);
}

cudaError_t launch_prefill_backward(const PrefillArgs& p, const float* dO, const float* dS_N,
                                    const float* dz_N, float* dq, float* dk, float* dv,
                                    float* dS0, float* dz0, cudaStream_t stream) {
  const Shape sh = bshape(p.dk, p.dv);
  if ((p.dk + sh.R - 1) / sh.R > kMaxRows) return cudaErrorInvalidValue;
  BwdArgs a = {};
  a.q = p.q; a.k = p.k; a.v = p.v; a.bf16 = p.bf16;
  a.N = p.N; a.dk = p.dk; a.dv = p.dv; a.eps = p.eps;
  a.S0 = p.S0; a.z0 = p.z0; a.dO = dO; a.dS_N = dS_N; a.dz_N = dz_N;
  a.dq = dq; a.dk_out = dk; a.dv_out = dv; a.dS0 = dS0; a.dz0 = dz0;
  const size_t smem = sizeof(float) * (5 * kTB * kMaxD + kTB + sh.R * sh.dvp + kMaxD * sh.G +
                                       kMaxD + 8);
  auto prep = [&](auto kern) -> cudaError_t {
    if (smem > 48 * 1024)
      return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return cudaSuccess;
  };
  const unsigned BH = (unsigned)((size_t)p.B * p.H);
  const size_t need = backward_simt_workspace_bytes(p.B, p.H, p.N, p.dk, p.dv);
  if (!p.workspace || need == 0 || p.ws_bytes < need) {  // one block per head
    cudaError_t e = prep(backward_simt_kernel<0>);
    if (e != cudaSuccess) return e;
    backward_simt_kernel<0><<<BH, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
  }
  a.NC = simt_chunking((int)BH, p.N, kBwdBlocks, &a.L);
  const size_t sz = (size_t)p.dk * p.dv + p.dk;
  float* E = static_cast<float*>(p.workspace);
  a.E = E;
  a.Gs = E + (size_t)BH * a.NC * sz;
  float* SN = a.Gs + (size_t)BH * a.NC * sz;
  cudaError_t e = launch_simt_entry_states(p, a.NC, a.L, E, SN, SN + (size_t)BH * p.dk * p.dv, stream);
  if (e == cudaSuccess) e = prep(backward_simt_kernel<1>);
  if (e == cudaSuccess) e = prep(backward_simt_kernel<2>);
  if (e != cudaSuccess) return e;
  const dim3 cgrid((unsigned)a.NC, BH);
  backward_simt_kernel<1><<<cgrid, kThreads, smem, stream>>>(a);
  bwd_increment_kernel<<<cgrid, kThreads, sizeof(float) * (2 * kTB * kMaxD + kTB), stream>>>(a);
  bwd_gscan_kernel<<<dim3((unsigned)((sz + kThreads - 1) / kThreads), BH), kThreads, 0, stream>>>(a);
  backward_simt_kernel<2><<<cgrid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace la
