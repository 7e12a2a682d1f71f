// decode.cu -- one decode step of normalized causal linear attention on a
// resident fp32 state, updated in place.
//
// Page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03: the step first
// writes the token (S += phi(k) v^T, z += phi(k)) and then reads it with the
// query, o = phi(q)^T S / (phi(q)^T z + eps); per step the cost is O(dk dv) and
// the state is the only thing that has to move.
//
// The step is HBM-bound: each head's S (64 KB at 128 x 128) is read once and
// written once, everything else is < 2 KB.  One block per head streams its S
// rows with 128-bit loads and stores (evict-first: the whole state is far
// larger than L2 and is not reused before the next step), fuses the rank-1
// update and the read phi(q)^T S_new in registers, and reduces the partial
// numerators over row groups in shared memory.  phi(q) . z_new goes through a
// warp-shuffle reduction.
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxD = 128;

template <int VEC>
struct DecodeShape {
  int G, R;
  __host__ __device__ DecodeShape(int dk, int dv) {
    G = (dv + VEC - 1) / VEC;
    R = kThreads / G;
    if (R > dk) R = dk;
  }
};

template <int VEC, int MAXR>
__global__ void __launch_bounds__(kThreads, 2)
decode_step_kernel(const void* __restrict__ q, const void* __restrict__ k,
                   const void* __restrict__ v, bool bf16, int dk, int dv,
                   float eps, float* __restrict__ S, float* __restrict__ z,
                   float* __restrict__ o) {
  __shared__ float fq[kMaxD], fk[kMaxD], fv[kMaxD];
  __shared__ float part[kThreads * VEC];  // [R][G*VEC]
  __shared__ float dred[kThreads / 32];

  const DecodeShape<VEC> sh(dk, dv);
  const int tid = threadIdx.x;
  const size_t head = blockIdx.x;
  const int g = tid % sh.G, rg = tid / sh.G;
  const bool active = rg < sh.R;
  const int col0 = g * VEC;

  if (tid < dk) {
    fq[tid] = phi_f32(load_in(q, head * dk + tid, bf16));
    fk[tid] = phi_f32(load_in(k, head * dk + tid, bf16));
  }
  if (tid < dv) fv[tid] = load_in(v, head * dv + tid, bf16);
  __syncthreads();

  float acc[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) acc[c] = 0.f;

  if (active) {
    float* Sh = S + head * (size_t)dk * dv;
    if constexpr (VEC == 4) {
      float4 s[MAXR];
      // issue every load of this thread's rows before using any of them
#pragma unroll
      for (int r = 0; r < MAXR; ++r) {
        const int i = rg + r * sh.R;
        if (i < dk) s[r] = __ldcs(reinterpret_cast<const float4*>(Sh + (size_t)i * dv + col0));
      }
      const float4 vv = *reinterpret_cast<const float4*>(&fv[col0]);
#pragma unroll
      for (int r = 0; r < MAXR; ++r) {
        const int i = rg + r * sh.R;
        if (i < dk) {
          const float a = fk[i], b = fq[i];
          s[r].x += a * vv.x;
          s[r].y += a * vv.y;
          s[r].z += a * vv.z;
          s[r].w += a * vv.w;
          __stcs(reinterpret_cast<float4*>(Sh + (size_t)i * dv + col0), s[r]);
          acc[0] += b * s[r].x;
          acc[1] += b * s[r].y;
          acc[2] += b * s[r].z;
          acc[3] += b * s[r].w;
        }
      }
    } else {
      if (col0 < dv) {
        for (int i = rg; i < dk; i += sh.R) {
          float s = __ldcs(Sh + (size_t)i * dv + col0);
          s += fk[i] * fv[col0];
          __stcs(Sh + (size_t)i * dv + col0, s);
          acc[0] += fq[i] * s;
        }
      }
    }
    const int W = sh.G * VEC;
#pragma unroll
    for (int c = 0; c < VEC; ++c) part[rg * W + col0 + c] = acc[c];
  }

  // denominator: phi(q) . (z + phi(k)), z written back
  float d = 0.f;
  if (tid < dk) {
    const float zn = z[head * dk + tid] + fk[tid];
    z[head * dk + tid] = zn;
    d = fq[tid] * zn;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
  if ((tid & 31) == 0) dred[tid >> 5] = d;
  __syncthreads();

  if (tid < dv) {
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) den += dred[w];
    const int W = sh.G * VEC;
    float num = 0.f;
    for (int r = 0; r < sh.R; ++r) num += part[r * W + tid];
    o[head * dv + tid] = num / (den + eps);
  }
}

}  // namespace

cudaError_t launch_decode_step(const void* q, const void* k, const void* v,
                               bool bf16, int B, int H, int dk, int dv,
                               float eps, float* S, float* z, float* o,
                               cudaStream_t stream) {
  const unsigned blocks = (unsigned)((size_t)B * H);
  if (dv % 4 == 0) {
    // rows per thread: dk / R with R = 512 / (dv / 4) >= 16, so <= 8
    decode_step_kernel<4, 8><<<blocks, kThreads, 0, stream>>>(
        q, k, v, bf16, dk, dv, eps, S, z, o);
  } else {
    decode_step_kernel<1, 1><<<blocks, kThreads, 0, stream>>>(
        q, k, v, bf16, dk, dv, eps, S, z, o);
  }
  return cudaGetLastError();
}

}  // namespace la
