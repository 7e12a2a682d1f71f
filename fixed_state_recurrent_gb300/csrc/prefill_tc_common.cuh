// prefill_tc_common.cuh -- pieces shared by the tensor-core prefill kernels:
// the chunk length, the ELU+1 feature map on packed bf16, the work split over
// the SMs, and tensor-map creation.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>

#include "la_internal.h"
#include "tc_primitives.cuh"

namespace la {
namespace tcp {

constexpr int C = 128;            // chunk length = MMA M = tile rows

// 2^x by the single-precision hardware approximation, subnormal results
// flushed to zero (exp(u) < 2^-126 is far below what bf16 sums of phi keep).
__device__ __forceinline__ float exp2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// phi on two bf16: phi(u) = exp(min(u, 0)) + max(u, 0), which is u + 1 for
// u > 0 and exp(u) otherwise.  min and max are taken on the bf16 pair, the
// exponentials as 2^(min(u, 0) log2 e) in fp32, and the sum is rounded to
// bf16, the precision of the tensor-core operand it feeds: the result is
// within one bf16 rounding of phi(u).
__device__ __forceinline__ uint32_t phi2(uint32_t x) {
  const __nv_bfloat162 u = *reinterpret_cast<const __nv_bfloat162*>(&x);
  const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
  const __nv_bfloat162 m = __hmin2(u, zero);
  const __nv_bfloat162 M = __hmax2(u, zero);
  const uint32_t mb = *reinterpret_cast<const uint32_t*>(&m);
  const uint32_t e = tc::pack_bf16x2(exp2_ftz(__uint_as_float(mb << 16) * 1.4426950408889634f),
                                 exp2_ftz(__uint_as_float(mb & 0xFFFF0000u) * 1.4426950408889634f));
  const __nv_bfloat162 r = __hadd2(*reinterpret_cast<const __nv_bfloat162*>(&e), M);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// phi on `nchunk` 16-byte chunks of row r of a tile starting at chunk `c0`;
// rows at or past `valid` become zero.  Loads first, then math, then stores.
// The row mask is applied with an AND after an unconditional phi: a
// conditional around phi2 lets the compiler branch around every pair, which
// serialises the 4 NCH independent exponential chains of a thread.
template <int NCH>
__device__ __forceinline__ void phi_row(uint8_t* tile, int r, int c0, int valid) {
  uint4 v[NCH];
#pragma unroll
  for (int i = 0; i < NCH; ++i) v[i] = *reinterpret_cast<const uint4*>(tile + tc::sw128_offset(r, c0 + i));
  const uint32_t keep = r < valid ? 0xFFFFFFFFu : 0u;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    v[i].x = phi2(v[i].x) & keep;
    v[i].y = phi2(v[i].y) & keep;
    v[i].z = phi2(v[i].z) & keep;
    v[i].w = phi2(v[i].w) & keep;
  }
#pragma unroll
  for (int i = 0; i < NCH; ++i) *reinterpret_cast<uint4*>(tile + tc::sw128_offset(r, c0 + i)) = v[i];
}

// The all-ones operand block: a [128 token rows x 64] bf16 swizzled tile whose
// column 0 is 1 (as the second atom of [V | 1], read MN-major or K-major).
// Contains a block-wide barrier.
__device__ __forceinline__ void init_ones(uint8_t* ones, int tid, int nthreads) {
  for (int i = tid; i < (int)(16384 / 16); i += nthreads)
    reinterpret_cast<uint4*>(ones)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (tid < C) *reinterpret_cast<uint16_t*>(ones + tc::sw128_offset(tid, 0)) = 0x3F80u;  // bf16 1.0
}

// ---------------------------------------------------------------------------
// work split (the kernels and the host share it)

struct Split {
  int BH, N, NC;  // heads, tokens per head, chunks per head
  int G;          // blocks of K1 and K3
  int MPH;        // piece slots per head
  __host__ __device__ long long TC() const { return (long long)BH * NC; }
  __host__ __device__ long long start(int j) const { return (long long)j * TC() / G; }
  // the block whose run contains global chunk x
  __host__ __device__ int owner(long long x) const {
    return (int)(((x + 1) * G - 1) / TC());
  }
};

struct Piece {
  int h, slot;
  int tok0, tok1, nch;
};

// Block j's run of chunks [a, b) and the pieces it is cut into.  The 64-bit
// divisions happen once, here; walking the pieces needs none.
struct Run {
  long long a, b;
  int h0;    // head of the first piece
  int idx0;  // position of block j among the blocks that meet head h0
  __host__ __device__ Run(const Split& s, int j) {
    a = s.start(j);
    b = s.start(j + 1);
    h0 = (int)(a / s.NC);
    idx0 = j - s.owner((long long)h0 * s.NC);
  }
  // Number of pieces.
  __host__ __device__ int count(const Split& s) const {
    int n = 0;
    Piece pc;
    while (piece(s, n, &pc)) ++n;
    return n;
  }
  // The i-th piece (pieces are ordered by position); false when there are
  // fewer.  Every piece after the first starts its head, so its slot index
  // within the head is 0.
  __host__ __device__ bool piece(const Split& s, int i, Piece* pc) const {
    if (a >= b) return false;
    const int h = h0 + i;
    const long long hs = (long long)h * s.NC;
    if (hs >= b || h >= s.BH) return false;
    const long long c0 = a > hs ? a : hs;
    const long long c1 = b < hs + s.NC ? b : hs + s.NC;
    pc->h = h;
    pc->slot = h * s.MPH + (i == 0 ? idx0 : 0);
    pc->tok0 = (int)(c0 - hs) * C;
    pc->tok1 = (int)(c1 - hs) * C;
    if (pc->tok1 > s.N) pc->tok1 = s.N;
    pc->nch = (int)(c1 - c0);
    return true;
  }
};

inline Split make_split(int BH, int N, int sms) {
  Split s;
  s.BH = BH;
  s.N = N;
  s.NC = (N + C - 1) / C;
  const long long tc = (long long)BH * s.NC;
  s.G = (int)(tc < sms ? tc : sms);
  // Runs are L = floor(TC / G) or L + 1 chunks long; a head's NC chunks meet at
  // most ceil(NC / L) + 1 of them (every run but the first and last lies inside).
  const long long L = tc / s.G;
  s.MPH = (int)((s.NC + L - 1) / L) + 1;
  return s;
}

// SMs of the current device (152 on a GB300 when no device is visible, so
// that host-only queries of the workspace size still answer).
inline int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    return 152;
  }
  return sms;
}

// ---------------------------------------------------------------------------
// host helpers

inline PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 3-D map over a [BH][N][d] tensor (innermost dimension first), 128-byte
// swizzle, boxes of box0 x box1 x 1.  Out-of-range elements load as zero and
// are not stored.
inline bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int d,
                     int N, int BH, int box0, int box1) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * esize, (cuuint64_t)N * d * esize};
  cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline unsigned long long env_ull(const char* name, unsigned long long dflt) {
  const char* s = getenv(name);
  if (!s || !*s) return dflt;
  return strtoull(s, nullptr, 10);
}

}  // namespace tcp
}  // namespace la
