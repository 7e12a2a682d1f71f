// prefill_scan.cuh -- the entry state of every piece of the tensor-core
// prefill's work split, and the final state, as the fold of the pieces'
// totals in head order.
//
// Per head (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03: the
// state after a span of tokens is the state before it plus the span's sum of
// phi(k) v^T and phi(k); with a scalar decay alpha, page "线性注意力与SSM",
// sections 3-4, the state before the span is first scaled by the span's
// product of alpha, and the span's own sum carries the later alphas):
//   E_0 = S0,  E_{w+1} = gamma_w E_w + R_w  (gamma_w = 1 without decay),
//   S_N = E_npieces,
// always in this order, in fp32, so results repeat bit for bit.
//
// Slots hold S^T rows (row j = value column, D floats over the key index i),
// then z (D floats).  A thread takes four consecutive floats of a slot, so the
// totals and entry states move as 16-byte loads and stores, every piece's load
// in flight at once.  S0 and S_N are stored [i][j] (the transpose of a slot's
// rows); a block's share of them goes through shared memory so that their
// global accesses are 16-byte runs too.  A block reads its share of S0 before
// it writes the same share of S_N, so S_N may be S0 (in place).
//
// Optionally the fold also writes each head's final state as the bf16
// operand tile of a product phi(Q) [S_N | z_N]^T (StateTile below).
#pragma once

#include "prefill_tc_common.cuh"

namespace la {
namespace tcp {

constexpr int kScanThreads = 256;

// A state as the K-major bf16 B operand of an M = 128 product over N_S = D + 16
// columns: D / 64 atoms (K = 64 each) of N_S rows of 128 swizzled bytes; row
// j < D holds column j of S (a slot's S^T row j), row D bf16(z), row D + 1 the
// rest of z (z - bf16(z), as bf16), the rows after that zero.
template <int D>
struct StateTile {
  static constexpr int NS = D + 16;
  static constexpr uint32_t XA = NS * 128;          // one atom
  static constexpr uint32_t BYTES = (D / 64) * XA;  // the tile
};

// Four consecutive K positions (col .. col + 3) of tile row `row`.
template <int D>
__device__ __forceinline__ void state_tile_put4(uint8_t* tile, int row, int col, uint2 v) {
  const int c = col % 64;
  *reinterpret_cast<uint2*>(tile + (col / 64) * StateTile<D>::XA + tc::sw128_offset(row, c / 8) + (c % 8) * 2) = v;
}

// acc (four floats of slot row `row`, keys col .. col + 3) into the tile: S
// rows as bf16, the z row as hi and lo rows.
template <int D>
__device__ __forceinline__ void state_tile_put(uint8_t* tile, int row, int col, float4 acc) {
  uint2 hi;
  hi.x = tc::pack_bf16x2(acc.x, acc.y);
  hi.y = tc::pack_bf16x2(acc.z, acc.w);
  if (row < D) {
    state_tile_put4<D>(tile, row, col, hi);
  } else {
    uint2 lo;
    lo.x = tc::pack_bf16x2(acc.x - __uint_as_float(hi.x << 16), acc.y - __uint_as_float(hi.x & 0xFFFF0000u));
    lo.y = tc::pack_bf16x2(acc.z - __uint_as_float(hi.y << 16), acc.w - __uint_as_float(hi.y & 0xFFFF0000u));
    state_tile_put4<D>(tile, D, col, hi);
    state_tile_put4<D>(tile, D + 1, col, lo);
  }
}

// Blocks per head: D * D / (4 kScanThreads) for the S rows, one for z.
template <int D>
constexpr int scan_blocks_per_head() {
  return D * D / (4 * kScanThreads) + 1;
}

// One block of the fold (blockIdx.x = part of the slot, blockIdx.y = head).
// `gam` (DECAY only) holds one factor per piece slot.  E (the entry states)
// and `tiles` (per head a StateTile of S_N, z_N) may be NULL.
template <int D, bool DECAY>
__device__ __forceinline__ void scan_fold(const Split& s, const float* __restrict__ agg,
                                          float* __restrict__ E, const float* __restrict__ gam,
                                          const float* __restrict__ S0, const float* __restrict__ z0,
                                          float* __restrict__ S_N, float* __restrict__ z_N,
                                          uint8_t* __restrict__ tiles = nullptr) {
  static_assert((D * D) % (4 * kScanThreads) == 0 && D % 4 == 0 && D / 4 <= kScanThreads,
                "slot split");
  constexpr int SZ = D * D + D;
  constexpr int RB = 4 * kScanThreads / D;  // S^T rows per block
  __shared__ float tile[D][RB + 1];         // [i][row - r0], padded against bank conflicts
  const int h = blockIdx.y, t = threadIdx.x;
  const bool zpart = blockIdx.x == D * D / (4 * kScanThreads);
  const int r0 = blockIdx.x * RB;
  // this thread's four floats: S^T row `row`, keys i0 .. i0 + 3 (or z[i0 ..])
  const int row = zpart ? D : r0 + 4 * t / D;
  const int i0 = (4 * t) % D;
  const bool mine = !zpart || t < D / 4;
  const int e = row * D + i0;

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!zpart) {
    if (S0) {  // S0[h][i][r0 .. r0 + RB) -> tile, 16 bytes per thread
      for (int f = 4 * t; f < D * RB; f += 4 * kScanThreads) {
        const int i = f / RB, k = f % RB;
        const float4 u = *reinterpret_cast<const float4*>(S0 + ((size_t)h * D + i) * D + r0 + k);
        tile[i][k] = u.x;
        tile[i][k + 1] = u.y;
        tile[i][k + 2] = u.z;
        tile[i][k + 3] = u.w;
      }
      __syncthreads();
      acc = make_float4(tile[i0][row - r0], tile[i0 + 1][row - r0], tile[i0 + 2][row - r0],
                        tile[i0 + 3][row - r0]);
      __syncthreads();
    }
  } else if (z0 && mine) {
    acc = *reinterpret_cast<const float4*>(z0 + (size_t)h * D + i0);
  }

  const int first = s.owner((long long)h * s.NC);
  const int npieces = s.owner((long long)(h + 1) * s.NC - 1) - first + 1;
  const size_t base = (size_t)h * s.MPH * SZ + e;
  constexpr int U = 8;
  if (mine) {
    for (int w0 = 0; w0 < npieces; w0 += U) {
      float4 a[U];
      float g[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        g[u] = 1.f;
        if (w0 + u < npieces) {
          a[u] = __ldcg(reinterpret_cast<const float4*>(agg + base + (size_t)(w0 + u) * SZ));
          if (DECAY) g[u] = __ldcg(gam + (size_t)h * s.MPH + w0 + u);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (w0 + u < npieces) {
          if (E) __stcg(reinterpret_cast<float4*>(E + base + (size_t)(w0 + u) * SZ), acc);
          if (DECAY) {
            acc.x = fmaf(g[u], acc.x, a[u].x);
            acc.y = fmaf(g[u], acc.y, a[u].y);
            acc.z = fmaf(g[u], acc.z, a[u].z);
            acc.w = fmaf(g[u], acc.w, a[u].w);
          } else {
            acc.x += a[u].x;
            acc.y += a[u].y;
            acc.z += a[u].z;
            acc.w += a[u].w;
          }
        }
      }
    }
  }

  if (tiles) {
    uint8_t* tile = tiles + (size_t)h * StateTile<D>::BYTES;
    if (mine) state_tile_put<D>(tile, row, i0, acc);
    if (zpart) {  // the zero rows D + 2 .. N_S - 1 of every atom
      constexpr int Z = (StateTile<D>::NS - D - 2) * 8;  // 16-byte units per atom
      for (int u = t; u < (D / 64) * Z; u += kScanThreads)
        *reinterpret_cast<uint4*>(tile + (u / Z) * StateTile<D>::XA + (D + 2) * 128 + (u % Z) * 16) =
            make_uint4(0, 0, 0, 0);
    }
  }
  if (zpart) {
    if (mine) *reinterpret_cast<float4*>(z_N + (size_t)h * D + i0) = acc;
    return;
  }
  // S_N[h][i][r0 .. r0 + RB) through the tile
  tile[i0][row - r0] = acc.x;
  tile[i0 + 1][row - r0] = acc.y;
  tile[i0 + 2][row - r0] = acc.z;
  tile[i0 + 3][row - r0] = acc.w;
  __syncthreads();
  for (int f = 4 * t; f < D * RB; f += 4 * kScanThreads) {
    const int i = f / RB, k = f % RB;
    *reinterpret_cast<float4*>(S_N + ((size_t)h * D + i) * D + r0 + k) =
        make_float4(tile[i][k], tile[i][k + 1], tile[i][k + 2], tile[i][k + 3]);
  }
}

}  // namespace tcp
}  // namespace la
