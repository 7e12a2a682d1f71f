// prefill_decay.cuh -- pieces of the decayed prefill (S_t = alpha_t S_{t-1} +
// phi(k_t) v_t^T, page "线性注意力与SSM", sections 3-4) shared by the
// three-launch forms at d = 64 and d = 128: the floor on alpha, and the row
// scalings of bf16 operand tiles by decay weights.
#pragma once

#include "prefill_tc_common.cuh"

namespace la {
namespace tcp {

constexpr float kAlphaMin = 1e-30f;  // a zero decay is taken as this (its log2 stays finite)

// Row r of a bf16 [128 x 64] swizzled tile, times f, rounded to bf16 again.
__device__ __forceinline__ void scale_row(uint8_t* tile, int r, float f) {
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = *reinterpret_cast<const uint4*>(tile + tc::sw128_offset(r, i));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t* w = reinterpret_cast<uint32_t*>(&v[i]);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      w[j] = tc::pack_bf16x2(__uint_as_float(w[j] << 16) * f, __uint_as_float(w[j] & 0xFFFF0000u) * f);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(tile + tc::sw128_offset(r, i)) = v[i];
}

// phi_row followed by scale_row on `nchunk` 16-byte chunks of row r from
// chunk c0, in one pass (the same two roundings to bf16, one shared-memory
// round trip).
template <int NCH>
__device__ __forceinline__ void phi_scale_row(uint8_t* tile, int r, int c0, int valid, float f) {
  uint4 v[NCH];
#pragma unroll
  for (int i = 0; i < NCH; ++i) v[i] = *reinterpret_cast<const uint4*>(tile + tc::sw128_offset(r, c0 + i));
  const uint32_t keep = r < valid ? 0xFFFFFFFFu : 0u;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    uint32_t* w = reinterpret_cast<uint32_t*>(&v[i]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t y = phi2(w[j]) & keep;
      w[j] = tc::pack_bf16x2(__uint_as_float(y << 16) * f, __uint_as_float(y & 0xFFFF0000u) * f);
    }
  }
#pragma unroll
  for (int i = 0; i < NCH; ++i) *reinterpret_cast<uint4*>(tile + tc::sw128_offset(r, c0 + i)) = v[i];
}

}  // namespace tcp
}  // namespace la
