// backward_tc64.cu -- the gradient of the causal prefill (la_prefill_backward)
// on the sm_103a tensor cores, for bf16 inputs at dk = dv = 64.
//
// Forward map (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03):
//   o_t = num_t / den_t,  num_t = phi(q_t)^T S_t,  den_t = phi(q_t)^T z_t + eps,
//   S_t = S0 + sum_{s<=t} phi(k_s) v_s^T,  z_t = z0 + sum_{s<=t} phi(k_s).
// The pages give no backward pass (the LinearMem page notes only that training
// recomputes states instead of keeping them).  With dnum_t = dO_t / den_t and
// dden_t = -(dO_t . o_t) / den_t, write W = phi(Q), U = phi(K), the C x 65
// blocks D = [dnum | dden] and V~ = [V | 1] of one chunk, S_c, z_c the state
// entering it and G_c, g_c the gradient state leaving it
// (G = dS_N + sum over later tokens of phi(q) dnum^T, g likewise with dden):
//   dW = mask(D V~^T) U + D [S_c | z_c]^T          (mask: s <= t)
//   dU = mask^T(V~ D^T) W + V~ [G_c | g_c]^T       (mask^T: tau >= t)
//   dV = mask^T(U W^T) dnum + U G_c
//   G before the chunk = G_c + W^T dnum,  g likewise with dden;
//   dS0 = G, dz0 = g before the first chunk; dq = dW phi'(q), dk = dU phi'(k).
// These are the token formulas of the CUDA-core backward gathered chunkwise.
//
// One block per head, two sweeps over its 128-token chunks:
//   forward:  recompute num and den (the prefill's products with the running
//             state in TMEM), form D, then dW = mask(D V~^T) U + D [S_c | z_c]^T
//             and dq; D (bf16) is parked in the head's rows of dv_out, which
//             the reverse sweep reads back before overwriting them with dv;
//   reverse:  from G = dS_N, g = dz_N, per chunk (last to first) dU and dV,
//             then G += W^T D on the tensor cores; finally dS0, dz0.
// The block's eight warps own the TMEM lane quadrants two by two (threads t
// and t + 128: token row t of the chunk, or state lane t, each one half of
// the row's 64 columns); one thread issues the TMA copies and the MMAs, and
// the steps of a chunk are separated by block barriers.  Every wait
// is bounded; a wait that gives up records LA_ERR_TIMEOUT in the library
// status word and the kernel finishes with unspecified outputs.
#include "prefill_tc_common.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcp;

namespace bw {

constexpr int D = 64;
constexpr uint32_t BLK = 16384;      // [128 rows x 128 B] swizzled tile
constexpr uint32_t SNAP = 80 * 128;  // [80 x 64] bf16: row j = column j of the state, 64/65 = z or g
// stage: Q | K | V | X, X = dO (fp32, two [128 x 32] boxes) in the forward
// sweep, the parked D (bf16, two [128 x 64] blocks) in the reverse sweep
constexpr uint32_t STAGE = 5 * BLK;
constexpr uint32_t OFF_DT = 2 * STAGE;        // forward: D being formed (two blocks)
constexpr uint32_t OFF_ONES = OFF_DT + 2 * BLK;
constexpr uint32_t OFF_SNAP = OFF_ONES + BLK;
constexpr uint32_t OFF_BAR = OFF_SNAP + SNAP;
constexpr uint32_t OFF_RED = OFF_BAR + 256;   // per thread: its half of a row's dot product
constexpr uint32_t SMEM = OFF_RED + 256 * 4 + 1024;
static_assert(SMEM <= 227 * 1024, "shared memory per block");
static_assert(OFF_SNAP % 1024 == 0, "swizzled tile alignment");
constexpr int kThreads = 256;  // two threads per chunk row / TMEM lane
constexpr uint32_t kCols = 512;
// TMEM columns.  Forward: A scores / P, O [num | den parts], dW, S (running
// state, lanes j).  Reverse: A2 (V~ D^T, then its mask), dU, A3 (U W^T, then
// its mask), dV, G (running gradient state, lanes j).
// Every N = 128 accumulator starts at a multiple of 128 columns, the others at
// multiples of 64.
constexpr uint32_t T_A = 0, T_O = 128, T_DW = 256, T_S = 384, T_DG = 448;
constexpr uint32_t T_A2 = 0, T_A3 = 128, T_DU = 256, T_DV = 320, T_G = 384;

constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);   // K-major x K-major, N = 128
constexpr uint32_t ID_QS = idesc_bf16_f32(128, 80, 0, 0);   // phi(Q) [S | z]
constexpr uint32_t ID_PV = idesc_bf16_f32(128, 80, 0, 1);   // P [V | 1]
constexpr uint32_t ID_N64_MN = idesc_bf16_f32(128, 64, 0, 1);  // A K-major, B MN-major, N = 64
constexpr uint32_t ID_N64_K = idesc_bf16_f32(128, 64, 0, 0);   // both K-major, N = 64
constexpr uint32_t ID_ADV = idesc_bf16_f32(128, 64, 1, 1);     // both MN-major (state advances)

constexpr int SZ = D * D + D;  // floats of a state slot: rows j = column j of the state, row 64 = z

struct Params {
  Split sp;  // pieces: whole heads (one block per head), or the split over the SMs
  int N;
  float eps;
  const float* S0;
  const float* z0;
  const float* dS_N;
  const float* dz_N;
  float* dq;
  float* dk;
  float* dv;
  float* dS0;
  float* dz0;
  unsigned* status;
  int force_wait;
  // split form: per piece slot, the entry state (from the prefill's scan), the
  // piece's gradient-state increment W^T D, and the gradient state after it
  const float* E;
  float* dG;
  const float* Gaft;
};

struct Bars {
  uint64_t full[2];  // stage loads
  uint64_t mma;      // the last MMA group complete
  uint64_t never;    // completed by nothing (the forced-timeout test hook)
  uint64_t drain;    // after a timeout: the MMAs in flight have ended
  uint32_t tmem_slot;
  int abort;
};

struct Ctx {
  const Params* p;
  Bars* B;
  unsigned long long ns;
};

// Bounded wait of one thread; false once the block has given up.
__device__ __forceinline__ bool waitb(const Ctx& x, uint64_t* bar, uint32_t parity) {
  if (*reinterpret_cast<volatile int*>(&x.B->abort)) return false;
  if (mbar_try_wait(bar, parity)) return true;
  if (mbar_wait(bar, parity, globaltimer_ns() + x.ns, reinterpret_cast<volatile int*>(&x.B->abort)))
    return true;
  x.B->abort = 1;
  atomicOr(x.p->status, kStatusTimeout);
  return false;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Half `hf` (columns 32 hf .. 32 hf + 31) of row r of a [128 x 64] bf16 tile,
// unpacked: out[i] = element 32 hf + i.
__device__ __forceinline__ void load_half_bf16(const uint8_t* tile, int r, int hf, float* out) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 u = *reinterpret_cast<const uint4*>(tile + sw128_offset(r, 4 * hf + c));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      out[8 * c + 2 * j] = __uint_as_float(w[j] << 16);
      out[8 * c + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

// Half `hf` of row r of a [128 x 64] bf16 tile from 32 floats (rounded to
// nearest even).
__device__ __forceinline__ void store_half_bf16(uint8_t* tile, int r, int hf, const float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
    u.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
    u.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
    u.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
    *reinterpret_cast<uint4*>(tile + sw128_offset(r, 4 * hf + c)) = u;
  }
}

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_row32(uint32_t taddr, float* out) {
  uint32_t a[32];
  tmem_ld32(taddr, a);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = __uint_as_float(a[i]);
}

// 32 floats into this thread's lane, columns [taddr, taddr + 32).
__device__ __forceinline__ void tmem_put32(uint32_t taddr, const float* v) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[16 * q + i]);
    tmem_st16(taddr + 16 * q, w);
  }
}

// The causal mask of a [128 x 128] fp32 score tile in TMEM (this thread's
// row t = 32 quad + lane), packed to bf16 in place over the tile's first 64
// columns: keep s <= t (lower), or s >= t (upper).  The two threads of a row
// split the columns: half hf reads column blocks 2 hf, 2 hf + 1 and writes
// packed columns [32 hf, 32 hf + 32), which half 0 reads; every thread's reads
// finish (the block barrier) before any packed column is written.  Called by
// every thread of the block.
template <bool UPPER>
__device__ __forceinline__ void mask_pack(uint32_t base, int quad, int lane, int hf) {
  uint32_t r0[32], r1[32];
  tmem_ld32(base + 64 * hf, r0);
  tmem_ld32(base + 64 * hf + 32, r1);
  tmem_ld_wait();
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int q4 = 2 * hf + h;
    const uint32_t* r = h ? r1 : r0;
    uint32_t w[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int s0 = 2 * t, s1 = 2 * t + 1;  // keys 32 q4 + s within the block
      bool k0, k1;
      if (UPPER) {
        k0 = q4 > quad || (q4 == quad && s0 >= lane);
        k1 = q4 > quad || (q4 == quad && s1 >= lane);
      } else {
        k0 = q4 < quad || (q4 == quad && s0 <= lane);
        k1 = q4 < quad || (q4 == quad && s1 <= lane);
      }
      w[t] = pack_bf16x2(k0 ? __uint_as_float(r[s0]) : 0.f, k1 ? __uint_as_float(r[s1]) : 0.f);
    }
    tmem_st16(base + 16 * q4, w);
  }
  tmem_st_wait();
}

// Row r of a float array in global memory, 32 floats from column 32 hf.
__device__ __forceinline__ void store_half_f32(float* rowp, int hf, const float* v) {
  float4* dst = reinterpret_cast<float4*>(rowp + 32 * hf);
#pragma unroll
  for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// MODE 0: one block per head, both sweeps (no workspace).  MODE 1: the
// forward sweep of every piece of the block's run, from the piece's entry
// state, also summing the piece's W^T D into dG.  MODE 2: the reverse sweep
// of every piece, from the gradient state after the piece.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
backward_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_park, const Params p,
                const unsigned long long mbar_ns) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array by pointer
  // arithmetic so that accesses through it stay shared-space accesses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* B = reinterpret_cast<Bars*>(smem + OFF_BAR);
  float* red = reinterpret_cast<float*>(smem + OFF_RED);
  const int t = threadIdx.x, warp = t / 32, lane = t % 32;
  // two threads per row: row (TMEM lane) t % 128, column half t / 128; warps w
  // and w + 4 share TMEM lane quadrant w % 4
  const int row = t & (C - 1), hf = t >> 7, quad = warp & 3;
  if (MODE != 0) pdl_launch_dependents();  // the next launch may be scheduled now
  uint8_t* dt = smem + OFF_DT;
  uint8_t* snap = smem + OFF_SNAP;
  if (t == 0) {
    mbar_init(&B->full[0], 1);
    mbar_init(&B->full[1], 1);
    mbar_init(&B->mma, 1);
    mbar_init(&B->never, 1);
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_park);
  }
  init_ones(smem + OFF_ONES, t, kThreads);  // (contains a block barrier)
  for (int i = t; i < (int)(2 * BLK / 16); i += kThreads)  // the D blocks
    reinterpret_cast<uint4*>(dt)[i] = make_uint4(0, 0, 0, 0);
  for (int i = t; i < (int)(SNAP / 16); i += kThreads)  // the snapshot (rows 66..79 stay 0)
    reinterpret_cast<uint4*>(snap)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    tmem_alloc(&B->tmem_slot, kCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot);
  const uint32_t tl = tm + ((uint32_t)(32 * quad) << 16);  // this thread's TMEM lane (row)
  const uint32_t th = 32 * hf;                              // and its column half
  const Ctx x{&p, B, mbar_ns};
  const uint32_t aOnes = smem_u32(smem + OFF_ONES), aSnap = smem_u32(snap), aDt = smem_u32(dt);
  // loads issued (thread 0) and loads consumed (every thread), in the same
  // order: load i goes to stage i % 2; MMA groups waited
  uint32_t nload = 0, nuse = 0, nmma = 0;

  // thread 0: the loads of chunk c (of head h) into stage `nload % 2`
  auto load = [&](int h, int c, bool forward) {
    const int s = nload % 2;
    uint8_t* st = smem + s * STAGE;
    const int tok = c * C;
    mbar_arrive_expect_tx(&B->full[s], 5 * BLK);
    tma_load_3d(st, &tm_q, 0, tok, h, &B->full[s]);
    tma_load_3d(st + BLK, &tm_k, 0, tok, h, &B->full[s]);
    tma_load_3d(st + 2 * BLK, &tm_v, 0, tok, h, &B->full[s]);
    if (forward) {
      tma_load_3d(st + 3 * BLK, &tm_do, 0, tok, h, &B->full[s]);
      tma_load_3d(st + 4 * BLK, &tm_do, 32, tok, h, &B->full[s]);
    } else {
      tma_load_3d(st + 3 * BLK, &tm_park, 0, tok, h, &B->full[s]);
      tma_load_3d(st + 4 * BLK, &tm_park, 64, tok, h, &B->full[s]);
    }
    ++nload;
  };
  // every thread: the MMA group thread 0 committed has completed
  auto mma_done = [&]() {
    waitb(x, &B->mma, nmma & 1);
    ++nmma;
    tc_fence_after();
  };
  // thread 0, before issuing MMAs
  auto issuing = [&]() {
    tc_fence_after();
    return !*reinterpret_cast<volatile int*>(&B->abort);
  };
  // the end of a CUDA-core step whose TMEM and shared-memory writes MMAs read
  auto step_done = [&]() {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
  };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&B->abort) != 0; };

  // =================== forward sweep of one piece ===================
  auto fwd_piece = [&](const Piece& pc) {
  const int h = pc.h, c0 = pc.tok0 / C, NC = pc.nch;
  // the entry state (S0, z0 for a whole head; the scan's E otherwise) -> the
  // running state (lane j: column j of S, lane 64: z) and its snapshot (row j;
  // rows 64, 65: z in two bf16 parts); each thread its column half
  {
    float e[32];
    if (MODE == 0) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        e[i] = row < D ? (p.S0 ? __ldg(p.S0 + ((size_t)h * D + th + i) * D + row) : 0.f)
                       : (row == D && p.z0 ? __ldg(p.z0 + (size_t)h * D + th + i) : 0.f);
    } else {
      const float* src = p.E + (size_t)pc.slot * SZ + (row <= D ? row : 0) * D + th;
#pragma unroll
      for (int i = 0; i < 32; ++i) e[i] = row <= D ? __ldcg(src + i) : 0.f;
    }
    tmem_put32(tl + T_S + th, e);
    tmem_st_wait();
    if (row < D) {
      store_half_bf16(snap, row, hf, e);
    } else if (row == D) {
      float lo[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) lo[i] = e[i] - __bfloat162float(__float2bfloat16_rn(e[i]));
      store_half_bf16(snap, D, hf, e);
      store_half_bf16(snap, D + 1, hf, lo);
    }
  }
  if (t == 0) load(h, c0, true);
  step_done();

  for (int c = 0; c < NC; ++c, ++nuse) {
    const int s = nuse % 2;
    uint8_t* st = smem + s * STAGE;
    const uint32_t aq = smem_u32(st), ak = aq + BLK, av = aq + 2 * BLK;
    const int tok = (c0 + c) * C;
    const int valid = min(C, p.N - tok);
    if (t == 0 && c + 1 < NC) load(h, c0 + c + 1, true);
    waitb(x, &B->full[s], (nuse / 2) & 1);
    phi_row<8>(st + hf * BLK, row, 0, valid);  // half 0: phi(Q), half 1: phi(K)
    step_done();

    // scores, and phi(Q) [S | z] into O
    if (t == 0 && (!p.force_wait || waitb(x, &B->never, 0)) && issuing()) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16_ss(tm + T_A, sdesc_sw128(aq + ks * 32, 16, 1024), sdesc_sw128(ak + ks * 32, 16, 1024),
                    ID_S, ks > 0);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16_ss(tm + T_O, sdesc_sw128(aq + ks * 32, 16, 1024), sdesc_sw128(aSnap + ks * 32, 16, 1024),
                    ID_QS, ks > 0);
    }
    if (t == 0) mma_commit(&B->mma);
    mma_done();
    mask_pack<false>(tl + T_A, quad, lane, hf);
    step_done();

    // O += P [V | 1]
    if (t == 0 && issuing()) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        mma_bf16_ts(tm + T_O, tm + T_A + 8 * ks, sdesc_sw128(av + ks * 2048, aOnes - av, 1024), ID_PV, 1u);
    }
    if (t == 0) mma_commit(&B->mma);
    mma_done();
    {  // den, o, then D = [dnum | dden] of the row; this thread's column half of dnum
      uint32_t nr[32], d2[2];
      tmem_ld32(tl + T_O + th, nr);
      tmem_ld2(tl + T_O + D, d2);
      tmem_ld_wait();
      const float den = __uint_as_float(d2[0]) + __uint_as_float(d2[1]) + p.eps;
      const float inv = 1.f / den;
      float dn[32], dot = 0.f;
      const uint8_t* x0 = st + 3 * BLK + hf * BLK;  // dO columns 32 hf .. 32 hf + 31
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const float4 g4 = *reinterpret_cast<const float4*>(x0 + sw128_offset(row, cc));
        const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          dot += gv[j] * (__uint_as_float(nr[4 * cc + j]) * inv);
          dn[4 * cc + j] = gv[j] * inv;
        }
      }
      red[t] = dot;
      store_half_bf16(dt, row, hf, dn);
      __syncthreads();
      const float dden = -(red[row] + red[row + C]) * inv;
      if (hf == 0)
        *reinterpret_cast<uint4*>(dt + BLK + sw128_offset(row, 0)) = make_uint4(pack_bf16x2(dden, dden), 0u, 0u, 0u);
      // parked in dv's row (256 bytes): 64 bf16 dnum, then dden twice and zeros,
      // the row-major form the reverse sweep's tile loads read back
      if (row < valid) {
        uint4* prow = reinterpret_cast<uint4*>(p.dv + ((size_t)h * p.N + tok + row) * D);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          prow[4 * hf + q] = make_uint4(pack_bf16x2(dn[8 * q], dn[8 * q + 1]), pack_bf16x2(dn[8 * q + 2], dn[8 * q + 3]),
                                        pack_bf16x2(dn[8 * q + 4], dn[8 * q + 5]), pack_bf16x2(dn[8 * q + 6], dn[8 * q + 7]));
        if (hf == 0) {
          prow[8] = make_uint4(pack_bf16x2(dden, dden), 0u, 0u, 0u);
        } else {
#pragma unroll
          for (int q = 9; q < 16; ++q) prow[q] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    step_done();

    // A = D V~^T, dW = D [S | z]^T; D goes to dv_out to wait for the reverse sweep
    if (t == 0 && issuing()) {
#pragma unroll
      for (int ks = 0; ks < 5; ++ks) {
        const uint32_t a = ks < 4 ? aDt + ks * 32 : aDt + BLK;
        const uint32_t b = ks < 4 ? av + ks * 32 : aOnes;
        mma_bf16_ss(tm + T_A, sdesc_sw128(a, 16, 1024), sdesc_sw128(b, 16, 1024), ID_S, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 5; ++ks) {
        const uint32_t a = ks < 4 ? aDt + ks * 32 : aDt + BLK;
        mma_bf16_ss(tm + T_DW, sdesc_sw128(a, 16, 1024), sdesc_sw128(aSnap + ks * 2048, 16, 1024),
                    ID_N64_MN, ks > 0);
      }
    }
    if (t == 0) mma_commit(&B->mma);
    mma_done();
    mask_pack<false>(tl + T_A, quad, lane, hf);
    step_done();

    // dW += mask(A) U;  S += [V | 1]^T U
    if (t == 0 && issuing()) {
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        mma_bf16_ts(tm + T_DW, tm + T_A + 8 * ks, sdesc_sw128(ak + ks * 2048, BLK, 1024), ID_N64_MN, 1u);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        mma_bf16_ss(tm + T_S, sdesc_sw128(av + ks * 2048, aOnes - av, 1024),
                    sdesc_sw128(ak + ks * 2048, BLK, 1024), ID_ADV, 1u);
      if (MODE == 1) {  // the piece's gradient-state increment W^T D (lanes j)
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks)
          mma_bf16_ss(tm + T_DG, sdesc_sw128(aDt + ks * 2048, BLK, 1024), sdesc_sw128(aq + ks * 2048, BLK, 1024),
                      ID_ADV, (c > 0 || ks > 0) ? 1u : 0u);
      }
    }
    if (t == 0) mma_commit(&B->mma);
    mma_done();
    {  // dq = dW phi'(q), phi'(u) = min(phi(u), 1); the state snapshot for the next chunk
      float g[32], f[32];
      tmem_row32(tl + T_DW + th, g);
      load_half_bf16(st, row, hf, f);
      if (row < valid && !aborted()) {
#pragma unroll
        for (int i = 0; i < 32; ++i) g[i] *= fminf(f[i], 1.f);
        store_half_f32(p.dq + ((size_t)h * p.N + tok + row) * D, hf, g);
      }
      if (c + 1 < NC && quad <= 2) {  // whole warps: tcgen05.ld is warp-collective
        float e[32];
        tmem_row32(tl + T_S + th, e);
        if (row < D) store_half_bf16(snap, row, hf, e);
        if (row == D) {
          store_half_bf16(snap, D, hf, e);
#pragma unroll
          for (int i = 0; i < 32; ++i) e[i] -= __bfloat162float(__float2bfloat16_rn(e[i]));
          store_half_bf16(snap, D + 1, hf, e);
        }
      }
    }
    step_done();
  }
  if (MODE == 1 && quad <= 2) {  // whole warps: tcgen05.ld is warp-collective
    float e[32];
    tmem_row32(tl + T_DG + th, e);
    if (row <= D && !aborted()) {
      float4* dst = reinterpret_cast<float4*>(p.dG + (size_t)pc.slot * SZ + row * D + th);
#pragma unroll
      for (int q = 0; q < 8; ++q) __stcg(dst + q, make_float4(e[4 * q], e[4 * q + 1], e[4 * q + 2], e[4 * q + 3]));
    }
  }
  step_done();
  };

  // =================== reverse sweep of one piece ===================
  auto rev_piece = [&](const Piece& pc) {
  const int h = pc.h, c0 = pc.tok0 / C, NC = pc.nch;
  // the gradient state after the piece (dS_N, dz_N for a whole head; the
  // reverse scan's otherwise) -> the running gradient state (lane j: column j
  // of G, lane 64: g) and its snapshot (row j; row 64: g; row 65 stays 0)
  {
    float e[32];
    if (MODE == 0) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        e[i] = row < D ? (p.dS_N ? __ldg(p.dS_N + ((size_t)h * D + th + i) * D + row) : 0.f)
                       : (row == D && p.dz_N ? __ldg(p.dz_N + (size_t)h * D + th + i) : 0.f);
    } else {
      const float* src = p.Gaft + (size_t)pc.slot * SZ + (row <= D ? row : 0) * D + th;
#pragma unroll
      for (int i = 0; i < 32; ++i) e[i] = row <= D ? __ldcg(src + i) : 0.f;
    }
    tmem_put32(tl + T_G + th, e);
    tmem_st_wait();
    if (row <= D) store_half_bf16(snap, row, hf, e);
    if (row == D + 1) {
#pragma unroll
      for (int i = 0; i < 32; ++i) e[i] = 0.f;
      store_half_bf16(snap, D + 1, hf, e);
    }
  }
  step_done();  // (also: every thread's parked rows are fenced before the first tile load)
  if (t == 0) load(h, c0 + NC - 1, false);

  for (int r = 0; r < NC; ++r, ++nuse) {
    const int c = NC - 1 - r;
    const int s = nuse % 2;
    uint8_t* st = smem + s * STAGE;
    const uint32_t aq = smem_u32(st), ak = aq + BLK, av = aq + 2 * BLK, ax = aq + 3 * BLK;
    const int tok = (c0 + c) * C;
    const int valid = min(C, p.N - tok);
    if (t == 0 && c > 0) load(h, c0 + c - 1, false);
    waitb(x, &B->full[s], (nuse / 2) & 1);
    phi_row<8>(st + hf * BLK, row, 0, valid);  // half 0: phi(Q), half 1: phi(K)
    step_done();

    // A2 = V~ D^T, dU = V~ [G | g]^T, A3 = U W^T, dV = U G
    if (t == 0 && issuing()) {
#pragma unroll
      for (int ks = 0; ks < 5; ++ks) {
        const uint32_t a = ks < 4 ? av + ks * 32 : aOnes;
        const uint32_t b = ks < 4 ? ax + ks * 32 : ax + BLK;
        mma_bf16_ss(tm + T_A2, sdesc_sw128(a, 16, 1024), sdesc_sw128(b, 16, 1024), ID_S, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 5; ++ks) {
        const uint32_t a = ks < 4 ? av + ks * 32 : aOnes;
        mma_bf16_ss(tm + T_DU, sdesc_sw128(a, 16, 1024), sdesc_sw128(aSnap + ks * 2048, 16, 1024),
                    ID_N64_MN, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16_ss(tm + T_A3, sdesc_sw128(ak + ks * 32, 16, 1024), sdesc_sw128(aq + ks * 32, 16, 1024),
                    ID_S, ks > 0);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16_ss(tm + T_DV, sdesc_sw128(ak + ks * 32, 16, 1024), sdesc_sw128(aSnap + ks * 32, 16, 1024),
                    ID_N64_K, ks > 0);
    }
    if (t == 0) mma_commit(&B->mma);
    mma_done();
    mask_pack<true>(tl + T_A2, quad, lane, hf);
    mask_pack<true>(tl + T_A3, quad, lane, hf);
    step_done();

    // dU += mask^T(A2) W, dV += mask^T(A3) dnum, G += W^T D
    if (t == 0 && issuing()) {
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        mma_bf16_ts(tm + T_DU, tm + T_A2 + 8 * ks, sdesc_sw128(aq + ks * 2048, BLK, 1024), ID_N64_MN, 1u);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        mma_bf16_ts(tm + T_DV, tm + T_A3 + 8 * ks, sdesc_sw128(ax + ks * 2048, BLK, 1024), ID_N64_MN, 1u);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        mma_bf16_ss(tm + T_G, sdesc_sw128(ax + ks * 2048, BLK, 1024), sdesc_sw128(aq + ks * 2048, BLK, 1024),
                    ID_ADV, 1u);
    }
    if (t == 0) mma_commit(&B->mma);
    mma_done();
    {  // dk = dU phi'(k), dv; the gradient-state snapshot for the chunk before
      float g[32], f[32];
      tmem_row32(tl + T_DU + th, g);
      load_half_bf16(st + BLK, row, hf, f);
      const bool out = row < valid && !aborted();
      if (out) {
#pragma unroll
        for (int i = 0; i < 32; ++i) g[i] *= fminf(f[i], 1.f);
        store_half_f32(p.dk + ((size_t)h * p.N + tok + row) * D, hf, g);
      }
      tmem_row32(tl + T_DV + th, g);
      if (out) store_half_f32(p.dv + ((size_t)h * p.N + tok + row) * D, hf, g);
      if (quad <= 2) {  // whole warps: tcgen05.ld is warp-collective; lanes 0..64 are kept
        float e[32];
        tmem_row32(tl + T_G + th, e);
        if (c > 0 && row <= D) store_half_bf16(snap, row, hf, e);
        if (MODE == 0 && c == 0 && row <= D && !aborted()) {  // dS0, dz0
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (row < D) {
              if (p.dS0) p.dS0[((size_t)h * D + th + i) * D + row] = e[i];
            } else if (p.dz0) {
              p.dz0[(size_t)h * D + th + i] = e[i];
            }
          }
        }
      }
    }
    step_done();
  }
  };

  const Run run(p.sp, blockIdx.x);
  Piece pc;
  if (MODE == 0) {  // the block's head: forward sweep, then reverse sweep
    if (run.piece(p.sp, 0, &pc)) {
      fwd_piece(pc);
      // every thread's parked rows are written before the tile loads read them
      __threadfence();
      fence_proxy_async_global();
      rev_piece(pc);
    }
  } else {
    pdl_wait();  // the entry (gradient) states come from the launches before
    for (int i = 0; run.piece(p.sp, i, &pc); ++i) {
      if (MODE == 1) fwd_piece(pc);
      else rev_piece(pc);
    }
  }

  if (t == 0 && aborted()) {  // MMAs in flight end first
    int never = 0;
    mma_commit(&B->drain);
    mbar_wait(&B->drain, 0, globaltimer_ns() + mbar_ns, &never);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, kCols);
  }
}

// The gradient state after every piece of a head, from the last piece back:
// G_after(last) = dS_N (z: dz_N), G_after(p) = G_after(p + 1) + dG(p + 1); what
// remains after the first piece is dS0, dz0.  One thread per slot element.
constexpr int kScanThreads = 256;

__global__ void __launch_bounds__(kScanThreads) gscan_kernel(const Params p, float* Gaft) {
  pdl_launch_dependents();  // the reverse sweep may be scheduled now
  pdl_wait();               // dG of every piece is complete
  const int e = blockIdx.x * kScanThreads + threadIdx.x;  // slot element: row * 64 + i
  const int h = blockIdx.y;
  if (e >= SZ) return;
  const Split& s = p.sp;
  const int row = e / D, i = e % D;  // row < 64: G[i][row]; row 64: g[i]
  float acc = 0.f;
  if (row < D) {
    if (p.dS_N) acc = p.dS_N[((size_t)h * D + i) * D + row];
  } else if (p.dz_N) {
    acc = p.dz_N[(size_t)h * D + i];
  }
  const int first = s.owner((long long)h * s.NC);
  const int npieces = s.owner((long long)(h + 1) * s.NC - 1) - first + 1;
  const size_t base = (size_t)h * s.MPH * SZ + e;
  constexpr int U = 8;
  for (int w1 = npieces; w1 > 0; w1 -= U) {  // pieces w1 - 1, w1 - 2, ... (eight at a time)
    float a[U];
#pragma unroll
    for (int u = 0; u < U; ++u) a[u] = (w1 - 1 - u >= 0) ? __ldcg(p.dG + base + (size_t)(w1 - 1 - u) * SZ) : 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (w1 - 1 - u >= 0) {
        __stcg(Gaft + base + (size_t)(w1 - 1 - u) * SZ, acc);
        acc += a[u];
      }
    }
  }
  if (row < D) {
    if (p.dS0) p.dS0[((size_t)h * D + i) * D + row] = acc;
  } else if (p.dz0) {
    p.dz0[(size_t)h * D + i] = acc;
  }
}

}  // namespace bw
}  // namespace

bool backward_tc64_supported(const PrefillArgs& a) {
  return a.bf16 && a.dk == 64 && a.dv == 64 && a.N > 0 && get_encode() != nullptr;
}

// The split form's workspace: agg, E, dG and G-after slots, S_N and z_N
// scratch for the prefill's scan.
size_t backward_tc64_workspace_bytes(int B, int H, int N) {
  using namespace bw;
  if (prefill_prefix64_chosen(B, H, N)) return backward_prefix64_workspace_bytes(B, H, N);
  const Split s = make_split(B * H, N, sm_count());
  const size_t slots = (size_t)s.BH * s.MPH;
  return (4 * slots + s.BH) * SZ * sizeof(float);
}

cudaError_t launch_backward_tc64(const PrefillArgs& a, const float* dO, const float* dS_N,
                                 const float* dz_N, float* dq, float* dk, float* dv, float* dS0,
                                 float* dz0, cudaStream_t stream) {
  using namespace bw;
  const int BH = a.B * a.H;
  CUtensorMap mq, mk, mv, mdo, mpark;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mdo, dO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C) ||
      // dv's rows seen as 128 bf16 each: two [128 x 64] blocks of D per chunk
      !make_map(&mpark, dv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2 * D, a.N, BH, 64, C))
    return cudaErrorInvalidValue;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const bool split = a.workspace && a.ws_bytes >= backward_tc64_workspace_bytes(a.B, a.H, a.N);
  if (split && prefill_prefix64_chosen(a.B, a.H, a.N))  // chunk-parallel, four launches
    return launch_backward_prefix64(a, dO, dS_N, dz_N, dq, dk, dv, dS0, dz0, stream);
  Params p = {};
  p.sp = make_split(BH, a.N, split ? sms : BH);  // without a workspace, block j runs head j
  p.N = a.N;
  p.eps = a.eps;
  p.S0 = a.S0;
  p.z0 = a.z0;
  p.dS_N = dS_N;
  p.dz_N = dz_N;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dS0 = dS0;
  p.dz0 = dz0;
  cudaError_t e = library_status_word(&p.status);
  if (e != cudaSuccess) return e;
  p.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  if (!split) {
    e = cudaFuncSetAttribute(backward_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
    if (e != cudaSuccess) return e;
    backward_kernel<0><<<p.sp.G, kThreads, SMEM, stream>>>(mq, mk, mv, mdo, mpark, p, mbar_ns);
    return cudaGetLastError();
  }
  const size_t slots = (size_t)BH * p.sp.MPH;
  float* agg = static_cast<float*>(a.workspace);
  float* E = agg + slots * SZ;
  float* dG = E + slots * SZ;
  float* Gaft = dG + slots * SZ;
  float* SNz = Gaft + slots * SZ;  // S_N (BH x 64 x 64), then z_N (BH x 64)
  p.E = E;
  p.dG = dG;
  p.Gaft = Gaft;
  // the prefill's aggregate and scan: every piece's entry state
  e = launch_prefill_entry_states64(a, agg, E, SNz, SNz + (size_t)BH * D * D, p.status, stream);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(backward_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(backward_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
  if (e != cudaSuccess) return e;
  // forward sweeps, the reverse scan of the gradient state, reverse sweeps:
  // programmatic dependents, each waiting for the launch before it
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SMEM;
  e = cudaLaunchKernelEx(&cfg, backward_kernel<1>, mq, mk, mv, mdo, mpark, p, mbar_ns);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((SZ + kScanThreads - 1) / kScanThreads, BH);
  cfg.blockDim = dim3(kScanThreads);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, gscan_kernel, p, Gaft);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SMEM;
  return cudaLaunchKernelEx(&cfg, backward_kernel<2>, mq, mk, mv, mdo, mpark, p, mbar_ns);
}

}  // namespace la
