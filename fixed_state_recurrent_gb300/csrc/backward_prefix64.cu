// backward_prefix64.cu -- the gradient of the causal prefill (la_prefill_backward)
// for bf16 inputs at dk = dv = 64, chunk-parallel on the sm_103a tensor cores,
// for calls whose intermediates stay in L2 (those of the two-launch prefill).
//
// Forward map (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03):
//   o_t = num_t / den_t,  num_t = phi(q_t)^T S_t,  den_t = phi(q_t)^T z_t + eps,
//   S_t = S0 + sum_{s<=t} phi(k_s) v_s^T,  z_t = z0 + sum_{s<=t} phi(k_s).
// The pages give no backward pass (the LinearMem page notes only that training
// recomputes states instead of keeping them).  With dnum_t = dO_t / den_t and
// dden_t = -(dO_t . o_t) / den_t, W = phi(Q), U = phi(K) of a 128-token chunk,
// S_c, z_c the state entering it and G_c, g_c the gradient state leaving it
// (G = dS_N + sum over later tokens of phi(q) dnum^T, g likewise with dden):
//   dW_t = sum_{s<=t} (dnum_t . v_s + dden_t) U_s + S_c dnum_t + dden_t z_c
//   dU_s = sum_{t>=s} (v_s . dnum_t + dden_t) W_t + G_c v_s + g_c
//   dV_s = sum_{t>=s} (U_s . W_t) dnum_t + G_c^T U_s
//   G before the chunk = G_c + W^T dnum,  g likewise with dden;
//   dS0 = G, dz0 = g before the first chunk; dq = dW phi'(q), dk = dU phi'(k),
//   phi'(u) = min(phi(u), 1).
// The dden terms are rank one (a row or column constant of a score tile, a
// vector added to a row), so they are added in fp32 on the CUDA cores and every
// product contracts over 64 or 128 without an extra operand block.
//
// Four launches over the split of prefill_tc_common.cuh (block j takes a run
// of the head-major chunk sequence, cut at head boundaries into pieces), none
// with a chain from chunk to chunk:
//   1, 2. the two launches of the prefill (prefill_prefix64.cu): per chunk the
//      prefix tile of the state before it (relative to the piece's entry),
//      piece totals, phi(K); then o (into the workspace) and den.
//   3. gprefix_kernel: per chunk D = [dnum | dden] from o, den and dO, phi(Q),
//      and the increment [dnum | dden]^T phi(Q) on the tensor cores, summed in
//      fp32 registers from each piece's last chunk back to its first: the tile
//      of the gradient state after every chunk (relative to the piece's exit,
//      with dS_N, dz_N for a piece that ends its head) and piece totals.
//      phi(Q) and dnum (bf16) and dden (fp32) go to the workspace.
//   4. grad_kernel: per chunk, from the state tiles (plus the sum of the
//      head's earlier blocks' totals for the block's first piece, and of its
//      later blocks' gradient totals for the last), the scores D V^T, V D^T
//      and U W^T with their masks, dq, dk and dv; dS0, dz0 from the gradient
//      totals.
// Every wait is bounded; one that gives up records a timeout in the library
// status word and the kernel finishes with unspecified outputs.
#include "prefill_tc_common.cuh"

#ifdef LA_TRACE
static __device__ unsigned long long g_bw_trace[2 * 160 * 64];
#define BW_TRACE(kern, ev)                                                              \
  do {                                                                                 \
    if ((ev) < 64 && blockIdx.x < 160)                                                 \
      g_bw_trace[((kern) * 160 + blockIdx.x) * 64 + (ev)] = la::tc::globaltimer_ns();  \
  } while (0)
extern "C" int la_backward64_trace_read(unsigned long long* host, int n) {
  return cudaMemcpyFromSymbol(host, g_bw_trace, (size_t)n * 8) == cudaSuccess ? 0 : -1;
}
extern "C" int la_backward64_trace_clear() {
  static unsigned long long zeros[2 * 160 * 64];
  return cudaMemcpyToSymbol(g_bw_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#else
#define BW_TRACE(kern, ev) ((void)0)
#endif

namespace la {
namespace {

using namespace tc;
using namespace tcp;

constexpr int D = 64;
constexpr int SZ = D * D + D;           // floats per state slot (transposed rows, then the vector)
constexpr uint32_t BLK = 16384;         // [128 rows x 128 B] swizzled tile
constexpr int XROWS = 66;               // rows of a state tile in the workspace
constexpr uint32_t XG = XROWS * 128;    // its bytes
constexpr uint32_t XT = 80 * 128;       // room for one in shared memory

constexpr uint64_t kStepK16 = 32 >> 4;       // K-major operand: the next 16 elements along K
constexpr uint64_t kStepRows16 = 2048 >> 4;  // MN-major operand: the next 16 rows along K

struct Ctx {
  unsigned* status;
  volatile int* abort;
  uint32_t tmem;
  unsigned long long mbar_ns;
};

// Bounded wait; false once the block has given up (this wait ran out of time
// and recorded it, or another role's did).
__device__ __forceinline__ bool waitb(const Ctx& x, uint64_t* bar, uint32_t parity) {
  if (*x.abort) return false;
  if (mbar_try_wait(bar, parity)) return true;
  if (mbar_wait(bar, parity, globaltimer_ns() + x.mbar_ns, x.abort)) return true;
  *x.abort = 1;
  atomicOr(x.status, kStatusTimeout);
  return false;
}

__device__ __forceinline__ bool waitb_warp(const Ctx& x, uint64_t* bar, uint32_t parity) {
  return __all_sync(0xFFFFFFFFu, waitb(x, bar, parity));
}

// Producer drain: the last loads that were issued (at most NS_) land before the
// block leaves.
template <int NS_>
__device__ __forceinline__ void drain_loads(uint64_t* full, uint32_t issued, unsigned long long ns) {
  int never = 0;
  const uint64_t dl = globaltimer_ns() + ns;
  for (uint32_t q = (issued > NS_ ? issued - NS_ : 0); q < issued; ++q)
    mbar_wait(&full[q % NS_], (q / NS_) & 1, dl, &never);
}

// Eight bf16 of one state row, K-major swizzled operand tile.
__device__ __forceinline__ void put8(uint8_t* tile, int row, int chunk, const float* v) {
  *reinterpret_cast<uint4*>(tile + sw128_offset(row, chunk)) =
      make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                 pack_bf16x2(v[6], v[7]));
}

// Plain bulk copy global -> shared of `bytes` (a multiple of 16; both addresses
// 16-byte aligned), completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Element (row, col) of a [rows x 64] bf16 swizzled tile, widened.
__device__ __forceinline__ float tile_at(const uint8_t* tile, int row, int col) {
  const uint16_t b = *reinterpret_cast<const uint16_t*>(tile + sw128_offset(row, col / 8) + (col % 8) * 2);
  return __uint_as_float((uint32_t)b << 16);
}

// ===========================================================================
// 3. D, phi(Q) and the gradient-state tiles

namespace gpx {

constexpr int NS = 3;
// stage: Q | o (bf16 tile) | dO (two [128 x 32] fp32 boxes).  The D warps
// overwrite Q with phi(Q), o with dnum (bf16 tile) and dO's second box with
// the dden block (column 0 = dden, the rest zero): the A operand
// [dnum | dden] of the increment, M = 128 over its two 64-column blocks
// (2 * BLK apart).
constexpr uint32_t OFF_O = BLK;
constexpr uint32_t OFF_DO = 2 * BLK;
constexpr uint32_t OFF_DD = OFF_DO + BLK;
constexpr uint32_t STAGE = 4 * BLK;
constexpr uint32_t PST = 9 * 1024;          // staging of one state tile (66 rows)
constexpr uint32_t OFF_PST = NS * STAGE;
constexpr uint32_t OFF_BAR = OFF_PST + 2 * PST;
constexpr uint32_t SMEM = OFF_BAR + 512 + 1024;
static_assert(PST >= XG && OFF_PST % 1024 == 0 && PST % 1024 == 0, "tile staging");
static_assert(SMEM <= 227 * 1024, "shared memory per block");
// 0 TMA, 1 MMA, 2-9 phi(Q) and D (half a row per thread), 10-13 the running
// gradient state (TMEM lanes 0..64 on warps 10, 12, 13), 14 phi(Q) and dnum stores
constexpr int kWarps = 15;
constexpr int NB = 4;                        // TMEM increment buffers, 64 columns each
constexpr uint32_t kCols = 256;
constexpr uint32_t ID_DG = idesc_bf16_f32(128, D, 1, 1);  // [dnum | dden]^T phi(Q)

struct Params {
  Split sp;
  const float* dS_N;  // [BH][64][64] or NULL
  const float* dz_N;  // [BH][64] or NULL
  const float* den;   // [BH][N]: den_t of the prefill
  float* dden;        // [BH * NC][128] out: dden of every chunk row (0 past the sequence)
  float* RG;          // [BH * MPH][SZ] gradient totals of the pieces (slot layout)
  unsigned* status;
};

struct Bars {
  uint64_t full[NS], xf[NS];
  uint64_t empty[NS];    // the stage's product done and its stores read: 2 arrivals
  uint64_t dsready[NB];  // increment in buffer b (MMA -> state warps)
  uint64_t dsfree[NB];   // buffer b read out (three state warps -> MMA)
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
  float4 zbuf[16];       // g, handed from its TMEM lane to the whole warp
};
static_assert(sizeof(Bars) <= 512, "barrier area");

// Chunks are taken piece by piece, each piece from its last chunk back to its
// first; every role walks them in this order.
__global__ void __launch_bounds__(32 * kWarps, 1)
gprefix_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
               const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_phiq,
               const __grid_constant__ CUtensorMap tm_dn, const __grid_constant__ CUtensorMap tm_gt,
               const Params p, const unsigned long long mbar_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* B = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Run run(p.sp, blockIdx.x);
  const int N = p.sp.N;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&B->full[s], 1);
      mbar_init(&B->xf[s], 8);
      mbar_init(&B->empty[s], 2);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&B->dsready[b], 1);
      mbar_init(&B->dsfree[b], 3);
    }
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_o);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_phiq);
    tma_prefetch_desc(&tm_dn);
    tma_prefetch_desc(&tm_gt);
  }
  if (warp == 1) {
    tmem_alloc(&B->tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const Ctx x{p.status, &B->abort, *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot), mbar_ns};
  if (threadIdx.x == 0) BW_TRACE(1, 0);
  pdl_launch_dependents();  // the gradient kernel may be scheduled now; it waits for this grid
  pdl_wait();               // o and den of the output kernel are complete
  if (threadIdx.x == 0) BW_TRACE(1, 1);

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer: Q, o, dO
      uint32_t sj = 0, issued = 0;
      Piece pc;
      for (int i = 0; run.piece(p.sp, i, &pc); ++i)
        for (int r = 0; r < pc.nch; ++r, ++sj) {
          const int c = pc.nch - 1 - r, s = sj % NS;
          if (sj >= NS && !waitb(x, &B->empty[s], ((sj / NS) - 1) & 1)) break;
          uint8_t* st = smem + s * STAGE;
          const int tok = pc.tok0 + c * C;
          mbar_arrive_expect_tx(&B->full[s], 4 * BLK);
          tma_load_3d_ef(st, &tm_q, 0, tok, pc.h, &B->full[s]);
          tma_load_3d_ef(st + OFF_O, &tm_o, 0, tok, pc.h, &B->full[s]);
          tma_load_3d_ef(st + OFF_DO, &tm_do, 0, tok, pc.h, &B->full[s]);
          tma_load_3d_ef(st + OFF_DO + BLK, &tm_do, 32, tok, pc.h, &B->full[s]);
          ++issued;
        }
      if (*x.abort) drain_loads<NS>(B->full, issued, mbar_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA: increment b = [dnum | dden]^T phi(Q), fresh per chunk
      const uint32_t total = (uint32_t)(run.b - run.a);
      for (uint32_t j = 0; j < total; ++j) {
        const int s = j % NS, b = j % NB;
        if (j >= NB && !waitb(x, &B->dsfree[b], ((j / NB) - 1) & 1)) break;
        if (!waitb(x, &B->xf[s], (j / NS) & 1)) break;
        if (j < 16) BW_TRACE(1, 2 + j);
        tc_fence_after();
        const uint32_t qt = smem_u32(smem + s * STAGE), dn = qt + OFF_O;
        const uint64_t a0 = sdesc_sw128(dn, OFF_DD - OFF_O, 1024), b0 = sdesc_sw128(qt, BLK, 1024);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks)
          mma_bf16_ss(x.tmem + 64 * b, a0 + ks * kStepRows16, b0 + ks * kStepRows16, ID_DG, ks > 0 ? 1u : 0u);
        mma_commit(&B->empty[s]);
        mma_commit(&B->dsready[b]);
      }
      if (*x.abort) {
        int never = 0;
        mma_commit(&B->drain);
        mbar_wait(&B->drain, 0, globaltimer_ns() + mbar_ns, &never);
      }
    }
    __syncwarp();
  } else if (warp < 10) {
    // ---- phi(Q) in place and D, half a tile row per thread (the two halves of
    // row r are adjacent lanes)
    const int t = threadIdx.x - 64, r = t >> 1, hf = t & 1;
    uint32_t sj = 0;
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i)
      for (int rr = 0; rr < pc.nch; ++rr, ++sj) {
        const int c = pc.nch - 1 - rr, s = sj % NS;
        const int tok = pc.tok0 + c * C, valid = pc.tok1 - tok;
        const float den = r < valid ? __ldcg(p.den + (size_t)pc.h * N + tok + r) : 1.f;
        if (!waitb_warp(x, &B->full[s], (sj / NS) & 1)) continue;
        uint8_t* st = smem + s * STAGE;
        phi_row<4>(st, r, 4 * hf, valid);
        // this thread's 32 columns of o (chunks 4 hf.. of its bf16 row) and of
        // dO (box hf)
        const uint8_t* gb = st + OFF_DO + hf * BLK;
        float g[32], dot = 0.f;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const float4 g4 = *reinterpret_cast<const float4*>(gb + sw128_offset(r, cc));
          g[4 * cc] = g4.x;
          g[4 * cc + 1] = g4.y;
          g[4 * cc + 2] = g4.z;
          g[4 * cc + 3] = g4.w;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 u = *reinterpret_cast<const uint4*>(st + OFF_O + sw128_offset(r, 4 * hf + q));
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dot += __uint_as_float(w4[e] << 16) * g[8 * q + 2 * e] +
                   __uint_as_float(w4[e] & 0xFFFF0000u) * g[8 * q + 2 * e + 1];
        }
        dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 1);
        const float inv = r < valid ? 1.f / den : 0.f;
        const float dden = -dot * inv;
#pragma unroll
        for (int e = 0; e < 32; ++e) g[e] *= inv;
        uint8_t* dn = st + OFF_O;  // dnum over the bytes of o this thread read
#pragma unroll
        for (int q = 0; q < 4; ++q) put8(dn, r, 4 * hf + q, g + 8 * q);
        if (hf == 1) {  // the dden block's row r, over the row of dO's box 1 this thread read
          uint8_t* db = st + OFF_DD;
          *reinterpret_cast<uint4*>(db + sw128_offset(r, 0)) = make_uint4(pack_bf16x2(dden, 0.f), 0u, 0u, 0u);
#pragma unroll
          for (int q = 1; q < 8; ++q) *reinterpret_cast<uint4*>(db + sw128_offset(r, q)) = make_uint4(0u, 0u, 0u, 0u);
        } else if (!*x.abort) {  // rows past the sequence: 0
          p.dden[((size_t)pc.h * p.sp.NC + pc.tok0 / C + c) * C + r] = dden;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->xf[s]);
      }
  } else if (warp < 14) {
    // ---- the running gradient state.  State lane `row` (0..64: quadrants
    // 0..2) holds slot row `row` in fp32 (row j < 64: column j of G; row 64:
    // g).  Per chunk: the state after it as a bf16 tile (rows 64, 65: g in two
    // parts), staged and stored by TMA (thread 352); then the chunk's
    // increment out of TMEM added.  After a piece's first chunk its total.
    const int quad = warp % 4, row = 32 * quad + lane, et = threadIdx.x - 320;
    const bool state_warp = quad <= 2;
    const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
    float acc[D];
    uint32_t sj = 0;
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i) {
      // a piece that ends its head starts from dS_N, dz_N
#pragma unroll
      for (int q = 0; q < D; ++q) acc[q] = 0.f;
      if (state_warp && pc.tok1 == N) {
        if (row < D && p.dS_N) {
#pragma unroll
          for (int q = 0; q < D; ++q) acc[q] = __ldg(p.dS_N + ((size_t)pc.h * D + q) * D + row);
        } else if (row == D && p.dz_N) {
#pragma unroll
          for (int q = 0; q < D; ++q) acc[q] = __ldg(p.dz_N + (size_t)pc.h * D + q);
        }
      }
      for (int rr = 0; rr < pc.nch; ++rr, ++sj) {
        const int c = pc.nch - 1 - rr;
        uint8_t* stg = smem + OFF_PST + (sj % 2) * PST;
        if (et == 32 && sj >= 2) bulk_wait_read_but_one();  // the store of chunk sj - 2 has read stg
        named_bar_sync(1, 128);
        if (state_warp) {
          if (row < D) {
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) put8(stg, row, cc, acc + 8 * cc);
          } else if (row == D) {
#pragma unroll
            for (int q = 0; q < 16; ++q)
              B->zbuf[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
          }
          if (quad == 2) {  // g -> rows 64 (hi) and 65 (lo), split by the whole warp
            __syncwarp();
            const float2 zz = reinterpret_cast<const float2*>(B->zbuf)[lane];
            const uint32_t hi = pack_bf16x2(zz.x, zz.y);
            const uint32_t lo = pack_bf16x2(zz.x - __uint_as_float(hi << 16),
                                            zz.y - __uint_as_float(hi & 0xFFFF0000u));
            *reinterpret_cast<uint32_t*>(stg + sw128_offset(64, lane / 4) + (lane % 4) * 4) = hi;
            *reinterpret_cast<uint32_t*>(stg + sw128_offset(65, lane / 4) + (lane % 4) * 4) = lo;
            __syncwarp();
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (et == 32 && !*x.abort) {
          tma_store_3d(&tm_gt, stg, 0, 0, (int)((long long)pc.h * p.sp.NC + pc.tok0 / C + c));
          bulk_commit();
        }
        const int b = sj % NB;
        const bool got = waitb_warp(x, &B->dsready[b], (sj / NB) & 1);
        if (et == 32 && sj < 16) BW_TRACE(1, 18 + sj);
        if (state_warp) {
          if (got) {
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tl + 64 * b, r0);
            tmem_ld32(tl + 64 * b + 32, r1);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              acc[q] += __uint_as_float(r0[q]);
              acc[32 + q] += __uint_as_float(r1[q]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && got) mbar_arrive(&B->dsfree[b]);
        }
      }
      if (state_warp && row <= D && !*x.abort) {  // the piece's total
        float4* dst = reinterpret_cast<float4*>(p.RG + (size_t)pc.slot * SZ + row * D);
#pragma unroll
        for (int q = 0; q < 16; ++q)
          __stcg(dst + q, make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]));
      }
    }
    if (et == 32) bulk_wait_all();
    if (et == 32) BW_TRACE(1, 63);
  } else if (lane == 0) {  // ---- phi(Q), dnum -> workspace; the stage is released once read
    uint32_t sj = 0;
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i)
      for (int rr = 0; rr < pc.nch; ++rr, ++sj) {
        const int c = pc.nch - 1 - rr, s = sj % NS;
        if (!waitb(x, &B->xf[s], (sj / NS) & 1)) continue;
        uint8_t* st = smem + s * STAGE;
        const int tok = pc.tok0 + c * C;
        tma_store_3d(&tm_phiq, st, 0, tok, pc.h);
        tma_store_3d(&tm_dn, st + OFF_O, 0, tok, pc.h);
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(&B->empty[s]);
      }
    bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(x.tmem, kCols);
  }
}

}  // namespace gpx

// ===========================================================================
// 4. dq, dk, dv (and dS0, dz0)

namespace grd {

// stage: phi(Q) | phi(K) | V | dnum (bf16 [128 x 64] tiles) | the state tile
// S_c - E and the gradient-state tile G_c - EG (66 rows each).  OFF_P1 holds
// P1 (bf16 [128 x 128], two column blocks), then stages dq for its TMA stores
// (two [128 x 32] fp32 boxes); once a chunk's products are done its stage
// stages dv (over phi(Q) and phi(K)) and dk (over V and dnum).
constexpr uint32_t OFF_KF = BLK, OFF_V = 2 * BLK, OFF_DN = 3 * BLK;
constexpr uint32_t OFF_ST = 4 * BLK, OFF_GT = 4 * BLK + XT;
constexpr uint32_t STAGE = 4 * BLK + 2 * XT;
constexpr uint32_t OFF_E = 2 * STAGE;        // E (66 rows, from the output kernel), EG (rows 0..63)
constexpr uint32_t OFF_EG = OFF_E + XT;
constexpr uint32_t OFF_P1 = OFF_EG + XT;     // P1, then the dq staging
constexpr uint32_t OFF_VEC = OFF_P1 + 2 * BLK;  // floats: dd[2][128], zc[64], gc[64], gE[64]
constexpr uint32_t OFF_BAR = OFF_VEC + (2 * 128 + 3 * 64) * 4;
constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;
static_assert(STAGE % 1024 == 0 && OFF_GT % 1024 == 0 && OFF_E % 1024 == 0 && OFF_EG % 1024 == 0 &&
              OFF_P1 % 1024 == 0, "swizzled tile alignment");
static_assert(SMEM <= 227 * 1024, "shared memory per block");
constexpr int kThreads = 256;  // two threads per chunk row / TMEM lane
constexpr uint32_t kCols = 512;
// TMEM: the scores A1 = dnum V^T (masked into P1 in shared memory) and
// A3 = U W^T (masked into P3, packed in place), dW, dU, dV.  V dnum^T, the
// scores of dU's product, is A1^T, and its mask P2 = P1^T (the dden_t term
// included): dU's product reads P1 from shared memory as an MN-major operand.
constexpr uint32_t T_A1 = 0, T_A3 = 128, T_DW = 256, T_DU = 320, T_DV = 384;

constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);      // both K-major, N = 128
constexpr uint32_t ID_N64_MN = idesc_bf16_f32(128, 64, 0, 1);  // A K-major, B MN-major, N = 64
constexpr uint32_t ID_N64_K = idesc_bf16_f32(128, 64, 0, 0);   // both K-major, N = 64
constexpr uint32_t ID_MN_MN = idesc_bf16_f32(128, 64, 1, 1);   // both MN-major, N = 64

struct Params {
  Split sp;
  const float* RG;    // gradient piece totals (slot layout; with dS_N)
  const float* dden;  // [BH * NC][128]
  float* dq;
  float* dk;
  float* dv;
  float* dS0;         // or NULL
  float* dz0;         // or NULL
  unsigned* status;
  int force_wait;     // test hook: the first products wait once on a barrier that nothing completes
};

struct Bars {
  uint64_t full[2];
  uint64_t mma;
  uint64_t never;
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};

// The sum of slots [k0, k1) of `tot` from `base` on (fp32, in order), threads t
// of nthr: rows 0..63 as a bf16 tile (if `tile`), row 64 into `vec` (if
// `vec`); with `own`, sum + own (the slot's transposed rows: row j = column j)
// also goes to dS (NULL allowed) and its vector to dz (NULL allowed).
__device__ __forceinline__ void sum_slots(const float* tot, size_t base, int k0, int k1, uint8_t* tile,
                                          float* vec, const float* own, float* dS, float* dz, int t,
                                          int nthr) {
  constexpr int U = 4;  // slots read at once for each of two float4 of a thread
  for (int f0 = t; f0 < SZ / 4; f0 += 2 * nthr) {
    float4 e[2];
    e[0] = e[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = k0; k < k1; k += U) {
      float4 r[2][U];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int kk = 0; kk < U; ++kk)
          r[u][kk] = (f0 + u * nthr < SZ / 4 && k + kk < k1)
                         ? __ldcg(reinterpret_cast<const float4*>(tot + (base + k + kk) * SZ) + f0 + u * nthr)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int kk = 0; kk < U; ++kk) {  // in slot order
          e[u].x += r[u][kk].x; e[u].y += r[u][kk].y; e[u].z += r[u][kk].z; e[u].w += r[u][kk].w;
        }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int f = f0 + u * nthr;
      if (f >= SZ / 4) continue;
      const int row = f / 16, col = 4 * (f % 16);
      if (row < D) {
        if (tile) {
          uint2 hi;
          hi.x = pack_bf16x2(e[u].x, e[u].y);
          hi.y = pack_bf16x2(e[u].z, e[u].w);
          *reinterpret_cast<uint2*>(tile + sw128_offset(row, col / 8) + (col % 8) * 2) = hi;
        }
      } else if (vec) {
        vec[col] = e[u].x; vec[col + 1] = e[u].y; vec[col + 2] = e[u].z; vec[col + 3] = e[u].w;
      }
      if (own) {
        const float4 o = __ldcg(reinterpret_cast<const float4*>(own) + f);
        const float v4[4] = {e[u].x + o.x, e[u].y + o.y, e[u].z + o.z, e[u].w + o.w};
        if (row < D) {
          if (dS)
#pragma unroll
            for (int w = 0; w < 4; ++w) dS[(size_t)(col + w) * D + row] = v4[w];
        } else if (dz) {
          reinterpret_cast<float4*>(dz)[col / 4] = make_float4(v4[0], v4[1], v4[2], v4[3]);
        }
      }
    }
  }
}

// Half `hf` (columns 32 hf .. 32 hf + 31) of row r of a [128 x 64] bf16 tile.
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

__device__ __forceinline__ void tmem_row32(uint32_t taddr, float* out) {
  uint32_t a[32];
  tmem_ld32(taddr, a);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = __uint_as_float(a[i]);
}

// A masked score tile in TMEM (this thread's row = 32 quad + lane), rounded to
// bf16 and packed in place: the thread of column half hf reads key blocks
// 2 hf, 2 hf + 1 and writes them packed over the first of them (columns
// 64 hf .. 64 hf + 31), so the two threads of a row never touch each other's
// columns; the products read keys 0..63 from columns 0..31 and keys 64..127
// from 64..95.  `upper` keeps columns >= the row (else <=).  `rowadd` is
// added to every kept element, and `coladd[col]` unless it is NULL.
__device__ __forceinline__ void mask_pack(uint32_t base, bool upper, int quad, int lane, int hf,
                                          float rowadd, const float* coladd) {
  uint32_t r0[32], r1[32];
  const int q0 = 2 * hf;
  if (upper ? q0 >= quad : q0 <= quad) tmem_ld32(base + 32 * q0, r0);
  if (upper ? q0 + 1 >= quad : q0 + 1 <= quad) tmem_ld32(base + 32 * (q0 + 1), r1);
  tmem_ld_wait();
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int q4 = q0 + k;
    const uint32_t* r = k ? r1 : r0;
    uint32_t w[16];
    if (upper ? q4 < quad : q4 > quad) {  // nothing kept
#pragma unroll
      for (int t2 = 0; t2 < 16; ++t2) w[t2] = 0u;
    } else {
      // the diagonal block keeps keys on the kept side of the lane; the
      // others keep all (lo..hi: the kept range of this block's columns)
      const int lo = (q4 == quad && upper) ? lane : 0, hi = (q4 == quad && !upper) ? lane : 31;
      const float* ca = coladd ? coladd + 32 * q4 : nullptr;
#pragma unroll
      for (int t2 = 0; t2 < 16; ++t2) {
        const int s0 = 2 * t2, s1 = 2 * t2 + 1;
        float a0 = __uint_as_float(r[s0]) + rowadd, a1 = __uint_as_float(r[s1]) + rowadd;
        if (ca) {
          const float2 c2 = reinterpret_cast<const float2*>(ca)[t2];  // the same address across the warp
          a0 += c2.x;
          a1 += c2.y;
        }
        w[t2] = pack_bf16x2(s0 >= lo && s0 <= hi ? a0 : 0.f, s1 >= lo && s1 <= hi ? a1 : 0.f);
      }
    }
    tmem_st16(base + 64 * hf + 16 * k, w);
  }
  tmem_st_wait();
}

__device__ __forceinline__ uint32_t pcol(int ks) { return ks < 4 ? 8 * ks : 64 + 8 * (ks - 4); }

// P1 = the lower-triangular mask (keys s <= t) of A1 + rowadd, rounded to
// bf16, into a [128 x 128] K-major tile in shared memory (column block hf
// holds keys 64 hf .. 64 hf + 63): this thread's half of row `row`.  Every
// element is written, zeros included.
__device__ __forceinline__ void mask_to_smem(uint32_t base, uint8_t* p1, int row, int quad, int lane,
                                             int hf, float rowadd) {
  uint32_t r0[32], r1[32];
  const int q0 = 2 * hf;
  if (q0 <= quad) tmem_ld32(base + 32 * q0, r0);
  if (q0 + 1 <= quad) tmem_ld32(base + 32 * (q0 + 1), r1);
  tmem_ld_wait();
  uint8_t* dst = p1 + hf * BLK;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int q4 = q0 + k;
    const uint32_t* r = k ? r1 : r0;
    const int hi = q4 < quad ? 31 : q4 == quad ? lane : -1;  // kept keys 0 .. hi of the block
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int s0 = 8 * c + 2 * e, s1 = s0 + 1;
        w[e] = pack_bf16x2(s0 <= hi ? __uint_as_float(r[s0]) + rowadd : 0.f,
                           s1 <= hi ? __uint_as_float(r[s1]) + rowadd : 0.f);
      }
      *reinterpret_cast<uint4*>(dst + sw128_offset(row, 4 * k + c)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}


__global__ void __launch_bounds__(kThreads, 1)
grad_kernel(const __grid_constant__ CUtensorMap tm_phiq, const __grid_constant__ CUtensorMap tm_phik,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dn,
            const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_gt,
            const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
            const __grid_constant__ CUtensorMap tm_dv, const __grid_constant__ CUtensorMap tm_e,
            const Params p, const unsigned long long mbar_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* B = reinterpret_cast<Bars*>(smem + OFF_BAR);
  float* dd = reinterpret_cast<float*>(smem + OFF_VEC);  // [2][128]
  float* zc = dd + 256;
  float* gc = zc + 64;
  float* gE = gc + 64;
  const int t = threadIdx.x, warp = t / 32, lane = t % 32;
  const int row = t & (C - 1), hf = t >> 7, quad = warp & 3;
  const Split& sp = p.sp;
  const int NC = sp.NC;
  const Run run(sp, blockIdx.x);
  const uint32_t total = (uint32_t)(run.b - run.a);
  if (t == 0) {
    mbar_init(&B->full[0], 1);
    mbar_init(&B->full[1], 1);
    mbar_init(&B->mma, 1);
    mbar_init(&B->never, 1);
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_phiq);
    tma_prefetch_desc(&tm_phik);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_dn);
    tma_prefetch_desc(&tm_p);
    tma_prefetch_desc(&tm_gt);
    tma_prefetch_desc(&tm_dq);
    tma_prefetch_desc(&tm_dk);
    tma_prefetch_desc(&tm_dv);
    tma_prefetch_desc(&tm_e);
  }
  if (warp == 0) {
    tmem_alloc(&B->tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot);
  const uint32_t tl = tm + ((uint32_t)(32 * quad) << 16);  // this thread's TMEM lane (row)
  const uint32_t th = 32 * hf;                              // and its column half
  const Ctx x{p.status, &B->abort, tm, mbar_ns};
  if (t == 0) BW_TRACE(0, 0);
  pdl_launch_dependents();
  pdl_wait();  // every earlier launch of the gradient is complete
  if (t == 0) BW_TRACE(0, 1);

  uint32_t nload = 0, nmma = 0;
  // thread 32 (kLd): the loads of the run's chunk j into stage j % 2 and its
  // dden into dd[j % 2]; it also issues the output stores
  constexpr int kLd = 32;
  const bool haveE = total > 0 && run.idx0 > 0;
  auto load = [&](uint32_t j) {
    const int s = j % 2;
    uint8_t* st = smem + s * STAGE;
    const long long gi = run.a + j;
    const int h = (int)(gi / NC), tok = (int)(gi % NC) * C;
    const bool withE = j == 0 && haveE;  // the first piece's entry-state tile comes with chunk 0
    mbar_arrive_expect_tx(&B->full[s], 4 * BLK + 2 * XG + C * 4 + (withE ? XG : 0));
    if (withE) tma_load_3d_ef(smem + OFF_E, &tm_e, 0, 0, (int)blockIdx.x, &B->full[s]);
    bulk_load(dd + s * C, p.dden + (size_t)gi * C, C * 4, &B->full[s]);
    tma_load_3d_ef(st, &tm_phiq, 0, tok, h, &B->full[s]);
    tma_load_3d_ef(st + OFF_KF, &tm_phik, 0, tok, h, &B->full[s]);
    tma_load_3d_ef(st + OFF_V, &tm_v, 0, tok, h, &B->full[s]);
    tma_load_3d_ef(st + OFF_DN, &tm_dn, 0, tok, h, &B->full[s]);
    tma_load_3d_ef(st + OFF_ST, &tm_p, 0, 0, (int)gi, &B->full[s]);
    tma_load_3d_ef(st + OFF_GT, &tm_gt, 0, 0, (int)gi, &B->full[s]);
    ++nload;
  };

  if (t == kLd && total > 0) load(0);

  // The first piece's entry state E (the forward totals of the head's earlier
  // blocks), the last piece's exit gradient state EG (the gradient totals of
  // the head's later blocks), and dS0, dz0 of every head that starts here.
  const int h0 = run.h0, hl = total > 0 ? (int)((run.b - 1) / NC) : h0;
  const bool lastContinues = total > 0 && (run.b - (long long)hl * NC) < NC;
  const int npieces = total > 0 ? hl - h0 + 1 : 0;
  // position of this block among the blocks meeting head hl, and their count
  const int idxl = npieces == 1 ? run.idx0 : 0;
  const int nbl = sp.owner((long long)hl * NC + NC - 1) - sp.owner((long long)hl * NC) + 1;
  if (lastContinues) {
    const bool starts = (long long)hl * NC >= run.a;  // head hl's first chunk is in this run
    const float* own = p.RG + ((size_t)hl * sp.MPH + idxl) * SZ;
    sum_slots(p.RG, (size_t)hl * sp.MPH, idxl + 1, nbl, smem + OFF_EG, gE, starts ? own : nullptr,
              p.dS0 ? p.dS0 + (size_t)hl * D * D : nullptr, p.dz0 ? p.dz0 + (size_t)hl * D : nullptr, t,
              kThreads);
  }
  for (int h = h0; h < h0 + npieces; ++h) {  // heads that start and end in this run
    if ((long long)h * NC < run.a || (h == hl && lastContinues)) continue;
    const float* own = p.RG + (size_t)h * sp.MPH * SZ;  // slot 0: the head's only piece
    sum_slots(p.RG, 0, 0, 0, nullptr, nullptr, own, p.dS0 ? p.dS0 + (size_t)h * D * D : nullptr,
              p.dz0 ? p.dz0 + (size_t)h * D : nullptr, t, kThreads);
  }
  __syncthreads();
  if (t == 0) BW_TRACE(0, 2);

  auto issuing = [&]() {
    tc_fence_after();
    return !*reinterpret_cast<volatile int*>(&B->abort);
  };
  auto mma_done = [&]() {
    waitb(x, &B->mma, nmma & 1);
    ++nmma;
    tc_fence_after();
  };
  auto step_done = [&]() {
    tc_fence_before();
    __syncthreads();
  };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&B->abort) != 0; };
  const uint64_t eS = sdesc_sw128(smem_u32(smem + OFF_E), 16, 1024);
  const uint64_t eG = sdesc_sw128(smem_u32(smem + OFF_EG), 16, 1024);

  // thread 0: A1 = dnum V^T, A3 = U W^T, dW = dnum (S_c)^T, dU = V (G_c)^T,
  // dV = U G_c of the run's chunk j, once its tiles are in
  auto issue_first = [&](uint32_t j) {
    const int s = j % 2;
    const int h = (int)((run.a + j) / NC);
    const bool useE = haveE && h == h0, useEG = lastContinues && h == hl;
    const uint32_t aQ = smem_u32(smem + s * STAGE);
    // K-major operands step 32 bytes along K, MN-major ones 16 rows
    const uint64_t dQ = sdesc_sw128(aQ, 16, 1024), dK = sdesc_sw128(aQ + OFF_KF, 16, 1024);
    const uint64_t dV = sdesc_sw128(aQ + OFF_V, 16, 1024), dD = sdesc_sw128(aQ + OFF_DN, 16, 1024);
    const uint64_t dS = sdesc_sw128(aQ + OFF_ST, 16, 1024), dG = sdesc_sw128(aQ + OFF_GT, 16, 1024);
    if (waitb(x, &B->full[s], (j / 2) & 1) && (!p.force_wait || j > 0 || waitb(x, &B->never, 0)) &&
        issuing()) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16_ss(tm + T_A1, dD + ks * kStepK16, dV + ks * kStepK16, ID_S, ks > 0);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16_ss(tm + T_A3, dK + ks * kStepK16, dQ + ks * kStepK16, ID_S, ks > 0);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16_ss(tm + T_DW, dD + ks * kStepK16, dS + ks * kStepRows16, ID_N64_MN, ks > 0);
      if (useE) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16_ss(tm + T_DW, dD + ks * kStepK16, eS + ks * kStepRows16, ID_N64_MN, 1u);
      }
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16_ss(tm + T_DU, dV + ks * kStepK16, dG + ks * kStepRows16, ID_N64_MN, ks > 0);
      if (useEG) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16_ss(tm + T_DU, dV + ks * kStepK16, eG + ks * kStepRows16, ID_N64_MN, 1u);
      }
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)  // dV = U G_c
        mma_bf16_ss(tm + T_DV, dK + ks * kStepK16, dG + ks * kStepK16, ID_N64_K, ks > 0);
      if (useEG) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16_ss(tm + T_DV, dK + ks * kStepK16, eG + ks * kStepK16, ID_N64_K, 1u);
      }
    }
    mma_commit(&B->mma);
  };
  if (t == 0 && total > 0) issue_first(0);

  for (uint32_t j = 0; j < total; ++j) {
    const int s = j % 2;
    uint8_t* st = smem + s * STAGE;
    const long long gi = run.a + j;
    const int h = (int)(gi / NC), tok = (int)(gi % NC) * C;
    const bool useE = haveE && h == h0, useEG = lastContinues && h == hl;
    const uint32_t aQ = smem_u32(st), aK = aQ + OFF_KF, aD = aQ + OFF_DN;
    // the stores of the chunk before have read their staging (P1's region and
    // the other stage); the next chunk's tiles into that stage
    if (t == kLd && j > 0) bulk_wait_read_all();
    if (t == kLd && j + 1 < total && !aborted()) load(j + 1);
    waitb(x, &B->full[s], (j / 2) & 1);
    if (t == 0 && j < 8) BW_TRACE(0, 3 + 6 * j);
    if (t < D) {
      zc[t] = tile_at(st + OFF_ST, 64, t) + tile_at(st + OFF_ST, 65, t) +
              (useE ? tile_at(smem + OFF_E, 64, t) + tile_at(smem + OFF_E, 65, t) : 0.f);
    } else if (t < 2 * D) {
      const int i = t - D;
      gc[i] = tile_at(st + OFF_GT, 64, i) + tile_at(st + OFF_GT, 65, i) + (useEG ? gE[i] : 0.f);
    }
    mma_done();       // the first products of chunk j
    __syncthreads();  // (also: P1's region has been read by the stores of the chunk before)
    if (t == 0 && j < 8) BW_TRACE(0, 4 + 6 * j);
    // P1 = mask(A1 + dden_t) (keys s <= t) into shared memory, P3 = mask^T(A3)
    // (queries t >= s) in place
    mask_to_smem(tl + T_A1, smem + OFF_P1, row, quad, lane, hf, dd[s * C + row]);
    mask_pack(tl + T_A3, true, quad, lane, hf, 0.f, nullptr);
    fence_proxy_async_smem();
    step_done();
    if (t == 0 && j < 8) BW_TRACE(0, 5 + 6 * j);

    // dW += P1 U, dU += P1^T W (P1 read MN-major: its rows t are the K index),
    // dV += P3 dnum
    if (t == 0 && issuing()) {
      const uint32_t aP1 = smem_u32(smem + OFF_P1);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        mma_bf16_ss(tm + T_DW, sdesc_sw128(aP1 + (ks < 4 ? 32 * ks : BLK + 32 * (ks - 4)), 16, 1024),
                    sdesc_sw128(aK + ks * 2048, BLK, 1024), ID_N64_MN, 1u);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        mma_bf16_ss(tm + T_DU, sdesc_sw128(aP1 + ks * 2048, BLK, 1024), sdesc_sw128(aQ + ks * 2048, BLK, 1024),
                    ID_MN_MN, 1u);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        mma_bf16_ts(tm + T_DV, tm + T_A3 + pcol(ks), sdesc_sw128(aD + ks * 2048, BLK, 1024), ID_N64_MN, 1u);
    }
    if (t == 0) mma_commit(&B->mma);
    mma_done();
    if (t == 0 && j < 8) BW_TRACE(0, 6 + 6 * j);
    // dq = (dW + dden_t z_c) phi'(q) over P1's region, dk = (dU + g_c) phi'(k)
    // over V | dnum, then (every read of phi(Q), phi(K) done) dv over them
    {
      float o[32], f[32];
      uint8_t* bq = smem + OFF_P1 + hf * BLK;
      const float dr = dd[s * C + row];
      tmem_row32(tl + T_DW + th, o);
      load_half_bf16(st, row, hf, f);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float4 v4;
        v4.x = (o[4 * cc] + dr * zc[th + 4 * cc]) * fminf(f[4 * cc], 1.f);
        v4.y = (o[4 * cc + 1] + dr * zc[th + 4 * cc + 1]) * fminf(f[4 * cc + 1], 1.f);
        v4.z = (o[4 * cc + 2] + dr * zc[th + 4 * cc + 2]) * fminf(f[4 * cc + 2], 1.f);
        v4.w = (o[4 * cc + 3] + dr * zc[th + 4 * cc + 3]) * fminf(f[4 * cc + 3], 1.f);
        *reinterpret_cast<float4*>(bq + sw128_offset(row, cc)) = v4;
      }
      tmem_row32(tl + T_DU + th, o);
      load_half_bf16(st + OFF_KF, row, hf, f);
      uint8_t* bk = st + OFF_V + hf * BLK;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float4 v4;
        v4.x = (o[4 * cc] + gc[th + 4 * cc]) * fminf(f[4 * cc], 1.f);
        v4.y = (o[4 * cc + 1] + gc[th + 4 * cc + 1]) * fminf(f[4 * cc + 1], 1.f);
        v4.z = (o[4 * cc + 2] + gc[th + 4 * cc + 2]) * fminf(f[4 * cc + 2], 1.f);
        v4.w = (o[4 * cc + 3] + gc[th + 4 * cc + 3]) * fminf(f[4 * cc + 3], 1.f);
        *reinterpret_cast<float4*>(bk + sw128_offset(row, cc)) = v4;
      }
      tmem_row32(tl + T_DV + th, o);
      if (t == 0 && j < 8) BW_TRACE(0, 7 + 6 * j);
      step_done();  // every read of this chunk's phi tiles and TMEM is done
      uint8_t* bv = st + hf * BLK;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<float4*>(bv + sw128_offset(row, cc)) =
            make_float4(o[4 * cc], o[4 * cc + 1], o[4 * cc + 2], o[4 * cc + 3]);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (t == 0 && j + 1 < total) issue_first(j + 1);  // while this chunk's outputs are stored
    if (t == kLd && !aborted()) {  // rows past the sequence are not stored
      tma_store_3d_ef(&tm_dq, smem + OFF_P1, 0, tok, h);
      tma_store_3d_ef(&tm_dq, smem + OFF_P1 + BLK, 32, tok, h);
      tma_store_3d_ef(&tm_dk, st + OFF_V, 0, tok, h);
      tma_store_3d_ef(&tm_dk, st + OFF_V + BLK, 32, tok, h);
      tma_store_3d_ef(&tm_dv, st, 0, tok, h);
      tma_store_3d_ef(&tm_dv, st + BLK, 32, tok, h);
      bulk_commit();
    }
    if (t == 0 && j < 8) BW_TRACE(0, 8 + 6 * j);
  }
  if (t == kLd) bulk_wait_all();
  if (t == 0) BW_TRACE(0, 63);

  if (t == 0 && aborted()) {  // MMAs in flight end first
    int never = 0;
    mma_commit(&B->drain);
    mbar_wait(&B->drain, 0, globaltimer_ns() + mbar_ns, &never);
  }
  if (t == kLd && aborted()) drain_loads<2>(B->full, nload, mbar_ns);  // and loads
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, kCols);
  }
}

}  // namespace grd

// Workspace layout (byte offsets, each 256-byte aligned).
struct Layout {
  size_t R, P, phik, o, den, E, SN, RG, GT, phiq, dn, dd, total;
};

inline size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

Layout layout(int BH, int N, const Split& s) {
  Layout L;
  const size_t slots = (size_t)BH * s.MPH, tok = (size_t)BH * N;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = up256(off + bytes);
    return at;
  };
  L.R = take(slots * SZ * sizeof(float));
  L.P = take((size_t)s.TC() * XG);
  L.phik = take(tok * D * 2);
  L.o = take(tok * D * 2);
  L.den = take(tok * sizeof(float));
  L.E = take((size_t)s.G * XG);
  L.SN = take((size_t)BH * SZ * sizeof(float));
  L.RG = take(slots * SZ * sizeof(float));
  L.GT = take((size_t)s.TC() * XG);
  L.phiq = take(tok * D * 2);
  L.dn = take(tok * D * 2);
  L.dd = take((size_t)s.TC() * C * sizeof(float));
  L.total = off;
  return L;
}

}  // namespace

size_t backward_prefix64_workspace_bytes(int B, int H, int N) {
  const Split s = make_split(B * H, N, sm_count());
  return layout(B * H, N, s).total;
}

cudaError_t launch_backward_prefix64(const PrefillArgs& a, const float* dO, const float* dS_N,
                                     const float* dz_N, float* dq, float* dk, float* dv, float* dS0,
                                     float* dz0, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const Split sp = make_split(BH, a.N, sms);
  const Layout L = layout(BH, a.N, sp);
  if (!a.workspace || a.ws_bytes < L.total) return cudaErrorInvalidValue;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  unsigned* status = nullptr;
  cudaError_t e = library_status_word(&status);
  if (e != cudaSuccess) return e;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);

  // 1, 2: prefix tiles, piece totals, phi(K); o and den
  Prefix64Buffers b = {};
  b.R = reinterpret_cast<float*>(ws + L.R);
  b.P = ws + L.P;
  b.phik = reinterpret_cast<__nv_bfloat16*>(ws + L.phik);
  b.o = ws + L.o;
  b.den = reinterpret_cast<float*>(ws + L.den);
  b.E = ws + L.E;
  b.S_N = reinterpret_cast<float*>(ws + L.SN);
  b.z_N = b.S_N + (size_t)BH * D * D;
  b.status = status;
  b.force_wait = 0;
  e = launch_prefix64_pair(a, b, stream);
  if (e != cudaSuccess) return e;

  CUtensorMap mq, mo, mdo, mphiq, mdn, mgt, mphik, mv, mp, mdq, mdk, mdv, me;
  uint8_t* GT = ws + L.GT;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mo, b.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&me, b.E, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, XROWS, sp.G, 64, XROWS) ||
      !make_map(&mdo, dO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C) ||
      !make_map(&mphiq, ws + L.phiq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mdn, ws + L.dn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mgt, GT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, XROWS, (int)sp.TC(), 64, XROWS) ||
      !make_map(&mphik, b.phik, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mp, b.P, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, XROWS, (int)sp.TC(), 64, XROWS) ||
      !make_map(&mdq, dq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C) ||
      !make_map(&mdk, dk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C) ||
      !make_map(&mdv, dv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C))
    return cudaErrorInvalidValue;

  gpx::Params gp = {};
  gp.sp = sp;
  gp.dS_N = dS_N;
  gp.dz_N = dz_N;
  gp.den = b.den;
  gp.dden = reinterpret_cast<float*>(ws + L.dd);
  gp.RG = reinterpret_cast<float*>(ws + L.RG);
  gp.status = status;

  grd::Params rp = {};
  rp.sp = sp;
  rp.RG = gp.RG;
  rp.dden = gp.dden;
  rp.dq = dq;
  rp.dk = dk;
  rp.dv = dv;
  rp.dS0 = dS0;
  rp.dz0 = dz0;
  rp.status = status;
  rp.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);

  e = cudaFuncSetAttribute(gpx::gprefix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gpx::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grd::grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)grd::SMEM);
  if (e != cudaSuccess) return e;
  // 3, 4: programmatic dependents, each waiting for the launch before it
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(sp.G);
  cfg.blockDim = dim3(32 * gpx::kWarps);
  cfg.dynamicSmemBytes = gpx::SMEM;
  e = cudaLaunchKernelEx(&cfg, gpx::gprefix_kernel, mq, mo, mdo, mphiq, mdn, mgt, gp, mbar_ns);
  if (e != cudaSuccess) return e;
  cfg.blockDim = dim3(grd::kThreads);
  cfg.dynamicSmemBytes = grd::SMEM;
  return cudaLaunchKernelEx(&cfg, grd::grad_kernel, mphiq, mphik, mv, mdn, mp, mgt, mdq, mdk, mdv, me, rp,
                            mbar_ns);
}

}  // namespace la
