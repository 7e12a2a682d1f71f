// prefill_chunked128.cu -- chunked causal prefill for dk = dv = 128 on the
// sm_103a tensor cores, as three launches with no waiting between blocks.
//
// Operator (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03):
//   o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps),  S_t = S_{t-1} + phi(k_t) v_t^T,
//   z_t = z_{t-1} + phi(k_t),  phi = ELU + 1,  write before read.
// Chunkwise evaluation (page "线性注意力与SSM", section 3: a masked
// phi(Q) phi(K)^T attention inside each chunk, and across chunks a recurrence
// that hands over only the state), chunk C = 128 tokens.
//
// The work split is the one of the d = 64 path (prefill_tc_common.cuh: block j
// of G takes an equal run of the head-major chunk sequence, cut at head
// boundaries into pieces).  What differs at d = 128 is the budget: a chunk's
// Q, K and V tiles are 32 KB each, and the state S^T takes all 128 TMEM lanes.
//   K1 (aggregate): per piece, R^T = sum_c V_c^T phi(K_c) (TMEM lanes = value
//      column j) and the key sum zeta = sum_c phi(K_c)^T 1 (lanes = key column
//      i, an N = 16 product against an all-ones operand), stored to the
//      piece's workspace slot as S^T rows and then z.  phi(K) is not stored:
//      K3 applies phi to K itself, so nothing per token goes through the
//      workspace.
//   K2 (scan): per head, each piece's entry state as the left fold S0 + R_0 +
//      R_1 + ... in fp32 (the same order every run), and S_N, z_N.
//   K3 (output): each piece replays its chunks from its entry state E; phi is
//      applied to each K tile in shared memory, in place.  phi(Q)
//      lives in TMEM (the A operand of the two products that read it), so a
//      chunk's Q tile frees its shared-memory slot as soon as it has been read;
//      the running state S^T, z lives in TMEM, is snapshotted to bf16 for the
//      product phi(Q) [S | z] (z as hi + lo rows), and advances by
//      V^T phi(K), phi(K)^T 1 after each chunk.  Per chunk: scores
//      phi(Q) phi(K)^T, P = causal mask (bf16, written back into TMEM),
//      [num | den] = phi(Q) [S | z_hi | z_lo] + P [V | 1], o = num / (den + eps)
//      stored through TMA.
#include "prefill_decay.cuh"
#include "prefill_scan.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcp;

constexpr int D = 128;
constexpr int SZ = D * D + D;              // floats per state slot (S^T rows, then z)
constexpr uint32_t BLK = 16384;            // [128 rows x 128 B] swizzled bf16 block
constexpr uint32_t TILE = 2 * BLK;         // [128 tokens x 128] bf16: two column blocks
constexpr uint32_t ONES = 2048;            // [16 rows x 64] bf16, row 0 = 1 (K-major B)
constexpr uint32_t SNAP_ATOM = 144 * 128;  // K-major [144 x 64]: S^T rows, z hi, z lo, zeros
constexpr uint32_t SNAP = 2 * SNAP_ATOM;   // both halves of K = dk

constexpr uint32_t ID_ST = idesc_bf16_f32(128, D, 1, 1);    // V^T phi(K)
constexpr uint32_t ID_Z = idesc_bf16_f32(128, 16, 1, 0);    // phi(K)^T 1
constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);   // phi(Q) phi(K)^T, phi(Q) in TMEM
constexpr uint32_t ID_QS = idesc_bf16_f32(128, 144, 0, 0);  // phi(Q) [S | z_hi | z_lo]
constexpr uint32_t ID_PV = idesc_bf16_f32(128, D, 0, 1);    // P V, P in TMEM
constexpr uint32_t ID_P1 = idesc_bf16_f32(128, 16, 0, 0);   // P 1

struct Params {
  Split sp;
  float eps;
  const float* S0;
  const float* z0;
  float* S_N;
  float* z_N;
  unsigned* status;      // sticky error bits (the workspace header's)
  float* agg;            // [BH * MPH][SZ] piece totals, S^T rows then z
  float* E;              // [BH * MPH][SZ] entry states, same layout
  const float* alpha;    // decayed form: [BH][N] per-token decay of the state
  float* gam;            // decayed form: [BH * MPH] the decay over each piece
  int force_wait;        // test hook: K3 waits once on a barrier that nothing completes
};

struct Ctx {
  const Params* p;
  volatile int* abort;
  uint32_t tmem;
  unsigned long long mbar_ns;
};

// Bounded wait.  false once the block has given up (this wait ran out of time
// and recorded a timeout in the status word, or another role's did).  After
// that no role starts new asynchronous work, every role still runs its loops
// (each wait returning at once) so that named barriers stay matched, and the
// issuers drain what they started before the tensor memory is freed.
__device__ __forceinline__ bool wait_b(const Ctx& x, uint64_t* bar, uint32_t parity) {
  if (*x.abort) return false;
  if (mbar_try_wait(bar, parity)) return true;
  if (mbar_wait(bar, parity, globaltimer_ns() + x.mbar_ns, x.abort)) return true;
  *x.abort = 1;
  atomicOr(x.p->status, kStatusTimeout);
  return false;
}

__device__ __forceinline__ bool wait_w(const Ctx& x, uint64_t* bar, uint32_t parity) {
  return __all_sync(0xFFFFFFFFu, wait_b(x, bar, parity));
}

// Bounded wait until a CTA-scope counter reaches `target` (acquire).
__device__ __forceinline__ bool count_reached(const Ctx& x, const unsigned* c, unsigned target) {
  if (*x.abort) return false;
  const uint64_t dl = globaltimer_ns() + x.mbar_ns;
  while (ld_acquire_cta(c) < target) {
    if (*x.abort) return false;
    if (globaltimer_ns() > dl) {
      *x.abort = 1;
      atomicOr(x.p->status, kStatusTimeout);
      return false;
    }
  }
  return true;
}

// The last `nmax` loads issued on a ring of barriers land before the block leaves.
__device__ __forceinline__ void drain_ring(uint64_t* full, int nring, uint32_t issued, uint32_t nmax,
                                           unsigned long long ns) {
  int never = 0;
  const uint64_t dl = globaltimer_ns() + ns;
  for (uint32_t q = (issued > nmax ? issued - nmax : 0); q < issued; ++q)
    mbar_wait(&full[q % nring], (q / nring) & 1, dl, &never);
}

__device__ __forceinline__ void drain_and_free(const Ctx& x, int warp, uint32_t ncols) {
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(x.tmem, ncols);
  }
}

// The ones operand of the N = 16 products: a K-major B block of 16 rows (the
// N index) whose row 0 is 1 at every K position and rows 1..15 are 0.  Every K
// step reads the same first 16 K positions of these rows.
__device__ __forceinline__ void init_ones16(uint8_t* ones, int tid, int nthreads) {
  for (int i = tid; i < (int)(ONES / 16); i += nthreads)
    reinterpret_cast<uint4*>(ones)[i] =
        i < 8 ? make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u)  // bf16 1.0 pairs
              : make_uint4(0, 0, 0, 0);
  __syncthreads();
}

// 32 fp32 values of one S^T row (state columns i = 32 g .. 32 g + 31) as bf16
// into the K-major snapshot row `n`.
__device__ __forceinline__ void snap_store32(uint8_t* snap, int n, int g, const uint32_t* v) {
  uint8_t* atom = snap + (g / 2) * SNAP_ATOM;
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint4 u;
    u.x = pack_bf16x2(__uint_as_float(v[8 * cc + 0]), __uint_as_float(v[8 * cc + 1]));
    u.y = pack_bf16x2(__uint_as_float(v[8 * cc + 2]), __uint_as_float(v[8 * cc + 3]));
    u.z = pack_bf16x2(__uint_as_float(v[8 * cc + 4]), __uint_as_float(v[8 * cc + 5]));
    u.w = pack_bf16x2(__uint_as_float(v[8 * cc + 6]), __uint_as_float(v[8 * cc + 7]));
    *reinterpret_cast<uint4*>(atom + sw128_offset(n, 4 * (g % 2) + cc)) = u;
  }
}

// z[i] as rows 128 (hi = bf16(z)) and 129 (lo = bf16(z - hi)) of the
// snapshot at K position i: about 16 bits of z.
__device__ __forceinline__ void snap_z(uint8_t* snap, int i, float z) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(z);
  const __nv_bfloat16 lo = __float2bfloat16_rn(z - __bfloat162float(hi));
  uint8_t* atom = snap + (i / 64) * SNAP_ATOM;
  const int c8 = (i % 64) / 8, e = i % 8;
  *reinterpret_cast<__nv_bfloat16*>(atom + sw128_offset(128, c8) + 2 * e) = hi;
  *reinterpret_cast<__nv_bfloat16*>(atom + sw128_offset(129, c8) + 2 * e) = lo;
}

// Columns 32 m .. 32 m + 31 of tile row r (16-byte chunks 4 m .. 4 m + 3 of
// the two column blocks) with phi applied, as 16 packed bf16 pairs (element
// pair (2 c, 2 c + 1) in w[c]); rows at or past `valid` are 0.
__device__ __forceinline__ void phi_quarter(const uint8_t* tile, int r, int m, int valid,
                                            uint32_t (&w)[16]) {
  const uint8_t* blk = tile + (m / 2) * BLK;
  uint4 u[4];
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
    u[cc] = *reinterpret_cast<const uint4*>(blk + sw128_offset(r, 4 * (m % 2) + cc));
  const uint32_t keep = r < valid ? 0xFFFFFFFFu : 0u;
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    w[4 * cc + 0] = phi2(u[cc].x) & keep;
    w[4 * cc + 1] = phi2(u[cc].y) & keep;
    w[4 * cc + 2] = phi2(u[cc].z) & keep;
    w[4 * cc + 3] = phi2(u[cc].w) & keep;
  }
}

// ===========================================================================
// K1: piece totals

namespace k1 {

constexpr int NS = 3;                   // K, V stages (64 KB each)
constexpr uint32_t STAGE = 2 * TILE;    // K | V
constexpr uint32_t OFF_ONES = NS * STAGE;
constexpr uint32_t OFF_BAR = OFF_ONES + ONES;
constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;
constexpr int kWarps = 10;  // 0 TMA, 1 MMA, 2-5 phi, 6-9 epilogue
constexpr uint32_t kCols = 512;
constexpr uint32_t RCOLS = 144;  // per buffer: R^T (128 columns), then zeta (16)

struct Bars {
  uint64_t full[NS], xf[NS];
  uint64_t empty[NS];  // the stage's MMA done
  uint64_t racc[2];    // a piece's totals complete in buffer b  (MMA -> epilogue)
  uint64_t rfree[2];   // buffer b stored                       (epilogue -> MMA)
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
  float part[4];       // decayed form: the phi warps' partial sums of log2 alpha
};
static_assert(sizeof(Bars) <= 256, "barrier area");

// DECAY: the piece total with each token weighted by the decay from it to the
// piece's end, R = sum_t 2^(G_end - G_t) [v_t | 1]^T phi(k_t) (G: running sum
// of log2 alpha over the piece), so that the scan chains pieces as
// E' = Gamma E + R with Gamma = 2^G_end (stored per piece slot).  The phi
// warps first sum log2 alpha over the piece, then scale each phi(K) row by its
// weight (at most 1) before the products read it; the run is walked forwards.
template <bool DECAY>
__global__ void __launch_bounds__(32 * kWarps, 1)
aggregate_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const Params p, const unsigned long long mbar_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* B = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&B->full[s], 1);
      mbar_init(&B->xf[s], 4);
      mbar_init(&B->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B->racc[b], 1);
      mbar_init(&B->rfree[b], 1);
    }
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  const Run run(p.sp, blockIdx.x);
  // The run is walked backwards (last piece, last chunk first): the K and V it
  // touches last are those of the run's first chunks, which the output kernel
  // reads first, so they are still in L2.  A piece's total does not depend on
  // the order.  (The decayed form walks forwards, the order of its weights.)
  const int npieces = DECAY ? 0 : run.count(p.sp);
  auto walk = [&](int i, Piece* pc) {
    if (DECAY) return run.piece(p.sp, i, pc);
    return i < npieces && run.piece(p.sp, npieces - 1 - i, pc);
  };
  auto chunk_of = [&](const Piece& pc, int c) { return DECAY ? c : pc.nch - 1 - c; };
  auto load_stage = [&](uint32_t s, int tok, int h) {
    uint8_t* st = smem + s * STAGE;
    mbar_arrive_expect_tx(&B->full[s], 2 * TILE);
    tma_load_3d(st, &tm_k, 0, tok, h, &B->full[s]);
    tma_load_3d(st + BLK, &tm_k, 64, tok, h, &B->full[s]);
    tma_load_3d(st + TILE, &tm_v, 0, tok, h, &B->full[s]);
    tma_load_3d(st + TILE + BLK, &tm_v, 64, tok, h, &B->full[s]);
  };
  uint32_t pre = 0;  // loads issued during the set-up (thread 0)
  if (threadIdx.x == 0) {  // the first stages' loads go out before the rest of the set-up
    // a programmatic dependent of what ran before it on the stream (its
    // set-up overlaps that kernel's last blocks): no global memory before the wait
    pdl_wait();
    Piece pc;
    for (int i = 0; pre < NS && walk(i, &pc); ++i)
      for (int c = 0; pre < NS && c < pc.nch; ++c, ++pre) load_stage(pre, pc.tok0 + chunk_of(pc, c) * C, pc.h);
  }
  init_ones16(smem + OFF_ONES, threadIdx.x, 32 * kWarps);
  if (warp == 1) {
    tmem_alloc(&B->tmem_slot, kCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const Ctx x{&p, &B->abort, *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot), mbar_ns};
  pdl_launch_dependents();  // the scan may be scheduled now; it waits for this grid's results
  pdl_wait();               // (see thread 0's first loads)

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer: K, V chunk tiles (the first `pre` went out above)
      uint32_t sj = 0, issued = pre;
      Piece pc;
      for (int i = 0; walk(i, &pc); ++i)
        for (int c = 0; c < pc.nch; ++c, ++sj) {
          const uint32_t s = sj % NS;
          if (sj < pre) continue;
          if (!wait_b(x, &B->empty[s], ((sj / NS) - 1) & 1)) break;
          load_stage(s, pc.tok0 + chunk_of(pc, c) * C, pc.h);
          ++issued;
        }
      if (*x.abort) drain_ring(B->full, NS, issued, NS, mbar_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA: buffer b = the piece's sum of V^T phi(K) and phi(K)^T 1
      const uint64_t ones = sdesc_sw128(smem_u32(smem + OFF_ONES), 16, 1024);
      uint32_t sj = 0;
      Piece pc;
      for (int i = 0; walk(i, &pc); ++i) {
        const int b = i % 2;
        if (i >= 2 && !wait_b(x, &B->rfree[b], ((i / 2) - 1) & 1)) break;
        for (int c = 0; c < pc.nch; ++c, ++sj) {
          const uint32_t s = sj % NS;
          if (!wait_b(x, &B->xf[s], (sj / NS) & 1)) break;
          tc_fence_after();
          const uint32_t kt = smem_u32(smem + s * STAGE), vt = kt + TILE;
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks) {
            const uint32_t acc = (c > 0 || ks > 0) ? 1u : 0u;
            const uint64_t kd = sdesc_sw128(kt + ks * 2048, BLK, 1024);  // phi(K), MN-major
            mma_bf16_ss(x.tmem + RCOLS * b, sdesc_sw128(vt + ks * 2048, BLK, 1024), kd, ID_ST, acc);
            mma_bf16_ss(x.tmem + RCOLS * b + D, kd, ones, ID_Z, acc);
          }
          mma_commit(&B->empty[s]);
        }
        if (*x.abort) break;
        mma_commit(&B->racc[b]);
      }
      if (*x.abort) {
        int never = 0;
        mma_commit(&B->drain);
        mbar_wait(&B->drain, 0, globaltimer_ns() + mbar_ns, &never);
      }
    }
    __syncwarp();
  } else if (warp < 6) {  // ---- phi on K (one tile row per thread, a quarter row per iteration)
    const int r = threadIdx.x - 64, w = r / 32;
    uint32_t sj = 0;
    Piece pc;
    // decayed form: the four warps' total of v (both named barriers run on
    // every call)
    auto sum4 = [&](float v) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      if (lane == 0) B->part[w] = v;
      named_bar_sync(2, 128);
      const float tot = (B->part[0] + B->part[1]) + (B->part[2] + B->part[3]);
      named_bar_sync(2, 128);
      return tot;
    };
    for (int i = 0; walk(i, &pc); ++i) {
      float rem = 0.f;  // decayed form: log2 of the decay from the chunk's start to the piece's end
      if (DECAY) {
        const float* al = p.alpha + (size_t)pc.h * p.sp.N;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        int t = pc.tok0 + r;
        for (; t + 7 * C < pc.tok1; t += 8 * C) {  // eight loads in flight
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[u] += __log2f(fmaxf(__ldg(al + t + u * C), kAlphaMin));
        }
        for (; t < pc.tok1; t += C) acc[0] += __log2f(fmaxf(__ldg(al + t), kAlphaMin));
        rem = sum4(((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7])));
        if (r == 0) p.gam[pc.slot] = exp2_ftz(rem);
      }
      for (int c = 0; c < pc.nch; ++c, ++sj) {
        const uint32_t s = sj % NS;
        const int valid = pc.tok1 - (pc.tok0 + chunk_of(pc, c) * C);
        // decayed form: the row's weight 2^(rem - g_r), g_r the inclusive sum of
        // log2 alpha over the chunk up to row r, found before the tile is waited for
        float wt = 1.f;
        if (DECAY) {
          float la = r < valid ? __log2f(fmaxf(__ldg(p.alpha + (size_t)pc.h * p.sp.N + pc.tok0 +
                                                    chunk_of(pc, c) * C + r), kAlphaMin))
                               : 0.f;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xFFFFFFFFu, la, off);
            if (lane >= off) la += y;
          }
          if (lane == 31) B->part[w] = la;
          named_bar_sync(2, 128);
          float g = la, tot = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float pq = B->part[q];
            if (q < w) g += pq;
            tot += pq;
          }
          named_bar_sync(2, 128);
          wt = exp2_ftz(rem - g);
          rem -= tot;
        }
        if (!wait_w(x, &B->full[s], (sj / NS) & 1)) continue;
        uint8_t* st = smem + s * STAGE;
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
          if (DECAY) phi_scale_row<4>(st + (m / 2) * BLK, r, 4 * (m % 2), valid, wt);
          else phi_row<4>(st + (m / 2) * BLK, r, 4 * (m % 2), valid);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->xf[s]);
      }
    }
  } else {  // ---- epilogue: buffer b -> workspace slot (S^T rows, then z)
    const int quad = warp % 4, row = 32 * quad + lane, et = threadIdx.x - 192;
    const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
    Piece pc;
    for (int i = 0; walk(i, &pc); ++i) {
      const int b = i % 2;
      wait_b(x, &B->racc[b], (i / 2) & 1);  // on a timeout the rest runs on, storing garbage
      __syncwarp();
      tc_fence_after();
      float* dst = p.agg + (size_t)pc.slot * SZ;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        uint32_t v[32];
        tmem_ld32(tl + RCOLS * b + 32 * g, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          __stcg(reinterpret_cast<float4*>(dst + row * D + 32 * g) + q,
                 make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                             __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
      }
      uint32_t zz[2];
      tmem_ld2(tl + RCOLS * b + D, zz);
      tmem_ld_wait();
      __stcg(dst + D * D + row, __uint_as_float(zz[0]));
      tc_fence_before();
      named_bar_sync(1, 128);
      if (et == 0) mbar_arrive(&B->rfree[b]);
    }
  }
  drain_and_free(x, warp, kCols);
}

}  // namespace k1

// ===========================================================================
// K2: entry state of every piece (left fold from S0), final state

namespace k2 {

// DECAY: each piece first decays what came before it, E' = Gamma E + R.
template <bool DECAY>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const Params p) {
  pdl_launch_dependents();  // the output kernel may be scheduled now
  pdl_wait();               // the totals of the aggregate kernel are complete
  scan_fold<D, DECAY>(p.sp, p.agg, p.E, p.gam, p.S0, p.z0, p.S_N, p.z_N);
}

}  // namespace k2

// ===========================================================================
// K3: outputs

namespace k3 {

constexpr int NS = 2;                         // K, V stages (64 KB each)
constexpr uint32_t STAGE = 2 * TILE;          // K (phi applied in place) | V
constexpr uint32_t OFF_Q = NS * STAGE;        // one Q slot: its rows go to TMEM as phi(Q)
constexpr uint32_t OFF_SNAP = OFF_Q + TILE;   // the state snapshot
constexpr uint32_t OFF_ONES = OFF_SNAP + SNAP;
constexpr uint32_t OFF_OUT = OFF_ONES + ONES;  // output staging: one [128 x 32] fp32 box
constexpr uint32_t OFF_BAR = OFF_OUT + BLK;
// decayed form, per stage: g_t (the inclusive sums of log2 alpha over the
// chunk), the four warp totals, then the key factors 2^(g_e - g_s) (g_e the
// sum at the last key of s's 32-key block)
constexpr uint32_t OFF_G = OFF_BAR + 512;
constexpr int GKF = C + 4;
constexpr int GSTRIDE = 2 * C + 4;
constexpr uint32_t SMEM = OFF_G + NS * GSTRIDE * 4 + 1024;
static_assert(SMEM <= 227 * 1024, "shared memory per block");
static_assert(OFF_SNAP % 1024 == 0 && OFF_ONES % 1024 == 0 && OFF_OUT % 1024 == 0, "atom alignment");
// 0 K/V producer, 1 MMA, 2-5 phi (K in place, then Q into TMEM), 6-9 P,
// 10-13 state snapshots and output epilogue, 14 state chain, 15 Q producer:
// 512 threads, 128 registers
constexpr int kWarps = 16;
constexpr uint32_t kCols = 512;
constexpr uint32_t TA = 0;    // scores, then P (packed bf16, columns 0..63)
constexpr uint32_t TQ = 128;  // phi(Q), packed bf16 (64 columns)
constexpr uint32_t TO = 192;  // 128 numerator + 16 denominator columns
constexpr uint32_t TS = 336;  // running state S^T (lane j = value column), 128 columns
constexpr uint32_t TZ = 464;  // running z (lane i = key column), 16 columns

struct Bars {
  uint64_t full[NS], empty[NS];  // stage landed; stage free (MMA commit + state chain: 2 arrivals)
  uint64_t xf[NS];               // phi applied to the stage's K        (phi warps -> MMA, state chain)
  uint64_t qfull, qempty;        // Q landed; Q read by the four phi(Q) warps
  uint64_t qready;               // phi(Q) in TMEM                     (phi(Q) warps -> MMA)
  uint64_t accS;                 // scores in A                         (MMA -> P warps)
  uint64_t pready;               // P in A                              (P warps -> MMA)
  uint64_t afree;                // P V and P 1 done: A reusable        (MMA -> MMA)
  uint64_t qsdone;               // phi(Q) [S | z] done: snapshot and phi(Q) reusable
  uint64_t oready;               // num, den in O                       (MMA -> epilogue)
  uint64_t ofree;                // O read                              (epilogue -> MMA)
  uint64_t sacc;                 // running state advanced              (state chain -> state warps)
  uint64_t tsread;               // running state read out of TMEM      (state warps -> state chain)
  uint64_t sready;               // snapshot written                    (state warps -> MMA)
  uint64_t drain, drain2, never;
  uint32_t tmem_slot;
  int abort;
  unsigned epieces;  // entry states stored in TMEM so far, times 4 (state warps -> state chain)
  unsigned pdone[4];  // decayed form: chunks whose K rows P warp q has rescaled (P warps -> state chain)
};
static_assert(sizeof(Bars) <= 512, "barrier area");

__device__ __forceinline__ float* gsums(uint8_t* smem, uint32_t s) {
  return reinterpret_cast<float*>(smem + OFF_G) + s * GSTRIDE;
}

// Every barrier of the chunk loop completes once per chunk (sacc and tsread
// once per state advance), and single buffers (A, O, phi(Q), the snapshot, the
// Q slot) are handed round in chunk order, so no waiter can fall two phases
// behind: each completion needs the waiter of the one before to have passed.
// STRICT: read before write (token t reads the state before its own write, so
// the mask keeps keys s < t; the state handed between chunks is the same; with
// DECAY that state is S_{t-1}, so the query side takes g_{t-1}, 0 for the
// chunk's first token, in place of g_t).
// DECAY: S_t = alpha_t S_{t-1} + phi(k_t) v_t^T, z likewise.  With g_t the
// inclusive sum of log2 alpha over the chunk up to t and gamma_t = 2^g_t, the
// chunk's entry state reaches token t as gamma_t S and its own tokens s <= t
// with weight 2^(g_t - g_s); after the chunk S <- gamma_C S + sum_s
// 2^(g_C - g_s) phi(k_s) [v_s | 1]^T.  The phi warps scan log2 alpha; the P
// warps weight each kept score by 2^(g_t - g_s) and, once the scores have read
// them, rescale phi(Q) in TMEM by gamma_t (for phi(Q) [S | z], issued after
// P) and the chunk's phi(K) rows by 2^(g_C - g_s) (for the advance); the state
// warps write the running state back as gamma_C S (gamma_C of the next chunk)
// when they snapshot it.  All factors are at most 1 for alpha <= 1.
template <bool STRICT, bool DECAY>
__global__ void __launch_bounds__(32 * kWarps, 1)
output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
              const Params p, const unsigned long long mbar_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* B = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&B->full[s], 1);
      mbar_init(&B->empty[s], 2);
      mbar_init(&B->xf[s], 4);
    }
    mbar_init(&B->qfull, 1);
    mbar_init(&B->qempty, 4);
    mbar_init(&B->qready, 4);
    mbar_init(&B->accS, 1);
    mbar_init(&B->pready, 4);
    mbar_init(&B->afree, 1);
    mbar_init(&B->qsdone, 1);
    mbar_init(&B->oready, 1);
    mbar_init(&B->ofree, 4);
    mbar_init(&B->sacc, 1);
    mbar_init(&B->tsread, 4);
    mbar_init(&B->sready, 4);
    mbar_init(&B->drain, 1);
    mbar_init(&B->drain2, 1);
    mbar_init(&B->never, 1);
    B->epieces = 0;
    for (int q = 0; q < 4; ++q) B->pdone[q] = 0;
    B->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  const Run run(p.sp, blockIdx.x);
  // The first stages' K and V tiles and the first Q tile go out before the
  // rest of the set-up (inputs only: the launches before this one have waited
  // for whatever precedes the call on the stream).
  uint32_t pre = 0;
  bool any = false;
  if (threadIdx.x == 0) {
    Piece pc;
    for (int i = 0; pre < NS && run.piece(p.sp, i, &pc); ++i)
      for (int c = 0; pre < NS && c < pc.nch; ++c, ++pre) {
        uint8_t* st = smem + pre * STAGE;
        const int tok = pc.tok0 + c * C;
        mbar_arrive_expect_tx(&B->full[pre], 2 * TILE);
        tma_load_3d_ef(st, &tm_k, 0, tok, pc.h, &B->full[pre]);
        tma_load_3d_ef(st + BLK, &tm_k, 64, tok, pc.h, &B->full[pre]);
        tma_load_3d_ef(st + TILE, &tm_v, 0, tok, pc.h, &B->full[pre]);
        tma_load_3d_ef(st + TILE + BLK, &tm_v, 64, tok, pc.h, &B->full[pre]);
        if (pre == 0) {
          mbar_arrive_expect_tx(&B->qfull, TILE);
          tma_load_3d_ef(smem + OFF_Q, &tm_q, 0, tok, pc.h, &B->qfull);
          tma_load_3d_ef(smem + OFF_Q + BLK, &tm_q, 64, tok, pc.h, &B->qfull);
        }
      }
  }
  {
    Piece pc;
    any = run.piece(p.sp, 0, &pc);
  }
  init_ones16(smem + OFF_ONES, threadIdx.x, 32 * kWarps);
  for (int i = threadIdx.x; i < (int)(SNAP / 16); i += 32 * kWarps)  // rows 130..143 stay 0
    reinterpret_cast<uint4*>(smem + OFF_SNAP)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 1) {
    tmem_alloc(&B->tmem_slot, kCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();  // a following launch may set up while this one runs
  const Ctx x{&p, &B->abort, *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot), mbar_ns};

  if (warp == 0) {
    if (lane == 0) {  // ---- K, V producer (the first stages went out above)
      uint32_t sj = 0, issued = pre;
      Piece pc;
      for (int i = 0; run.piece(p.sp, i, &pc); ++i)
        for (int c = 0; c < pc.nch; ++c, ++sj) {
          const uint32_t s = sj % NS;
          uint8_t* st = smem + s * STAGE;
          const int tok = pc.tok0 + c * C;
          if (sj < pre) continue;
          if (!wait_b(x, &B->empty[s], ((sj / NS) - 1) & 1)) break;
          mbar_arrive_expect_tx(&B->full[s], 2 * TILE);
          tma_load_3d_ef(st, &tm_k, 0, tok, pc.h, &B->full[s]);
          tma_load_3d_ef(st + BLK, &tm_k, 64, tok, pc.h, &B->full[s]);
          tma_load_3d_ef(st + TILE, &tm_v, 0, tok, pc.h, &B->full[s]);
          tma_load_3d_ef(st + TILE + BLK, &tm_v, 64, tok, pc.h, &B->full[s]);
          ++issued;
        }
      if (*x.abort) drain_ring(B->full, NS, issued, NS, mbar_ns);
    }
    __syncwarp();
  } else if (warp == 15) {
    if (lane == 0) {  // ---- Q producer (the first Q went out above)
      uint32_t qj = 0, issued = any ? 1u : 0u;
      Piece pc;
      for (int i = 0; run.piece(p.sp, i, &pc); ++i)
        for (int c = 0; c < pc.nch; ++c, ++qj) {
          if (qj == 0) continue;
          if (!wait_b(x, &B->qempty, (qj - 1) & 1)) break;
          const int tok = pc.tok0 + c * C;
          mbar_arrive_expect_tx(&B->qfull, TILE);
          tma_load_3d_ef(smem + OFF_Q, &tm_q, 0, tok, pc.h, &B->qfull);
          tma_load_3d_ef(smem + OFF_Q + BLK, &tm_q, 64, tok, pc.h, &B->qfull);
          ++issued;
        }
      if (*x.abort) drain_ring(&B->qfull, 1, issued, 1, mbar_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issue: scores, phi(Q) [S | z], P [V | 1]
      const uint32_t tm = x.tmem;
      const uint64_t ones = sdesc_sw128(smem_u32(smem + OFF_ONES), 16, 1024);
      const uint32_t aSnap = smem_u32(smem + OFF_SNAP);
      uint32_t g = 0;
      bool ok = !p.force_wait || wait_b(x, &B->never, 0);
      Piece pc;
      for (int i = 0; ok && run.piece(p.sp, i, &pc); ++i)
        for (int c = 0; ok && c < pc.nch; ++c, ++g) {
          const uint32_t s = g % NS;
          ok = wait_b(x, &B->qready, g & 1) && wait_b(x, &B->xf[s], (g / NS) & 1) &&
               (g == 0 || wait_b(x, &B->afree, (g - 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint32_t kt = smem_u32(smem + s * STAGE), vt = kt + TILE;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)  // scores: phi(Q) from TMEM, phi(K) K-major
            mma_bf16_ts(tm + TA, tm + TQ + 8 * ks,
                        sdesc_sw128(kt + (ks / 4) * BLK + (ks % 4) * 32, 16, 1024), ID_S,
                        ks > 0 ? 1u : 0u);
          mma_commit(&B->accS);
          ok = wait_b(x, &B->sready, g & 1) && (g == 0 || wait_b(x, &B->ofree, (g - 1) & 1)) &&
               (!DECAY || wait_b(x, &B->pready, g & 1));  // decayed: phi(Q) rescaled with P
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)  // [num | den] = phi(Q) [S | z_hi | z_lo]
            mma_bf16_ts(tm + TO, tm + TQ + 8 * ks,
                        sdesc_sw128(aSnap + (ks / 4) * SNAP_ATOM + (ks % 4) * 32, 16, 1024), ID_QS,
                        ks > 0 ? 1u : 0u);
          mma_commit(&B->qsdone);
          if (!DECAY && !(ok = wait_b(x, &B->pready, g & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks) {  // += P [V | 1], P from TMEM
            mma_bf16_ts(tm + TO, tm + TA + 8 * ks, sdesc_sw128(vt + ks * 2048, BLK, 1024), ID_PV, 1u);
            mma_bf16_ts(tm + TO + D, tm + TA + 8 * ks, ones, ID_P1, 1u);
          }
          mma_commit(&B->oready);
          mma_commit(&B->afree);
          mma_commit(&B->empty[s]);
        }
      if (*x.abort) {
        int never = 0;
        mma_commit(&B->drain);
        mbar_wait(&B->drain, 0, globaltimer_ns() + mbar_ns, &never);
      }
    }
    __syncwarp();
  } else if (warp < 6) {  // ---- phi: K in place, then Q into TMEM (one row per thread)
    const int quad = warp % 4, row = 32 * quad + lane;
    const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
    uint32_t g = 0;
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i)
      for (int c = 0; c < pc.nch; ++c, ++g) {
        const int valid = pc.tok1 - (pc.tok0 + c * C);
        const uint32_t s = g % NS;
        // decayed form: this row's alpha, loaded before the wait for the tiles
        float av = 1.f;
        if (DECAY && row < valid) av = __ldg(p.alpha + (size_t)pc.h * p.sp.N + pc.tok0 + c * C + row);
        const bool got = wait_w(x, &B->full[s], (g / NS) & 1);
        if (got) {  // the chunk's K tile: phi in place
          uint8_t* kt = smem + s * STAGE;
#pragma unroll 1
          for (int m = 0; m < 4; ++m) phi_row<4>(kt + (m / 2) * BLK, row, 4 * (m % 2), valid);
        }
        if (DECAY) {
          // g_t: inclusive sums of log2 alpha over the chunk (alpha = 1 past the
          // end); a warp scan, then the totals of the warps before.  The named
          // barrier runs whether or not the wait succeeded, so that all four
          // warps always meet it.
          float la = 0.f;
          if (got && row < valid) la = __log2f(fmaxf(av, kAlphaMin));
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xFFFFFFFFu, la, off);
            if (lane >= off) la += y;
          }
          float* gs = gsums(smem, s);
          // the key factor from the warp's own sums (the earlier warps' totals cancel)
          gs[GKF + row] = exp2_ftz(__shfl_sync(0xFFFFFFFFu, la, 31) - la);
          if (lane == 31) gs[C + quad] = la;
          named_bar_sync(2, 128);
          for (int w = 0; w < quad; ++w) la += gs[C + w];
          gs[row] = la;
        }
        if (got) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&B->xf[s]);
        }
        // Q landed, and the products of the chunk before have read phi(Q)
        if (!wait_w(x, &B->qfull, g & 1)) continue;
        if (g > 0 && !wait_w(x, &B->qsdone, (g - 1) & 1)) continue;
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {  // a quarter row per iteration
          uint32_t w[16];
          phi_quarter(smem + OFF_Q, row, m, valid, w);
          tmem_st16(tl + TQ + 16 * m, w);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&B->qempty);
          mbar_arrive(&B->qready);
        }
      }
  } else if (warp < 10) {  // ---- P = causal mask of the scores, bf16, in place in TMEM
    const int quad = warp % 4, row = 32 * quad + lane;
    const uint32_t base = x.tmem + ((uint32_t)(32 * quad) << 16) + TA;
    uint32_t g = 0;
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i)
      for (int c = 0; c < pc.nch; ++c, ++g) {
        if (!wait_w(x, &B->accS, g & 1)) continue;
        tc_fence_after();
        const float* gs = gsums(smem, g % NS);
        // decayed form: gt the query side's sum (g_t, or g_{t-1} before write),
        // gkey the key side's (g_s for key s = row)
        const float gkey = DECAY ? gs[row] : 0.f;
        const float gt = !DECAY ? 0.f : !STRICT ? gkey : row > 0 ? gs[row - 1] : 0.f;
        // this warp's query rows are 32 quad .. +31: key blocks before `quad`
        // are fully visible, block `quad` holds the diagonal (kept), later
        // blocks are zero.  Packed keys 32 q4 .. go to columns 16 q4 ..; block
        // q4 is read completely before its packed columns (in block q4 / 2 <=
        // q4) are written.  Decayed form: kept scores are weighted by
        // 2^(g_t - g_s); for a block before the diagonal that is
        // 2^(g_t - g_e) 2^(g_e - g_s), g_e the sum at the block's last key (one
        // exponential per block and row, the key factors from the phi warps).
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t w[16];
          if (q4 > quad) {
#pragma unroll
            for (int t = 0; t < 16; ++t) w[t] = 0u;
          } else {
            uint32_t r[32];
            tmem_ld32(base + 32 * q4, r);
            tmem_ld_wait();
            if (q4 < quad) {
              float rf = 1.f;
              const float* ck = gs + GKF + 32 * q4;
              if (DECAY) rf = exp2_ftz(gt - gs[32 * q4 + 31]);
#pragma unroll
              for (int t = 0; t < 16; ++t) {
                float a0 = __uint_as_float(r[2 * t]), a1 = __uint_as_float(r[2 * t + 1]);
                if (DECAY) {
                  a0 *= rf * ck[2 * t];
                  a1 *= rf * ck[2 * t + 1];
                }
                w[t] = pack_bf16x2(a0, a1);
              }
            } else {
#pragma unroll
              for (int t = 0; t < 16; ++t) {
                float a0 = __uint_as_float(r[2 * t]), a1 = __uint_as_float(r[2 * t + 1]);
                if (DECAY) {
                  a0 *= exp2_ftz(gt - gs[32 * q4 + 2 * t]);
                  a1 *= exp2_ftz(gt - gs[32 * q4 + 2 * t + 1]);
                }
                w[t] = pack_bf16x2((STRICT ? 2 * t < lane : 2 * t <= lane) ? a0 : 0.f,
                                   (STRICT ? 2 * t + 1 < lane : 2 * t + 1 <= lane) ? a1 : 0.f);
              }
            }
          }
          tmem_st16(base + 16 * q4, w);
        }
        tmem_st_wait();
        if (DECAY) {
          // The scores have read phi(Q) and phi(K): phi(Q) [S | z] takes phi(Q)
          // times gamma_t (TMEM, packed bf16 pairs), the advance phi(K) rows
          // times 2^(g_C - g_t) (shared memory).
          const float gq = exp2_ftz(gt), gk = exp2_ftz(gs[C - 1] - gkey);
          const uint32_t tq = x.tmem + ((uint32_t)(32 * quad) << 16) + TQ;
#pragma unroll 1
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t r[32];
            tmem_ld32(tq + 32 * h2, r);
            tmem_ld_wait();
            uint32_t w0[16], w1[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              w0[t] = pack_bf16x2(__uint_as_float(r[t] << 16) * gq, __uint_as_float(r[t] & 0xFFFF0000u) * gq);
              w1[t] = pack_bf16x2(__uint_as_float(r[16 + t] << 16) * gq,
                                  __uint_as_float(r[16 + t] & 0xFFFF0000u) * gq);
            }
            tmem_st16(tq + 32 * h2, w0);
            tmem_st16(tq + 32 * h2 + 16, w1);
          }
          tmem_st_wait();
          uint8_t* kt = smem + (g % NS) * STAGE;
          scale_row(kt, row, gk);
          scale_row(kt + BLK, row, gk);
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&B->pready);
          if (DECAY) red_add_release_cta(&B->pdone[quad], 1u);
        }
      }
  } else if (warp < 14) {  // ---- state snapshots and output epilogue
    const int quad = warp % 4, row = 32 * quad + lane, et = threadIdx.x - 320;
    const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
    uint8_t* snap = smem + OFF_SNAP;
    uint8_t* out = smem + OFF_OUT;
    uint32_t g = 0, nsa = 0;
    pdl_wait();  // the entry states E are the scan kernel's output
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i) {
      // The piece's entry state E: into TMEM (running state) and the snapshot,
      // once the products of the chunk before have read the snapshot (the
      // previous piece's advances were all waited for below).
      if (g == 0 || wait_w(x, &B->qsdone, (g - 1) & 1)) {
        // decayed form: the running state enters the first advance as
        // gamma_C E (gamma_C of the piece's first chunk); the snapshot is E
        float gC = 1.f;
        if (DECAY) {
          wait_w(x, &B->xf[g % NS], (g / NS) & 1);  // the chunk's sums of log2 alpha
          gC = exp2_ftz(gsums(smem, g % NS)[C - 1]);
        }
        const float* src = p.E + (size_t)pc.slot * SZ;
#pragma unroll 1
        for (int grp = 0; grp < 4; ++grp) {
          uint32_t v[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 u = __ldcg(reinterpret_cast<const float4*>(src + row * D + 32 * grp) + q);
            v[4 * q] = __float_as_uint(u.x);
            v[4 * q + 1] = __float_as_uint(u.y);
            v[4 * q + 2] = __float_as_uint(u.z);
            v[4 * q + 3] = __float_as_uint(u.w);
          }
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            w0[t] = DECAY ? __float_as_uint(__uint_as_float(v[t]) * gC) : v[t];
            w1[t] = DECAY ? __float_as_uint(__uint_as_float(v[16 + t]) * gC) : v[16 + t];
          }
          tmem_st16(tl + TS + 32 * grp, w0);
          tmem_st16(tl + TS + 32 * grp + 16, w1);
          snap_store32(snap, row, grp, v);
        }
        const float z = __ldcg(src + D * D + row);
        uint32_t wz[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) wz[t] = 0u;
        wz[0] = __float_as_uint(z * gC);
        tmem_st16(tl + TZ, wz);
        snap_z(snap, row, z);
        tmem_st_wait();
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          red_add_release_cta(&B->epieces, 1u);
          mbar_arrive(&B->sready);
        }
      }

      for (int c = 0; c < pc.nch; ++c, ++g) {
        if (c + 1 < pc.nch) {  // the snapshot of the state after chunk g, for chunk g + 1
          const bool ok = wait_w(x, &B->sacc, nsa & 1) && wait_w(x, &B->qsdone, g & 1) &&
                          (!DECAY || wait_w(x, &B->xf[(g + 1) % NS], ((g + 1) / NS) & 1));
          ++nsa;
          if (ok) {
            tc_fence_after();
            // decayed form: the next advance adds onto gamma_C S, gamma_C of
            // the next chunk; the snapshot is S
            const float gC = DECAY ? exp2_ftz(gsums(smem, (g + 1) % NS)[C - 1]) : 1.f;
#pragma unroll 1
            for (int grp = 0; grp < 4; ++grp) {
              uint32_t v[32];
              tmem_ld32(tl + TS + 32 * grp, v);
              tmem_ld_wait();
              if (DECAY) {
                uint32_t w0[16], w1[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                  w0[t] = __float_as_uint(__uint_as_float(v[t]) * gC);
                  w1[t] = __float_as_uint(__uint_as_float(v[16 + t]) * gC);
                }
                tmem_st16(tl + TS + 32 * grp, w0);
                tmem_st16(tl + TS + 32 * grp + 16, w1);
              }
              snap_store32(snap, row, grp, v);
            }
            uint32_t zz[2];
            tmem_ld2(tl + TZ, zz);
            tmem_ld_wait();
            if (DECAY) {
              uint32_t wz[16];
#pragma unroll
              for (int t = 0; t < 16; ++t) wz[t] = 0u;
              wz[0] = __float_as_uint(__uint_as_float(zz[0]) * gC);
              tmem_st16(tl + TZ, wz);
              tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B->tsread);  // the running state may advance again
            snap_z(snap, row, __uint_as_float(zz[0]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B->sready);
          }
        }
        // o = num / (den + eps), one [128 x 32] box at a time through the staging
        // buffer and TMA; O is released once its last columns have been read
        const bool ok = wait_w(x, &B->oready, g & 1);
        tc_fence_after();
        uint32_t d2[2];
        tmem_ld2(tl + TO + D, d2);
        tmem_ld_wait();
        const float inv = 1.f / (__uint_as_float(d2[0]) + __uint_as_float(d2[1]) + p.eps);
        const int tok = pc.tok0 + c * C;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t n[32];
          tmem_ld32(tl + TO + 32 * q, n);
          tmem_ld_wait();
          if (q == 3) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(&B->ofree);
          }
          if (et == 0) bulk_wait_read_all();  // the previous box's store has read the staging
          named_bar_sync(1, 128);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<float4*>(out + sw128_offset(row, cc)) =
                make_float4(__uint_as_float(n[4 * cc]) * inv, __uint_as_float(n[4 * cc + 1]) * inv,
                            __uint_as_float(n[4 * cc + 2]) * inv, __uint_as_float(n[4 * cc + 3]) * inv);
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (et == 0 && !*x.abort) {
            tma_store_3d_ef(&tm_o, out, 32 * q, tok, pc.h);
            bulk_commit();
          }
        }
      }
    }
    if (et == 0) bulk_wait_all();
  } else {  // ---- the state chain: S^T += V^T phi(K), z += phi(K)^T 1, chunk by chunk
    if (lane == 0) {
      const uint64_t ones = sdesc_sw128(smem_u32(smem + OFF_ONES), 16, 1024);
      // The advance of chunk j (its stage loaded and phi applied to its K; the
      // running state read), or, for a piece's last chunk, which has none, just
      // this issuer's share of the stage's release.  Chunk j is loaded, so its
      // stage's previous use has been released and the release counts for
      // chunk j.
      auto advance = [&](uint32_t j, bool any_adv) {
        const uint32_t s = j % NS;
        if (!wait_b(x, &B->xf[s], (j / NS) & 1)) return false;
        if (!any_adv) {
          mbar_arrive(&B->empty[s]);
          return true;
        }
        if (DECAY) {  // phi(K) of chunk j rescaled by all four P warps
          for (int q = 0; q < 4; ++q)
            if (!count_reached(x, &B->pdone[q], j + 1)) return false;
        }
        tc_fence_after();
        const uint32_t kt = smem_u32(smem + s * STAGE), vt = kt + TILE;
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t kd = sdesc_sw128(kt + ks * 2048, BLK, 1024);
          mma_bf16_ss(x.tmem + TS, sdesc_sw128(vt + ks * 2048, BLK, 1024), kd, ID_ST, 1u);
          mma_bf16_ss(x.tmem + TZ, kd, ones, ID_Z, 1u);
        }
        mma_commit(&B->sacc);
        mma_commit(&B->empty[s]);
        return true;
      };
      uint32_t sj = 0, ntr = 0;
      bool ok = true;
      Piece pc;
      for (int i = 0; ok && run.piece(p.sp, i, &pc); ++i) {
        ok = count_reached(x, &B->epieces, 4u * (unsigned)(i + 1));  // E in TMEM
        if (ok) tc_fence_after();
        ok = ok && advance(sj, pc.nch > 1);  // chunk 0 advances from E
        for (int c = 0; ok && c + 1 < pc.nch; ++c, ++ntr)
          ok = wait_b(x, &B->tsread, ntr & 1) && advance(sj + c + 1, c + 2 < pc.nch);
        sj += pc.nch;
      }
      if (*x.abort) {  // the state advances in flight end before TMEM is freed
        int never = 0;
        mma_commit(&B->drain2);
        mbar_wait(&B->drain2, 0, globaltimer_ns() + mbar_ns, &never);
      }
    }
    __syncwarp();
  }
  drain_and_free(x, warp, kCols);
}

}  // namespace k3

}  // namespace

// agg and E slots
size_t prefill_chunked128_workspace_bytes(int B, int H, int N) {
  const Split s = make_split(B * H, N, sm_count());
  return 2 * (size_t)s.BH * s.MPH * SZ * sizeof(float);
}

cudaError_t launch_prefill_chunked128(const PrefillArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mo, a.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C))
    return cudaErrorInvalidValue;
  Params p = {};
  p.sp = make_split(BH, a.N, sms);
  p.eps = a.eps;
  p.S0 = a.S0;
  p.z0 = a.z0;
  p.S_N = a.S_N;
  p.z_N = a.z_N;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.status = a.status ? a.status : &reinterpret_cast<WsHeader*>(ws)->status;
  const size_t slots = (size_t)BH * p.sp.MPH;
  if (sizeof(WsHeader) + prefill_chunked128_workspace_bytes(a.B, a.H, a.N) > a.ws_bytes)
    return cudaErrorInvalidValue;
  p.agg = reinterpret_cast<float*>(ws + sizeof(WsHeader));
  p.E = p.agg + slots * SZ;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  p.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);

  cudaError_t e = cudaFuncSetAttribute(k1::aggregate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)k1::SMEM);
  auto* const out = a.strict ? k3::output_kernel<true, false> : k3::output_kernel<false, false>;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(out, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k3::SMEM);
  if (e != cudaSuccess) return e;
  // All three launches are programmatic dependents of what precedes them on
  // the stream: their blocks may start while the kernel before them runs, and
  // wait for it (griddepcontrol.wait) before touching what it may write.
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(32 * k1::kWarps);
  cfg.dynamicSmemBytes = k1::SMEM;
  e = cudaLaunchKernelEx(&cfg, k1::aggregate_kernel<false>, mk, mv, p, mbar_ns);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(scan_blocks_per_head<D>(), BH);
  cfg.blockDim = dim3(kScanThreads);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, k2::scan_kernel<false>, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(32 * k3::kWarps);
  cfg.dynamicSmemBytes = k3::SMEM;
  return cudaLaunchKernelEx(&cfg, out, mq, mk, mv, mo, p, mbar_ns);
}

// the decayed form's slots: agg and E, then one decay factor per piece slot
size_t prefill_decay128_workspace_bytes(int B, int H, int N) {
  const Split s = make_split(B * H, N, sm_count());
  const size_t slots = (size_t)s.BH * s.MPH;
  return (2 * slots * SZ + slots) * sizeof(float);
}

cudaError_t launch_prefill_decay128(const PrefillArgs& a, const float* alpha, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  if (!a.workspace || a.ws_bytes < prefill_decay128_workspace_bytes(a.B, a.H, a.N)) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mo, a.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C))
    return cudaErrorInvalidValue;
  Params p = {};
  p.sp = make_split(BH, a.N, sms);
  p.eps = a.eps;
  p.S0 = a.S0;
  p.z0 = a.z0;
  p.S_N = a.S_N;
  p.z_N = a.z_N;
  p.alpha = alpha;
  const size_t slots = (size_t)BH * p.sp.MPH;
  p.agg = static_cast<float*>(a.workspace);
  p.E = p.agg + slots * SZ;
  p.gam = p.E + slots * SZ;
  cudaError_t e = library_status_word(&p.status);
  if (e != cudaSuccess) return e;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  p.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);
  auto* const out = a.strict ? k3::output_kernel<true, true> : k3::output_kernel<false, true>;
  e = cudaFuncSetAttribute(k1::aggregate_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k1::SMEM);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(out, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k3::SMEM);
  if (e != cudaSuccess) return e;
  // the three launches, each a programmatic dependent of what precedes it
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(32 * k1::kWarps);
  cfg.dynamicSmemBytes = k1::SMEM;
  e = cudaLaunchKernelEx(&cfg, k1::aggregate_kernel<true>, mk, mv, p, mbar_ns);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(scan_blocks_per_head<D>(), BH);
  cfg.blockDim = dim3(kScanThreads);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, k2::scan_kernel<true>, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(32 * k3::kWarps);
  cfg.dynamicSmemBytes = k3::SMEM;
  return cudaLaunchKernelEx(&cfg, out, mq, mk, mv, mo, p, mbar_ns);
}

size_t aggregate128_totals_bytes(int B, int H, int N) {
  const Split s = make_split(B * H, N, sm_count());
  return (size_t)s.BH * s.MPH * SZ * sizeof(float);
}

cudaError_t launch_aggregate128_totals(const PrefillArgs& a, float* agg, unsigned* status,
                                       cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  CUtensorMap mk, mv;
  if (!make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C))
    return cudaErrorInvalidValue;
  Params p = {};
  p.sp = make_split(BH, a.N, sms);
  p.eps = a.eps;
  p.status = status;
  p.agg = agg;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  cudaError_t e = cudaFuncSetAttribute(k1::aggregate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)k1::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(32 * k1::kWarps);
  cfg.dynamicSmemBytes = k1::SMEM;
  return cudaLaunchKernelEx(&cfg, k1::aggregate_kernel<false>, mk, mv, p, mbar_ns);
}

}  // namespace la

