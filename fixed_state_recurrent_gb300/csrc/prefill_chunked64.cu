// prefill_chunked64.cu -- chunked causal prefill for dk = dv = 64 on the
// sm_103a tensor cores, as three launches with no waiting between blocks.
//
// Operator (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03):
//   o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps),  S_t = S_{t-1} + phi(k_t) v_t^T,
//   z_t = z_{t-1} + phi(k_t),  phi = ELU + 1,  write before read.
// Chunkwise evaluation (page "线性注意力与SSM", section 3: a small masked
// phi(Q) phi(K)^T attention inside each chunk, and across chunks a recurrence
// that hands over only the state), chunk C = 128 tokens.
//
// Work split: the B*H heads' chunks form one head-major sequence; block j of G
// takes the contiguous run [j TC / G, (j+1) TC / G) of it (TC = total chunks,
// so every block gets the same number of chunks to within one), cut at head
// boundaries into "pieces".  Piece slots are numbered (head, index of the
// block within the head's blocks).
//   K1 (aggregate): each piece's state increment, accumulated on the tensor
//      cores as the transposed product R = sum [V_c | 1]^T phi(K_c) (TMEM lanes
//      0..63 = R^T, lane 64 = z), stored transposed to the workspace; phi(K)
//      itself (bf16, the layout of K) is stored to the workspace for K3.
//   K2 (scan): per head, the exclusive prefix of every piece as the left fold
//      S0 + R_0 + R_1 + ... in fp32 (the same order every run), and the final
//      state S_N, z_N.
//   K3 (output): each piece replays its chunks from its prefix E (reading Q,
//      phi(K) and V; phi is applied to Q only): the running
//      state lives in TMEM (initialised to E, advanced by [V_c | 1]^T phi(K_c)
//      after each chunk) and is snapshotted to bf16 for the next chunk; per
//      chunk, scores phi(Q) phi(K)^T, P = causal mask of the scores (bf16,
//      written back into TMEM), [num | den] = P [V | 1] + phi(Q) [S | z] as two
//      N = 80 products, o = num / (den + eps) stored through TMA.
// V and phi(K) are read again by K3 (from L2 when the workload fits in it).
#include "prefill_decay.cuh"
#include "prefill_scan.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcp;

constexpr int D = 64;
constexpr int SZ = D * D + D;                // floats per state slot (R^T rows, then z)
constexpr uint32_t BLK = 16384;              // [128 rows x 128 B] swizzled bf16 tile
constexpr uint32_t SNAP = 80 * 128;          // K-major [80 x 64]: S^T rows, z hi, z lo, zeros

constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);     // phi(Q) phi(K)^T
constexpr uint32_t ID_PV = idesc_bf16_f32(128, D + 16, 0, 1); // P [V | 1]
constexpr uint32_t ID_QS = idesc_bf16_f32(128, D + 16, 0, 0); // phi(Q) [S | z]
constexpr uint32_t ID_DS = idesc_bf16_f32(128, D, 1, 1);      // [V | 1]^T phi(K)

struct Params3 {
  Split sp;
  float eps;
  const float* S0;
  const float* z0;
  float* S_N;
  float* z_N;
  unsigned* status;  // sticky error bits (the workspace header's, or the library's)
  const float* alpha;  // [BH][N] per-token decay of the state, or NULL
  float* agg;  // [BH * MPH][SZ], transposed slots
  float* E;    // [BH * MPH][SZ], exclusive prefixes, transposed slots
  float* gam;  // decayed form: [BH * MPH] the decay over each piece (product of its alphas)
  int force_wait;       // test hook: K3 waits once on a barrier that nothing completes
};

struct Ctx3 {
  const Params3* p;
  uint8_t* smem;
  uint64_t* bars;
  volatile int* abort;
  uint32_t tmem;
  unsigned long long mbar_ns;
};

// Bounded wait.  false once the block has given up (this wait ran out of time
// and recorded a timeout in the status word, or another role's did).  After
// that no role starts new asynchronous work (TMA, MMA, stores), every role
// still runs its loops, with each wait returning at once, so that the named
// barriers of a warp group stay matched, and the issuers drain what they
// started before the tensor memory is freed.
__device__ __forceinline__ bool wait3(const Ctx3& x, uint64_t* bar, uint32_t parity) {
  if (*x.abort) return false;
  if (mbar_try_wait(bar, parity)) return true;
  if (mbar_wait(bar, parity, globaltimer_ns() + x.mbar_ns, x.abort)) return true;
  *x.abort = 1;
  atomicOr(x.p->status, kStatusTimeout);
  return false;
}

// The same decision for a whole warp (all lanes wait on the same barrier).
__device__ __forceinline__ bool wait3_warp(const Ctx3& x, uint64_t* bar, uint32_t parity) {
  return __all_sync(0xFFFFFFFFu, wait3(x, bar, parity));
}

// Bounded wait until a CTA-scope counter reaches `target` (acquire).
__device__ __forceinline__ bool count_reached(const Ctx3& x, const unsigned* c, unsigned target) {
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

// Producer drain: the last loads that were issued (at most NS) land before the
// block leaves.
template <int NS_>
__device__ __forceinline__ void drain_loads(uint64_t* full, uint32_t issued, unsigned long long ns) {
  int never = 0;
  const uint64_t dl = globaltimer_ns() + ns;
  for (uint32_t q = (issued > NS_ ? issued - NS_ : 0); q < issued; ++q)
    mbar_wait(&full[q % NS_], (q / NS_) & 1, dl, &never);
}

// The running-state / snapshot helpers.  State lane `row` (0..64) of the
// transposed state owns slot floats [64 row, 64 row + 64): row j < 64 is
// column j of S (row j of S^T), row 64 is z.
__device__ __forceinline__ void store_snap_half(uint8_t* snap, int n, int half, const float* v) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * cc + 0], v[8 * cc + 1]);
    u.y = pack_bf16x2(v[8 * cc + 2], v[8 * cc + 3]);
    u.z = pack_bf16x2(v[8 * cc + 4], v[8 * cc + 5]);
    u.w = pack_bf16x2(v[8 * cc + 6], v[8 * cc + 7]);
    *reinterpret_cast<uint4*>(snap + sw128_offset(n, 4 * half + cc)) = u;
  }
}

// Snapshot rows of one state lane: S^T row `row`, or for lane 64 rows 64
// (hi = bf16(z)) and 65 (lo = bf16(z - hi)): about 16 bits of z.  Works on
// eight values at a time, so that no second copy of the half row is live.
__device__ __forceinline__ void snap_half(uint8_t* snap, int row, int half, const float* v) {
  if (row < D) {
    store_snap_half(snap, row, half, v);
  } else {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      float hi[8], lo[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        hi[i] = __bfloat162float(__float2bfloat16_rn(v[8 * cc + i]));
        lo[i] = v[8 * cc + i] - hi[i];
      }
      uint4 uh, ul;
      uh.x = pack_bf16x2(hi[0], hi[1]); uh.y = pack_bf16x2(hi[2], hi[3]);
      uh.z = pack_bf16x2(hi[4], hi[5]); uh.w = pack_bf16x2(hi[6], hi[7]);
      ul.x = pack_bf16x2(lo[0], lo[1]); ul.y = pack_bf16x2(lo[2], lo[3]);
      ul.z = pack_bf16x2(lo[4], lo[5]); ul.w = pack_bf16x2(lo[6], lo[7]);
      *reinterpret_cast<uint4*>(snap + sw128_offset(64, 4 * half + cc)) = uh;
      *reinterpret_cast<uint4*>(snap + sw128_offset(65, 4 * half + cc)) = ul;
    }
  }
}

__device__ __forceinline__ void tmem_ld_half(uint32_t taddr, float* out /*32*/) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void drain_and_free(const Ctx3& x, int warp, uint32_t ncols) {
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(x.tmem, ncols);
  }
}

// ===========================================================================
// K1: piece aggregates

namespace k1 {

constexpr int NS = 6;  // K, V stages: enough to cover a load from HBM, phi and the MMA
constexpr uint32_t STAGE = 2 * BLK;  // K | V
constexpr uint32_t OFF_ONES = NS * STAGE;
constexpr uint32_t OFF_BAR = OFF_ONES + BLK;
constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;
constexpr int kWarps = 10;  // 0 TMA, 1 MMA, 2-5 phi, 6-9 epilogue
constexpr uint32_t kCols = 128;

struct Bars {
  uint64_t full[NS], xf[NS];
  uint64_t empty[NS];  // the stage's MMA done
  uint64_t racc[2];   // a piece's R complete in R[b]   (MMA -> epilogue)
  uint64_t rfree[2];  // R[b] stored                    (epilogue -> MMA)
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
  float part[4];      // decayed form: the phi warps' partial sums of log2 alpha
};
static_assert(sizeof(Bars) <= 256, "barrier area");

// DECAY: the piece total with each token weighted by the decay from it to the
// piece's end, R = sum_t 2^(G_end - G_t) [v_t | 1]^T phi(k_t) (G: running sum of
// log2 alpha over the piece), so that the scan can chain pieces as
// E' = Gamma E + R with Gamma = 2^G_end.  The phi warps first sum log2 alpha
// over the piece, then scale each phi(K) row by that weight (at most 1) before
// the MMA reads it.  In either form phi(K) is not stored: the output kernel
// applies phi to K itself, so K is read twice (the second time largely from L2:
// both kernels walk a run in opposite orders) but phi(K) never goes through
// DRAM.
template <bool DECAY>
__global__ void __launch_bounds__(32 * kWarps, 1)
aggregate_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
       const Params3 p, const unsigned long long mbar_ns) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array by pointer
  // arithmetic so that accesses through it stay shared-space accesses
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
  // The plain form walks its run backwards (last piece and last chunk first),
  // so that the phi(K) and V it touches last -- those of its first chunks,
  // which the output kernel reads first -- are the ones L2 still holds when
  // that kernel starts (on calls too large for L2 to hold them all).  The
  // decayed form walks forwards: its weights run to each piece's end.
  const int npieces = DECAY ? 0 : run.count(p.sp);
  auto walk = [&](int i, Piece* pc) -> bool {
    if (!DECAY) {
      if (i >= npieces) return false;
      i = npieces - 1 - i;
    }
    return run.piece(p.sp, i, pc);
  };
  auto chunk_of = [&](const Piece& pc, int c) { return DECAY ? c : pc.nch - 1 - c; };
  uint32_t pre = 0;  // loads issued during the set-up (thread 0)
  if (threadIdx.x == 0) {  // the first stages' loads go out before the rest of the set-up
    // a programmatic dependent of what ran before it on the stream (its
    // set-up overlaps that kernel's last blocks): no global memory before the wait
    pdl_wait();
    Piece pc;
    for (int i = 0; pre < NS && walk(i, &pc); ++i)
      for (int c = 0; pre < NS && c < pc.nch; ++c, ++pre) {
        uint8_t* st = smem + pre * STAGE;
        const int tok = pc.tok0 + chunk_of(pc, c) * C;
        mbar_arrive_expect_tx(&B->full[pre], 2 * BLK);
        tma_load_3d(st, &tm_k, 0, tok, pc.h, &B->full[pre]);
        tma_load_3d(st + BLK, &tm_v, 0, tok, pc.h, &B->full[pre]);
      }
  }
  init_ones(smem + OFF_ONES, threadIdx.x, 32 * kWarps);
  if (warp == 1) {
    tmem_alloc(&B->tmem_slot, kCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const Ctx3 x{&p, smem, reinterpret_cast<uint64_t*>(B), &B->abort,
               *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot), mbar_ns};
  pdl_launch_dependents();  // the scan may be scheduled now; it waits for this grid's results
  pdl_wait();               // (see thread 0's first loads)

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer: K, V chunk tiles (the first `pre` went out above)
      uint32_t sj = 0, issued = pre;
      Piece pc;
      for (int i = 0; walk(i, &pc); ++i)
        for (int c = 0; c < pc.nch; ++c, ++sj) {
          const int s = sj % NS;
          if (sj < pre) continue;
          if (sj >= NS && !wait3(x, &B->empty[s], ((sj / NS) - 1) & 1)) break;
          uint8_t* st = smem + s * STAGE;
          const int tok = pc.tok0 + chunk_of(pc, c) * C;
          mbar_arrive_expect_tx(&B->full[s], 2 * BLK);
          tma_load_3d(st, &tm_k, 0, tok, pc.h, &B->full[s]);
          tma_load_3d(st + BLK, &tm_v, 0, tok, pc.h, &B->full[s]);
          ++issued;
        }
      if (*x.abort) drain_loads<NS>(B->full, issued, mbar_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA: R[b] = sum over the piece's chunks of [V | 1]^T phi(K)
      const uint32_t aOnes = smem_u32(smem + OFF_ONES);
      uint32_t sj = 0;
      Piece pc;
      for (int i = 0; walk(i, &pc); ++i) {
        const int b = i % 2;
        if (i >= 2 && !wait3(x, &B->rfree[b], ((i / 2) - 1) & 1)) break;
        for (int c = 0; c < pc.nch; ++c, ++sj) {
          const int s = sj % NS;
          if (!wait3(x, &B->xf[s], (sj / NS) & 1)) break;
          tc_fence_after();
          const uint32_t kt = smem_u32(smem + s * STAGE), vt = kt + BLK;
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks) {
            const uint64_t a = sdesc_sw128(vt + ks * 2048, aOnes - vt, 1024);
            const uint64_t bd = sdesc_sw128(kt + ks * 2048, BLK, 1024);
            mma_bf16_ss(x.tmem + 64 * b, a, bd, ID_DS, (c > 0 || ks > 0) ? 1u : 0u);
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
  } else if (warp < 6) {  // ---- phi on K (one tile row per thread)
    const int r = threadIdx.x - 64, w = r / 32;
    uint32_t sj = 0;
    Piece pc;
    // decayed form: the four warps' sum of v over their lanes (block-wide
    // total of the phi warps); both named barriers run on every call
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
        const int s = sj % NS;
        const int valid = pc.tok1 - (pc.tok0 + chunk_of(pc, c) * C);
        // the decay of this row's token, loaded before the wait for the tiles
        float av = 1.f;
        if (DECAY && r < valid) av = __ldg(p.alpha + (size_t)pc.h * p.sp.N + pc.tok0 + chunk_of(pc, c) * C + r);
        // decayed form: the row's weight 2^(rem - g_r), g_r the inclusive sum
        // of log2 alpha over the chunk up to row r (rem - g_r: the decay over
        // the piece's later tokens), found before the tiles are waited for;
        // both named barriers run on every call
        float wt = 1.f;
        if (DECAY) {
          float la = r < valid ? __log2f(fmaxf(av, kAlphaMin)) : 0.f;
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
        const bool got = wait3_warp(x, &B->full[s], (sj / NS) & 1);
        if (!got) continue;
        // half a row per iteration: one small copy of the loop body
#pragma unroll 1
        for (int m = 0; m < 2; ++m) {
          if (DECAY) phi_scale_row<4>(smem + s * STAGE, r, 4 * m, valid, wt);
          else phi_row<4>(smem + s * STAGE, r, 4 * m, valid);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->xf[s]);
      }
    }
  } else {  // ---- epilogue: R[b] -> workspace slot (transposed rows)
    const int quad = warp % 4, row = 32 * quad + lane, et = threadIdx.x - 192;
    const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
    Piece pc;
    for (int i = 0; walk(i, &pc); ++i) {
      const int b = i % 2;
      wait3(x, &B->racc[b], (i / 2) & 1);  // on a timeout the rest runs on, storing garbage
      tc_fence_after();
      if (quad <= 2) {
        float* dst = p.agg + (size_t)pc.slot * SZ + row * D;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tmem_ld_half(tl + 64 * b + 32 * half, v);
          if (row <= D) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              __stcg(reinterpret_cast<float4*>(dst + 32 * half) + q,
                     make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
          }
        }
      }
      tc_fence_before();
      named_bar_sync(1, 128);
      if (et == 0) mbar_arrive(&B->rfree[b]);
    }
  }
  drain_and_free(x, warp, kCols);
}

}  // namespace k1

// ===========================================================================
// K2: exclusive prefix of every piece (left fold from S0), final state

namespace k2 {

// DECAY: each piece first decays what came before it, E' = Gamma E + R.
template <bool DECAY>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const Params3 p) {
  pdl_launch_dependents();  // the output kernel may be scheduled now
  pdl_wait();               // the aggregates of the aggregate kernel are complete
  scan_fold<D, DECAY>(p.sp, p.agg, p.E, p.gam, p.S0, p.z0, p.S_N, p.z_N);
}

}  // namespace k2

// ===========================================================================
// K3: outputs

namespace k3 {

constexpr int NS = 3;
constexpr uint32_t STAGE = 3 * BLK;                // Q | K (phi applied here) | V
constexpr uint32_t OFF_ONES = NS * STAGE;
constexpr uint32_t OFF_SNAP = OFF_ONES + BLK;      // two snapshots
constexpr uint32_t OFF_OUT = OFF_SNAP + 2 * SNAP;  // output staging: two [128 x 32] fp32 boxes
constexpr uint32_t OFF_BAR = OFF_OUT + 2 * BLK;
// decayed form only: per stage, the inclusive sums g_t of log2 alpha over the
// chunk (128 floats), the four warps' totals of the scan, then per key s the
// factor 2^(g_e - g_s), g_e the sum at the last key of s's 32-key block
constexpr uint32_t OFF_G = OFF_BAR + 512;
constexpr int GKF = C + 4;  // offset of the key factors
constexpr int GSTRIDE = 2 * C + 4;
constexpr uint32_t SMEM = OFF_G + NS * GSTRIDE * 4 + 1024;
static_assert(SMEM <= 227 * 1024, "shared memory per block");
static_assert(OFF_OUT % 1024 == 0, "swizzled staging alignment");
// 0 TMA, 1 MMA, 2-5 phi(Q), 6-9 P, 10-13 output epilogue (10, 12, 13 also
// write the state snapshots), 14 state chain: at most four warps per SM
// sub-partition, so 128 registers per thread
constexpr int kWarps = 15;
constexpr uint32_t kCols = 512;
constexpr uint32_t TA = 0;    // A[b]: scores, then P (packed bf16) -- cols 128 b
constexpr uint32_t TO = 256;  // O[ob]: 64 numerator + 16 denominator cols -- 256 + 80 ob
constexpr uint32_t TS = 416;  // running state S^T (lanes 0..63) and z (lane 64), 64 cols

struct Bars {
  uint64_t full[NS], xf[NS];
  uint64_t empty[NS];  // the stage's products done: 2 arrivals  (both MMA issuers -> TMA)
  uint64_t accB[2];    // scores in A[b]                       (MMA -> P warps)
  uint64_t pready[2];  // P in A[b]                            (P warps -> MMA)
  uint64_t freeb[2];   // A[b] reusable                        (MMA -> MMA)
  uint64_t oready[2];  // num, den in O[ob]                    (MMA -> epilogue)
  uint64_t ofree[2];   // O[ob] read                           (epilogue -> MMA)
  uint64_t sacc;       // running state advanced               (state MMA -> epilogue)
  uint64_t sready[2];  // chunk j's snapshot written, in [j % 2] (epilogue -> MMA): two,
                       // as the snapshots may run one chunk ahead of the MMA warp
  uint64_t tsread;     // the running state read out of TMEM   (state warps -> state MMA)

  uint64_t drain, drain2;
  uint64_t never;      // completed by nothing (the forced-timeout test hook)
  uint32_t tmem_slot;
  int abort;
  unsigned epieces;    // entry states stored in TMEM so far, times 3 (state warps -> state MMA):
                       // a counter, as the state warps may run pieces ahead of the state MMA
  unsigned pdone[4];   // decayed form: chunks whose phi(K) rows P warp q has rescaled
                       // (P warps -> state MMA); counters, as the P warps may run two chunks
                       // ahead of the state MMA and apart from each other
  float4 zbuf[16];     // z, handed from its TMEM lane to the whole warp
};
static_assert(sizeof(Bars) <= 512, "barrier area");

__device__ __forceinline__ const float* gsums(uint8_t* smem, uint32_t s) {
  return reinterpret_cast<const float*>(smem + OFF_G) + s * GSTRIDE;
}

__device__ __forceinline__ uint8_t* stage_ptr(uint8_t* smem, uint32_t s) { return smem + s * STAGE; }

// Q, K, V and o go through TMA with the evict-first L2 policy here (the
// aggregate kernel loads K and V with the normal one, so that what both
// launches read is what L2 keeps).  The phi warps apply phi to Q and K.
//
// Two threads issue MMAs.  The MMA warp issues, per chunk a, the scores of
// chunk a + 1 and then P [V | 1] and phi(Q) [S | z] of chunk a, so that P of
// chunk a + 1 is built while the products of chunk a run.  The state chain has
// a warp of its own: the advance S += [V | 1]^T phi(K) of chunk a goes out as
// soon as the snapshot of the state before chunk a has been read out of TMEM.
// The three warps that hold state lanes publish each snapshot through
// mbarriers (three arrivals), never waiting for the issuers.  A stage is
// released by both issuers (a commit each, or an arrival where no state
// advance reads it).
//
// DECAY (one block per head, entry state S0, no aggregate kernel):
// S_t = alpha_t S_{t-1} + phi(k_t) v_t^T, z likewise.  With g_t the inclusive
// sum of log2 alpha over the chunk up to t and gamma_t = 2^g_t, a chunk's
// state enters token t as gamma_t S and its own tokens s <= t with weight
// 2^(g_t - g_s); after the chunk, S <- gamma_C S + sum_s 2^(g_C - g_s) phi(k_s)
// [v_s | 1]^T (gamma_C = gamma of the chunk's last token).  The phi warps load
// K (phi is applied here) and scan log2 alpha; the P warps weight each kept
// score by 2^(g_t - g_s) and, once the scores have read them, rescale the
// phi(Q) rows by gamma_t and the phi(K) rows by 2^(g_C - g_t) in place for the
// two later products; the state warps scale the running state by gamma_C of
// the next chunk before its advance, and after the last advance store S_N,
// z_N.  All factors are at most 1 for alpha <= 1.
// STRICT: read before write, token t reads the state before its own write,
// so the mask keeps keys s < t; with DECAY that state is S_{t-1}, so the query
// side takes g_{t-1} (0 for the chunk's first token) in place of g_t.
template <bool DECAY, bool STRICT = false>
__global__ void __launch_bounds__(32 * kWarps, 1)
output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
       const Params3 p, const unsigned long long mbar_ns) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array by pointer
  // arithmetic so that accesses through it stay shared-space accesses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* B = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&B->full[s], 1);
      mbar_init(&B->xf[s], 4);
      mbar_init(&B->empty[s], 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B->accB[b], 1);
      mbar_init(&B->pready[b], 4);
      mbar_init(&B->freeb[b], 1);
      mbar_init(&B->oready[b], 1);
      mbar_init(&B->ofree[b], 4);
    }
    mbar_init(&B->sacc, 1);
    mbar_init(&B->sready[0], 3);
    mbar_init(&B->sready[1], 3);
    B->epieces = 0;
    for (int q = 0; q < 4; ++q) B->pdone[q] = 0;
    mbar_init(&B->drain, 1);
    mbar_init(&B->drain2, 1);
    mbar_init(&B->tsread, 3);
    mbar_init(&B->never, 1);
    B->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  const Run run(p.sp, blockIdx.x);
  const bool whole = DECAY && !p.E;  // decayed form without a workspace: one block per head
  // The first stages' Q and V tiles (and K in the decayed form, which depends
  // on no other kernel) go out before the rest of the set-up; each stage's
  // barrier expects all three tiles, so phi(K) of the aggregate kernel joins
  // it later without another arrival.
  uint32_t pre = 0;
  if (threadIdx.x == 0) {
    Piece pc;
    for (int i = 0; pre < NS && run.piece(p.sp, i, &pc); ++i)
      for (int c = 0; pre < NS && c < pc.nch; ++c, ++pre) {
        uint8_t* st = stage_ptr(smem, pre);
        const int tok = pc.tok0 + c * C;
        mbar_arrive_expect_tx(&B->full[pre], 3 * BLK);
        tma_load_3d_ef(st, &tm_q, 0, tok, pc.h, &B->full[pre]);
        tma_load_3d_ef(st + 2 * BLK, &tm_v, 0, tok, pc.h, &B->full[pre]);
        tma_load_3d_ef(st + BLK, &tm_k, 0, tok, pc.h, &B->full[pre]);
      }
  }
  init_ones(smem + OFF_ONES, threadIdx.x, 32 * kWarps);
  for (int i = threadIdx.x; i < (int)(2 * SNAP / 16); i += 32 * kWarps)  // snapshot rows 66..79 stay 0
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
  const Ctx3 x{&p, smem, reinterpret_cast<uint64_t*>(B), &B->abort,
               *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot), mbar_ns};

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer: Q, K, V chunk tiles (see the set-up for the first)
      uint32_t sj = 0, issued = pre;
      Piece pc;
      for (int i = 0; run.piece(p.sp, i, &pc); ++i)
        for (int c = 0; c < pc.nch; ++c, ++sj) {
          const int s = sj % NS;
          uint8_t* st = stage_ptr(smem, s);
          const int tok = pc.tok0 + c * C;
          if (sj < pre) continue;  // went out during the set-up
          if (!wait3(x, &B->empty[s], ((sj / NS) - 1) & 1)) break;
          mbar_arrive_expect_tx(&B->full[s], 3 * BLK);
          tma_load_3d_ef(st, &tm_q, 0, tok, pc.h, &B->full[s]);
          tma_load_3d_ef(st + 2 * BLK, &tm_v, 0, tok, pc.h, &B->full[s]);
          tma_load_3d_ef(st + BLK, &tm_k, 0, tok, pc.h, &B->full[s]);
          ++issued;
        }
      if (*x.abort) drain_loads<NS>(B->full, issued, mbar_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issue
      const uint32_t tm = x.tmem;
      const uint32_t aOnes = smem_u32(smem + OFF_ONES);
      const uint32_t aSnap = smem_u32(smem + OFF_SNAP);
      uint32_t aj = 0, oj = 0;
      auto acquire = [&](uint32_t a) {  // job a: its stage transformed, A[a % 2] free
        if (!wait3(x, &B->xf[a % NS], (a / NS) & 1)) return false;
        if (a >= 2 && !wait3(x, &B->freeb[a % 2], ((a / 2) - 1) & 1)) return false;
        tc_fence_after();
        return true;
      };
      auto scores = [&](uint32_t a) {
        const uint32_t st = smem_u32(stage_ptr(smem, a % NS));
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16_ss(tm + TA + 128 * (a % 2), sdesc_sw128(st + ks * 32, 16, 1024),
                      sdesc_sw128(st + BLK + ks * 32, 16, 1024), ID_S, ks > 0 ? 1u : 0u);
        mma_commit(&B->accB[a % 2]);
      };
      bool ok = !p.force_wait || wait3(x, &B->never, 0);
      Piece pc;
      for (int i = 0; ok && run.piece(p.sp, i, &pc); ++i) {
        const uint32_t a0 = aj;
        if (!acquire(a0)) break;
        scores(a0);
        for (int c = 0; ok && c < pc.nch; ++c) {
          const uint32_t a = a0 + c;
          const bool more = c + 1 < pc.nch;
          if (more) {
            if (!(ok = acquire(a + 1))) break;
            scores(a + 1);
          }
          const uint32_t st = smem_u32(stage_ptr(smem, a % NS)), vt = st + 2 * BLK;
          const int b = a % 2, ob = oj % 2;
          ok = wait3(x, &B->sready[a % 2], (a / 2) & 1) &&  // this chunk's state snapshot
               wait3(x, &B->pready[b], (a / 2) & 1) &&
               (oj < 2 || wait3(x, &B->ofree[ob], ((oj / 2) - 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint32_t dO = tm + TO + 80 * ob, aP = tm + TA + 128 * b;
          const uint32_t sn = aSnap + (c % 2) * SNAP;
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks)  // P [V | 1], P from TMEM
            mma_bf16_ts(dO, aP + 8 * ks, sdesc_sw128(vt + ks * 2048, aOnes - vt, 1024), ID_PV,
                        ks > 0 ? 1u : 0u);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)  // phi(Q) [S | z]
            mma_bf16_ss(dO, sdesc_sw128(st + ks * 32, 16, 1024), sdesc_sw128(sn + ks * 32, 16, 1024),
                        ID_QS, 1u);
          mma_commit(&B->oready[ob]);
          mma_commit(&B->freeb[b]);
          mma_commit(&B->empty[a % NS]);
          ++oj;
        }
        aj = a0 + pc.nch;
      }
      if (*x.abort) {
        int never = 0;
        mma_commit(&B->drain);
        mbar_wait(&B->drain, 0, globaltimer_ns() + mbar_ns, &never);
      }
    }
    __syncwarp();
  } else if (warp < 6) {  // ---- phi on Q and K (one tile row per thread)
    const int r = threadIdx.x - 64;
    uint32_t sj = 0;
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i)
      for (int c = 0; c < pc.nch; ++c, ++sj) {
        const int s = sj % NS;
        const int valid = pc.tok1 - (pc.tok0 + c * C);
        // the decay of this row's token, loaded before the wait for the tiles
        float av = 1.f;
        if (DECAY && r < valid) av = __ldg(p.alpha + (size_t)pc.h * p.sp.N + pc.tok0 + c * C + r);
        const bool got = wait3_warp(x, &B->full[s], (sj / NS) & 1);
        if (!DECAY && !got) continue;
        uint8_t* st = stage_ptr(smem, s);
        if (got) {
          // Q, and in the decayed form K too: one copy of the loop body (the
          // roles' code together must stay within the instruction caches)
#pragma unroll 1
          for (int m = 0; m < 4; ++m) phi_row<4>(st + (m / 2) * BLK, r, 4 * (m % 2), valid);
        }
        if (DECAY) {
          // g_t: inclusive sums of log2 alpha over the chunk (alpha = 1 past the
          // end); a warp scan, then the totals of the warps before.  The named
          // barrier runs whether or not the wait succeeded, so that all four
          // warps always meet it.
          float la = 0.f;
          if (got && r < valid) la = __log2f(fmaxf(av, kAlphaMin));
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xFFFFFFFFu, la, off);
            if (lane >= off) la += y;
          }
          float* g = reinterpret_cast<float*>(smem + OFF_G) + s * GSTRIDE;
          // the key factor from the warp's own sums (the earlier warps' totals cancel)
          g[GKF + r] = exp2_ftz(__shfl_sync(0xFFFFFFFFu, la, 31) - la);
          if (lane == 31) g[C + r / 32] = la;
          named_bar_sync(2, 128);
          for (int w = 0; w < r / 32; ++w) la += g[C + w];
          g[r] = la;
          if (!got) continue;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->xf[s]);
      }
  } else if (warp < 10) {  // ---- P = causal mask of the scores, bf16, in place in TMEM
    const int quad = warp % 4;
    const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
    uint32_t aj = 0;
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i)
      for (int c = 0; c < pc.nch; ++c, ++aj) {
        const int b = aj % 2;
        if (!wait3_warp(x, &B->accB[b], (aj / 2) & 1)) continue;
        tc_fence_after();
        const uint32_t base = tl + TA + 128 * b;
        const int row = 32 * quad + lane;
        const float* g = gsums(smem, aj % NS);
        // decayed form: gt the query side's sum (g_t, or g_{t-1} before write),
        // gk the key side's (g_s for key s = row)
        const float gk = DECAY ? g[row] : 0.f;
        const float gt = !DECAY ? 0.f : !STRICT ? gk : row > 0 ? g[row - 1] : 0.f;
        // this warp's query rows are 32 quad .. +31: key blocks before `quad` are
        // fully visible, block `quad` holds the diagonal, later blocks are zero;
        // packed keys 32 q4.. go to columns 16 q4..  One key block at a time
        // (one copy of the loop body: the roles' code together must stay
        // within the instruction caches): block q4 is read completely before
        // its packed columns, which lie in block q4 / 2 <= q4, are written.
        // Decayed form: kept scores are weighted by 2^(g_t - g_s); for a block
        // before the diagonal that is 2^(g_t - g_e) 2^(g_e - g_s), g_e the sum
        // at the block's last key: one exponential per block and row, the key
        // factors from the phi warps (each factor <= 1 when alpha <= 1).
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
              const float* ck = g + GKF + 32 * q4;
              if (DECAY) rf = exp2_ftz(gt - g[32 * q4 + 31]);
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
                  a0 *= exp2_ftz(gt - g[32 * q4 + 2 * t]);
                  a1 *= exp2_ftz(gt - g[32 * q4 + 2 * t + 1]);
                }
                w[t] = pack_bf16x2((STRICT ? 2 * t < lane : 2 * t <= lane) ? a0 : 0.f,
                                   (STRICT ? 2 * t + 1 < lane : 2 * t + 1 <= lane) ? a1 : 0.f);
              }
            }
          }
          tmem_st16(base + 16 * q4, w);
        }
        tmem_st_wait();
        if (DECAY) {  // the scores have read phi(Q), phi(K): rescale them for the later products
          uint8_t* st = stage_ptr(smem, aj % NS);
          // phi(Q) [S | z]: gamma_t; the advance: phi(K) by 2^(g_C - g_t)
#pragma unroll 1
          for (int m = 0; m < 2; ++m) scale_row(st + m * BLK, row, exp2_ftz(m ? g[C - 1] - gk : gt));
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&B->pready[b]);
          if (DECAY) red_add_release_cta(&B->pdone[quad], 1u);
        }
      }
  } else if (warp < 14) {  // ---- state snapshots (state lanes only) and output epilogue
    const int quad = warp % 4, row = 32 * quad + lane, et = threadIdx.x - 320;
    const bool state_warp = quad <= 2, state_row = row <= D;
    const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
    uint8_t* snap = smem + OFF_SNAP;
    uint8_t* out = smem + OFF_OUT;
    uint32_t oj = 0, nsa = 0, sj = 0;
    if (!whole) pdl_wait();  // the entry states E are the scan kernel's output
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i) {
      // The piece's entry state E: into TMEM (running state) and snapshot 0.
      // The previous piece's products have all completed: its last output was
      // read below, and every state advance was waited for.
      if (state_warp) {
        // decayed form: the state enters the first advance as gamma_C E
        float gC = 1.f;
        if (DECAY) {
          wait3_warp(x, &B->xf[sj % NS], (sj / NS) & 1);  // the chunk's decay sums
          gC = exp2_ftz(gsums(smem, sj % NS)[C - 1]);
        }
        const float* src = p.E + (size_t)pc.slot * SZ + (state_row ? row : 0) * D;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float e[32];
          if (whole) {  // S0 and z0 themselves (the whole head is the piece)
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              const int i = 32 * half + q;
              e[q] = !state_row ? 0.f
                     : row < D ? (p.S0 ? __ldg(p.S0 + ((size_t)pc.h * D + i) * D + row) : 0.f)
                               : (p.z0 ? __ldg(p.z0 + (size_t)pc.h * D + i) : 0.f);
            }
          } else if (state_row) {
            float4 u[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) u[q] = __ldcg(reinterpret_cast<const float4*>(src + 32 * half) + q);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              e[4 * q] = u[q].x; e[4 * q + 1] = u[q].y; e[4 * q + 2] = u[q].z; e[4 * q + 3] = u[q].w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) e[q] = 0.f;
          }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t w[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) w[t] = __float_as_uint(e[16 * q + t] * gC);
            tmem_st16(tl + TS + 32 * half + 16 * q, w);
          }
          if (state_row) snap_half(snap, row, half, e);
        }
        tmem_st_wait();
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          red_add_release_cta(&B->epieces, 1u);
          mbar_arrive(&B->sready[sj % 2]);
        }
      }

      for (int c = 0; c < pc.nch; ++c, ++oj, ++sj) {
        if (c + 1 < pc.nch && state_warp) {  // snapshot of the state after chunk c, for chunk c + 1
          wait3(x, &B->sacc, nsa & 1);
          ++nsa;
          tc_fence_after();
          uint32_t r0[32], r1[32];
          tmem_ld32(tl + TS, r0);
          tmem_ld32(tl + TS + 32, r1);
          tmem_ld_wait();
          if (DECAY) {  // the next advance adds onto gamma_C S, gamma_C of the next chunk
            const uint32_t sn1 = sj + 1;
            wait3_warp(x, &B->xf[sn1 % NS], (sn1 / NS) & 1);
            const float gC = exp2_ftz(gsums(smem, sn1 % NS)[C - 1]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t* rr = q < 2 ? r0 + 16 * q : r1 + 16 * (q - 2);
              uint32_t w[16];
#pragma unroll
              for (int t = 0; t < 16; ++t) w[t] = __float_as_uint(__uint_as_float(rr[t]) * gC);
              tmem_st16(tl + TS + 16 * q, w);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&B->tsread);  // the running state may advance again
          uint8_t* sn = snap + ((c + 1) % 2) * SNAP;
          if (quad < 2) {  // S^T rows
            store_snap_half(sn, row, 0, reinterpret_cast<const float*>(r0));
            store_snap_half(sn, row, 1, reinterpret_cast<const float*>(r1));
          } else {  // z (lane 64 only) -> rows 64 (hi) and 65 (lo), split by the whole warp
            if (lane == 0) {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                B->zbuf[q] = make_float4(__uint_as_float(r0[4 * q]), __uint_as_float(r0[4 * q + 1]),
                                         __uint_as_float(r0[4 * q + 2]), __uint_as_float(r0[4 * q + 3]));
                B->zbuf[8 + q] = make_float4(__uint_as_float(r1[4 * q]), __uint_as_float(r1[4 * q + 1]),
                                             __uint_as_float(r1[4 * q + 2]), __uint_as_float(r1[4 * q + 3]));
              }
            }
            __syncwarp();
            const float2 zz = reinterpret_cast<const float2*>(B->zbuf)[lane];  // z[2 lane], z[2 lane + 1]
            const uint32_t hi = pack_bf16x2(zz.x, zz.y);
            const uint32_t lo = pack_bf16x2(zz.x - __uint_as_float(hi << 16), zz.y - __uint_as_float(hi & 0xFFFF0000u));
            *reinterpret_cast<uint32_t*>(sn + sw128_offset(64, lane / 4) + (lane % 4) * 4) = hi;
            *reinterpret_cast<uint32_t*>(sn + sw128_offset(65, lane / 4) + (lane % 4) * 4) = lo;
          }
          fence_proxy_async_smem();
          __syncwarp();  // (also: zbuf is rewritten only by the next snapshot)
          if (lane == 0) mbar_arrive(&B->sready[(sj + 1) % 2]);
        }
        // o = num / (den + eps), staged in shared memory, stored by TMA
        const int ob = oj % 2;
        wait3(x, &B->oready[ob], (oj / 2) & 1);
        tc_fence_after();
        const uint32_t base = tl + TO + 80 * ob;
        uint32_t n0[32], n1[32], d2[2];
        tmem_ld32(base, n0);
        tmem_ld32(base + 32, n1);
        tmem_ld2(base + D, d2);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->ofree[ob]);
        const float inv = 1.f / (__uint_as_float(d2[0]) + __uint_as_float(d2[1]) + p.eps);
        if (et == 32) bulk_wait_read_all();  // the previous chunk's store has read the staging
        named_bar_sync(1, 128);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<float4*>(out + sw128_offset(row, cc)) =
              make_float4(__uint_as_float(n0[4 * cc]) * inv, __uint_as_float(n0[4 * cc + 1]) * inv,
                          __uint_as_float(n0[4 * cc + 2]) * inv, __uint_as_float(n0[4 * cc + 3]) * inv);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<float4*>(out + BLK + sw128_offset(row, cc)) =
              make_float4(__uint_as_float(n1[4 * cc]) * inv, __uint_as_float(n1[4 * cc + 1]) * inv,
                          __uint_as_float(n1[4 * cc + 2]) * inv, __uint_as_float(n1[4 * cc + 3]) * inv);
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (et == 32 && !*x.abort) {
          const int tok = pc.tok0 + c * C;
          tma_store_3d_ef(&tm_o, out, 0, tok, pc.h);
          tma_store_3d_ef(&tm_o, out + BLK, 32, tok, pc.h);
          bulk_commit();
        }
      }
      if (whole && state_warp) {  // the state after the last advance: S_N, z_N
        wait3(x, &B->sacc, nsa & 1);
        ++nsa;
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32(tl + TS, r0);
        tmem_ld32(tl + TS + 32, r1);
        tmem_ld_wait();
        tc_fence_before();
        if (state_row && pc.tok1 == p.sp.N && !*x.abort) {
#pragma unroll
          for (int i = 0; i < D; ++i) {
            const float f = __uint_as_float(i < 32 ? r0[i] : r1[i - 32]);
            if (row < D) p.S_N[((size_t)pc.h * D + i) * D + row] = f;
            else p.z_N[(size_t)pc.h * D + i] = f;
          }
        }
      }
    }
    if (et == 32) bulk_wait_all();
  } else {  // ---- the state chain: S += [V | 1]^T phi(K), chunk by chunk (one thread)
    if (lane == 0) {
      const uint32_t aOnes = smem_u32(smem + OFF_ONES);
      // The advance of global chunk j (its stage loaded; the running state
      // read), or, for a piece's last chunk, which has none, just this
      // issuer's share of the stage's release.  Chunk j is loaded, so its
      // stage's previous use has been released and the release counts for
      // chunk j (an earlier arrival would count for the previous use, and the
      // stage could be refilled while read).
      auto advance = [&](uint32_t j, bool any) {
        const int s = j % NS;
        if (!wait3(x, &B->full[s], (j / NS) & 1)) return false;
        if (!any) {
          mbar_arrive(&B->empty[s]);
          return true;
        }
        if (DECAY) {  // phi(K) of chunk j rescaled by all four P warps
          for (int q = 0; q < 4; ++q)
            if (!count_reached(x, &B->pdone[q], j + 1)) return false;
        } else if (!wait3(x, &B->xf[s], (j / NS) & 1)) {  // phi applied to K by the phi warps
          return false;
        }
        tc_fence_after();
        const uint32_t st = smem_u32(stage_ptr(smem, s)), vt = st + 2 * BLK;
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks)
          mma_bf16_ss(x.tmem + TS, sdesc_sw128(vt + ks * 2048, aOnes - vt, 1024),
                      sdesc_sw128(st + BLK + ks * 2048, BLK, 1024), ID_DS, 1u);
        mma_commit(&B->sacc);
        mma_commit(&B->empty[s]);
        return true;
      };
      // piece i's entry state is in TMEM once the three state warps have
      // counted it (bounded wait, like the mbarrier waits)
      auto entry_stored = [&](int i) {
        if (*x.abort) return false;
        const uint64_t dl = globaltimer_ns() + mbar_ns;
        while (ld_acquire_cta(&B->epieces) < 3u * (unsigned)(i + 1)) {
          if (*x.abort) return false;
          if (globaltimer_ns() > dl) {
            *x.abort = 1;
            atomicOr(p.status, kStatusTimeout);
            return false;
          }
        }
        tc_fence_after();
        return true;
      };
      uint32_t sj = 0, ntr = 0;
      bool ok = true;
      Piece pc;
      for (int i = 0; ok && run.piece(p.sp, i, &pc); ++i) {
        // a piece's last chunk advances only in the decayed form (whose final
        // state comes from the running state)
        ok = entry_stored(i) && advance(sj, whole || pc.nch > 1);  // chunk 0 reads E in TMEM
        for (int c = 0; ok && c + 1 < pc.nch; ++c, ++ntr)
          ok = wait3(x, &B->tsread, ntr & 1) && advance(sj + c + 1, whole || c + 2 < pc.nch);
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

// agg and E slots, then phi(K)
// the piece totals and the entry states (phi(K) does not go through the
// workspace: the output kernel applies phi to K itself)
size_t prefill_chunked64_workspace_bytes(int B, int H, int N) {
  const Split s = make_split(B * H, N, sm_count());
  return 2 * (size_t)s.BH * s.MPH * SZ * sizeof(float);
}

cudaError_t launch_prefill_chunked64(const PrefillArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mo, a.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C))
    return cudaErrorInvalidValue;
  Params3 p;
  p.sp = make_split(BH, a.N, sms);
  p.eps = a.eps;
  p.S0 = a.S0;
  p.z0 = a.z0;
  p.S_N = a.S_N;
  p.z_N = a.z_N;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.status = a.status ? a.status : &reinterpret_cast<WsHeader*>(ws)->status;
  p.alpha = nullptr;
  p.gam = nullptr;
  const size_t slots = (size_t)BH * p.sp.MPH;
  if (sizeof(WsHeader) + prefill_chunked64_workspace_bytes(a.B, a.H, a.N) > a.ws_bytes)
    return cudaErrorInvalidValue;
  p.agg = reinterpret_cast<float*>(ws + sizeof(WsHeader));
  p.E = p.agg + slots * SZ;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  p.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);

  cudaError_t e = cudaFuncSetAttribute(k1::aggregate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)k1::SMEM);
  auto* const out = a.strict ? k3::output_kernel<false, true> : k3::output_kernel<false, false>;
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

size_t aggregate64_totals_bytes(int B, int H, int N) {
  const Split s = make_split(B * H, N, sm_count());
  return (size_t)s.BH * s.MPH * SZ * sizeof(float);
}

cudaError_t launch_aggregate64_totals(const PrefillArgs& a, float* agg, unsigned* status,
                                      cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  CUtensorMap mk, mv;
  if (!make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C))
    return cudaErrorInvalidValue;
  Params3 p = {};
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

// the decayed form's slots: agg and E, then one decay factor per piece slot
size_t prefill_decay64_workspace_bytes(int B, int H, int N) {
  const Split s = make_split(B * H, N, sm_count());
  const size_t slots = (size_t)s.BH * s.MPH;
  const size_t three = (2 * slots * SZ + slots) * sizeof(float);
  // calls that the two-launch form takes need its workspace
  if (prefill_prefix64_chosen(B, H, N)) {
    const size_t two = prefill_prefix64_decay_workspace_bytes(B, H, N);
    return two > three ? two : three;
  }
  return three;
}

// The entry state of every piece of the d = 64 split, for other kernels that
// walk the same pieces (the gradient): the aggregate and scan launches of the
// plain form into agg and E (slot layout), with S_N and z_N as scratch the
// scan fills; bounded-wait failures go to `status`.  The scan is a
// programmatic dependent, and so may be the launch that follows.
cudaError_t launch_prefill_entry_states64(const PrefillArgs& a, float* agg, float* E, float* S_N, float* z_N,
                                          unsigned* status, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  CUtensorMap mk, mv;
  if (!make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C))
    return cudaErrorInvalidValue;
  Params3 p = {};
  p.sp = make_split(BH, a.N, sms);
  p.S0 = a.S0;
  p.z0 = a.z0;
  p.S_N = S_N;
  p.z_N = z_N;
  p.status = status;
  p.agg = agg;
  p.E = E;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  cudaError_t e = cudaFuncSetAttribute(k1::aggregate_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k1::SMEM);
  if (e != cudaSuccess) return e;
  k1::aggregate_kernel<false><<<p.sp.G, 32 * k1::kWarps, k1::SMEM, stream>>>(mk, mv, p, mbar_ns);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(scan_blocks_per_head<D>(), BH);
  cfg.blockDim = dim3(kScanThreads);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, k2::scan_kernel<false>, p);
}

bool prefill_decay64_supported(const PrefillArgs& a) {
  return a.bf16 && a.dk == 64 && a.dv == 64 && a.N > 0 && get_encode() != nullptr;
}

// The decayed write-then-read prefill.  With a workspace of at least
// prefill_decay64_workspace_bytes: the three launches of the plain form in
// their decayed instantiations (decayed piece totals, the chain
// E' = Gamma E + R, the outputs).  Without one: the output kernel alone, one
// block per head (the whole head is the piece and S0 its entry state).  phi is
// applied to K inside the output kernel either way.  Bounded-wait failures go
// to the library status word.
cudaError_t launch_prefill_decay64(const PrefillArgs& a, const float* alpha, cudaStream_t stream) {
  const int BH = a.B * a.H;
  // calls whose re-read data stays in L2: the two launches of prefill_prefix64.cu
  if (!a.strict && a.workspace && prefill_prefix64_chosen(a.B, a.H, a.N) &&
      a.ws_bytes >= prefill_prefix64_decay_workspace_bytes(a.B, a.H, a.N))
    return launch_prefill_prefix64_decay(a, alpha, stream);
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mo, a.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C))
    return cudaErrorInvalidValue;
  const bool pieces = a.workspace && a.ws_bytes >= prefill_decay64_workspace_bytes(a.B, a.H, a.N);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  Params3 p = {};
  p.sp = make_split(BH, a.N, pieces ? sms : BH);  // without a workspace, block j runs head j
  p.eps = a.eps;
  p.S0 = a.S0;
  p.z0 = a.z0;
  p.S_N = a.S_N;
  p.z_N = a.z_N;
  p.alpha = alpha;
  if (pieces) {
    const size_t slots = (size_t)BH * p.sp.MPH;
    p.agg = static_cast<float*>(a.workspace);
    p.E = p.agg + slots * SZ;
    p.gam = p.E + slots * SZ;
  }
  cudaError_t e = library_status_word(&p.status);
  if (e != cudaSuccess) return e;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  p.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);
  auto* const out = a.strict ? k3::output_kernel<true, true> : k3::output_kernel<true, false>;
  e = cudaFuncSetAttribute(out, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k3::SMEM);
  if (e != cudaSuccess) return e;
  if (!pieces) {
    out<<<p.sp.G, 32 * k3::kWarps, k3::SMEM, stream>>>(mq, mk, mv, mo, p, mbar_ns);
    return cudaGetLastError();
  }
  e = cudaFuncSetAttribute(k1::aggregate_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)k1::SMEM);
  if (e != cudaSuccess) return e;
  // (the decayed aggregate kernel stores no phi(K): its third map is unused)
  k1::aggregate_kernel<true><<<p.sp.G, 32 * k1::kWarps, k1::SMEM, stream>>>(mk, mv, p, mbar_ns);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
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

}  // namespace la
