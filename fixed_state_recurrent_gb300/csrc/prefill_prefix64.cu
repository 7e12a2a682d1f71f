// prefill_prefix64.cu -- causal prefill for dk = dv = 64 on the sm_103a
// tensor cores in two launches: per-chunk prefix tiles, then the outputs.
//
// Operator (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03):
//   o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps),  S_t = S_{t-1} + phi(k_t) v_t^T,
//   z_t = z_{t-1} + phi(k_t),  phi = ELU + 1,  write before read.
// Chunkwise evaluation (page "线性注意力与SSM", section 3), chunk C = 128: the
// outputs of a chunk are the masked phi(Q) phi(K)^T attention inside the chunk
// plus phi(Q) times the state before the chunk.
//
// Work split (prefill_tc_common.cuh): the heads' chunks form one head-major
// sequence, block j of G takes a contiguous run of it, cut at head boundaries
// into pieces.  The state before chunk c of a piece is E + P_c: E the piece's
// entry state (the totals of the head's earlier blocks, zero for a piece that
// starts its head), P_c the piece's own prefix (for a piece that starts its
// head, from S0).
//   prefix_kernel: per chunk the increment [V_c | 1]^T phi(K_c) on the tensor
//      cores (TMEM lanes 0..63 = dS^T, lane 64 = dz), added in fp32 registers
//      to the piece's running prefix; before each chunk the prefix P_c is
//      stored as an operand tile (bf16: rows 0..63 = S^T, row 64 = bf16(z),
//      row 65 = the rest of z), and after the piece its total R (fp32, with S0
//      for a piece that starts its head).  phi(K) (bf16, the layout of K) goes
//      to the workspace too.
//   output_kernel: E of the block's first piece = the sum of the totals of the
//      head's earlier blocks (fp32, then a bf16 tile), built while the first
//      tiles load; the final states.  Per chunk: [scores | num | den] =
//      phi(Q) [phi(K) ; P_c]^T as one N = 208 product (phi(Q) in TMEM),
//      [num | den] += phi(Q) E^T where E is nonzero, P = causal mask of the
//      scores (bf16, in place in TMEM), [num | den] += P [V | 1],
//      o = num / (den + eps).
// No launch carries a state from chunk to chunk on the tensor cores: the
// prefix lives in the registers of the first launch, and the second has no
// chain at all.  V, phi(K) and the tiles are read again from L2 while the call
// fits in it; larger calls take the three launches of prefill_chunked64.cu.
#include "prefill_tc_common.cuh"

#ifdef LA_TRACE
static __device__ unsigned long long g_la_trace[4 * 160 * 64];
#define LA_TRACE_AT(kern, blk, ev)                                                      \
  do {                                                                                 \
    if ((ev) < 64 && (blk) < 160)                                                      \
      g_la_trace[((kern) * 160 + (blk)) * 64 + (ev)] = la::tc::globaltimer_ns();       \
  } while (0)
extern "C" int la_prefill64_trace_read(unsigned long long* host, int n) {
  return cudaMemcpyFromSymbol(host, g_la_trace, (size_t)n * 8) == cudaSuccess ? 0 : -1;
}
extern "C" int la_prefill64_trace_clear() {
  static unsigned long long zeros[4 * 160 * 64];
  return cudaMemcpyToSymbol(g_la_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#else
#define LA_TRACE_AT(kern, blk, ev) ((void)0)
#endif
#define LA_TRACE(kern, ev) LA_TRACE_AT(kern, blockIdx.x, ev)

namespace la {
namespace {

using namespace tc;
using namespace tcp;

constexpr int D = 64;
constexpr int SZ = D * D + D;           // floats per state slot (S^T rows, then z)
constexpr uint32_t BLK = 16384;         // [128 rows x 128 B] swizzled bf16 tile
constexpr int XROWS = 66;               // rows of a state tile that are stored and loaded
constexpr uint32_t XG = XROWS * 128;    // bytes of one prefix tile in the workspace
constexpr uint32_t XT = 80 * 128;       // a state tile in shared memory: [80 x 64] bf16, rows 66.. zero
constexpr uint32_t ONES = 2048;         // [V | 1]'s second atom: 16 rows, column 0 = 1

constexpr uint32_t ID_DS = idesc_bf16_f32(128, D, 1, 1);            // [V | 1]^T phi(K)
constexpr uint32_t ID_SX = idesc_bf16_f32(128, 128 + 80, 0, 0);     // phi(Q) [phi(K) ; P]^T
constexpr uint32_t ID_X = idesc_bf16_f32(128, D + 16, 0, 0);        // phi(Q) E^T
constexpr uint32_t ID_PV = idesc_bf16_f32(128, D + 16, 0, 1);       // P [V | 1]

// Shared-memory descriptor steps along K for one 16-deep MMA: K-major operands
// advance 32 bytes within the swizzle atom, MN-major ones 16 rows (2048 bytes),
// and for [V | 1] the leading-byte offset shrinks by the same 2048 bytes, so
// that the ones atom stays where it is (its 16 rows serve every step).
constexpr uint64_t kStepK16 = 32 >> 4;
constexpr uint64_t kStepRows16 = 2048 >> 4;
constexpr uint64_t kStepMN = (2048 >> 4) - ((uint64_t)(2048 >> 4) << 16);

struct Params {
  Split sp;
  float eps;
  const float* S0;
  const float* z0;
  float* S_N;
  float* z_N;
  unsigned* status;    // sticky error bits (the workspace header's, or the library's)
  float* R;            // [BH * MPH][SZ] piece totals (slot layout)
  uint8_t* P;          // [TC][66][64] bf16 prefix tiles
  float* den;          // [BH][N] den_t = phi(q_t)^T z_t + eps (the output kernel's BWD form only)
  int totals_only;     // the prefix kernel stores neither the prefix tiles nor phi(K)
  // decayed form (S_t = alpha_t S_{t-1} + phi(k_t) v_t^T, z likewise):
  const float* alpha;  // [BH][N] per-token decay
  float* G;            // [TC][128] per chunk row: g_t, the inclusive sum of log2 alpha over the chunk
  float* gamc;         // [TC] per chunk: the decay from its piece's start to the chunk's start
  float* gam;          // [BH * MPH] per piece slot: the decay over the whole piece
  int force_wait;      // test hook: the output kernel waits once on a barrier that nothing completes
};

struct Ctx {
  unsigned* status;
  volatile int* abort;
  uint32_t tmem;
  unsigned long long mbar_ns;
};

// Bounded wait.  false once the block has given up (this wait ran out of time
// and recorded a timeout in the status word, or another role's did).  After
// that no role starts new asynchronous work, every role still runs its loops,
// with each wait returning at once, so that the named barriers of a warp group
// stay matched, and the issuers drain what they started before the tensor
// memory is freed.
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

// The ones atom of [V | 1]: 16 token rows whose column 0 is 1.  Contains a
// block-wide barrier.
__device__ __forceinline__ void init_ones_atom(uint8_t* ones, int tid, int nthreads) {
  for (int i = tid; i < (int)(ONES / 16); i += nthreads)
    reinterpret_cast<uint4*>(ones)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (tid < 16) *reinterpret_cast<uint16_t*>(ones + sw128_offset(tid, 0)) = 0x3F80u;  // bf16 1.0
}

__device__ __forceinline__ void free_tmem(const Ctx& x, int warp, uint32_t ncols) {
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(x.tmem, ncols);
  }
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

// Eight bf16 of one state row, K-major swizzled operand tile.
__device__ __forceinline__ void put8(uint8_t* tile, int row, int chunk, const float* v) {
  *reinterpret_cast<uint4*>(tile + sw128_offset(row, chunk)) =
      make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                 pack_bf16x2(v[6], v[7]));
}

// ===========================================================================
// Prefix tiles and piece totals

namespace pfx {

constexpr int NS = 4;                       // K | V stages (decayed form: K | V | weights)
constexpr uint32_t PST = 9 * 1024;          // staging of one prefix tile (66 rows, 1024-byte aligned)
template <bool DECAY>
struct Layout {
  static constexpr uint32_t STAGE = DECAY ? 3 * BLK : 2 * BLK;
  static constexpr uint32_t OFF_PST = NS * STAGE;
  static constexpr uint32_t OFF_ONES = OFF_PST + 2 * PST;
  static constexpr uint32_t OFF_BAR = OFF_ONES + ONES;
  static constexpr uint32_t OFF_DBAR = OFF_BAR + 512;  // decayed form's extra barriers
  static constexpr uint32_t SMEM = OFF_BAR + (DECAY ? 1024 : 512) + 1024;
  static_assert(PST >= XG && OFF_PST % 1024 == 0 && PST % 1024 == 0, "prefix staging");
  static_assert(SMEM <= 227 * 1024, "shared memory per block");
};
constexpr uint32_t SMEM_PLAIN = Layout<false>::SMEM;
constexpr uint32_t SMEM_DECAY = Layout<true>::SMEM;
// 0 TMA, 1 MMA, 2-9 phi(K) (half a row per thread), 10-13 prefix (TMEM lanes
// 0..64 on warps 10, 12, 13), 14 phi(K) stores
constexpr int kWarps = 15;
constexpr int NB = 4;                       // TMEM increment buffers, 64 columns each
constexpr uint32_t kCols = 256;

struct Bars {
  uint64_t full[NS], xf[NS];
  uint64_t empty[NS];    // the stage's product done and its phi(K) store read: 2 arrivals
  uint64_t dsready[NB];  // increment in buffer b     (MMA -> prefix warps)
  uint64_t dsfree[NB];   // buffer b read out         (three prefix warps -> MMA)
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
  float4 zbuf[16];       // z, handed from its TMEM lane to the whole warp
};
static_assert(sizeof(Bars) <= 512, "barrier area");
// decayed form: each chunk's decay gamma_C (phi warps -> prefix warps, a ring
// of eight: the phi warps run at most seven chunks ahead of the prefix warps)
struct DBars {
  uint64_t gready[8];
  float gring[8];
};

// DECAY: per chunk the phi warps also take g_t (the inclusive sum of
// log2 alpha over the chunk, a zero alpha taken as 1e-30), scale V's rows by
// w_s = 2^(g_C - g_s) (the decay from token s to the chunk's end, <= 1) and
// write w_s as the only column of a weights block, so that the product
// [w V | w]^T phi(K) is the chunk's decayed increment; phi(K) itself stays
// unscaled (the output kernel's scores).  The prefix advances as
// P <- gamma_C P + increment.
template <bool DECAY>
__global__ void __launch_bounds__(32 * kWarps, 1)
prefix_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_phik, const __grid_constant__ CUtensorMap tm_p,
              const Params p, const unsigned long long mbar_ns) {
  using L = Layout<DECAY>;
  constexpr uint32_t STAGE = L::STAGE, OFF_PST = L::OFF_PST, OFF_ONES = L::OFF_ONES;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array by pointer
  // arithmetic so that accesses through it stay shared-space accesses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* B = reinterpret_cast<Bars*>(smem + L::OFF_BAR);
  DBars* DB = reinterpret_cast<DBars*>(smem + L::OFF_DBAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Run run(p.sp, blockIdx.x);
  if (threadIdx.x == 0) LA_TRACE(0, 0);
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
    if (DECAY)
      for (int q = 0; q < 8; ++q) mbar_init(&DB->gready[q], 1);
    B->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_phik);
    tma_prefetch_desc(&tm_p);
  }
  if (DECAY)  // the weights blocks: only column 0 is ever rewritten
    for (int i = threadIdx.x; i < (int)(NS * BLK / 16); i += 32 * kWarps) {
      const int st = i / (BLK / 16), k = i % (BLK / 16);
      reinterpret_cast<uint4*>(smem + st * STAGE + 2 * BLK)[k] = make_uint4(0, 0, 0, 0);
    }
  uint32_t pre = 0;  // loads issued during the set-up (thread 0)
  if (threadIdx.x == 0) {
    // This launch is a programmatic dependent of whatever ran before it on
    // the stream (so that its set-up overlaps that kernel's last blocks): no
    // global memory is touched before the wait.
    pdl_wait();
    Piece pc;
    for (int i = 0; pre < NS && run.piece(p.sp, i, &pc); ++i)
      for (int c = 0; pre < NS && c < pc.nch; ++c, ++pre) {
        uint8_t* st = smem + pre * STAGE;
        const int tok = pc.tok0 + c * C;
        mbar_arrive_expect_tx(&B->full[pre], 2 * BLK);
        tma_load_3d_ef(st, &tm_k, 0, tok, pc.h, &B->full[pre]);
        tma_load_3d(st + BLK, &tm_v, 0, tok, pc.h, &B->full[pre]);  // V: read again by the output kernel
      }
  }
  init_ones_atom(smem + OFF_ONES, threadIdx.x, 32 * kWarps);
  if (warp == 1) {
    tmem_alloc(&B->tmem_slot, kCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const Ctx x{p.status, &B->abort, *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot), mbar_ns};
  pdl_launch_dependents();  // the output kernel may be scheduled now; it waits for this grid's results
  pdl_wait();               // (see thread 0's loads above)
  if (threadIdx.x == 0) LA_TRACE(0, 1);

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer: K, V (the first `pre` went out above)
      uint32_t sj = 0, issued = pre;
      Piece pc;
      for (int i = 0; run.piece(p.sp, i, &pc); ++i)
        for (int c = 0; c < pc.nch; ++c, ++sj) {
          const int s = sj % NS;
          if (sj < pre) continue;
          if (sj >= NS && !waitb(x, &B->empty[s], ((sj / NS) - 1) & 1)) break;
          uint8_t* st = smem + s * STAGE;
          const int tok = pc.tok0 + c * C;
          mbar_arrive_expect_tx(&B->full[s], 2 * BLK);
          tma_load_3d_ef(st, &tm_k, 0, tok, pc.h, &B->full[s]);
          tma_load_3d(st + BLK, &tm_v, 0, tok, pc.h, &B->full[s]);
          ++issued;
        }
      if (*x.abort) drain_loads<NS>(B->full, issued, mbar_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA: D[b] = [V | 1]^T phi(K), fresh per chunk
      const uint32_t aOnes = smem_u32(smem + OFF_ONES);
      const uint32_t total = (uint32_t)(run.b - run.a);
      for (uint32_t j = 0; j < total; ++j) {
        const int s = j % NS, b = j % NB;
        if (j >= NB && !waitb(x, &B->dsfree[b], ((j / NB) - 1) & 1)) break;
        if (!waitb(x, &B->xf[s], (j / NS) & 1)) break;
        tc_fence_after();
        const uint32_t kt = smem_u32(smem + s * STAGE), vt = kt + BLK;
        const uint64_t b0 = sdesc_sw128(kt, BLK, 1024);
        if (DECAY) {  // [w V | weights block]: two 64-row atoms along M, BLK apart
          const uint64_t a0 = sdesc_sw128(vt, BLK, 1024);
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks)
            mma_bf16_ss(x.tmem + 64 * b, a0 + ks * kStepRows16, b0 + ks * kStepRows16, ID_DS, ks > 0 ? 1u : 0u);
        } else {
          const uint64_t a0 = sdesc_sw128(vt, aOnes - vt, 1024);
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks)
            mma_bf16_ss(x.tmem + 64 * b, a0 + ks * kStepMN, b0 + ks * kStepRows16, ID_DS, ks > 0 ? 1u : 0u);
        }
        mma_commit(&B->empty[s]);
        mma_commit(&B->dsready[b]);
        if (j < 8) LA_TRACE(0, 18 + j);
      }
      if (*x.abort) {
        int never = 0;
        mma_commit(&B->drain);
        mbar_wait(&B->drain, 0, globaltimer_ns() + mbar_ns, &never);
      }
    }
    __syncwarp();
  } else if (warp < 10) {  // ---- phi on K, half a tile row per thread
    const int t = threadIdx.x - 64, r = t >> 1, c0 = 4 * (t & 1);
    uint32_t sj = 0;
    // decayed form: every phi warp scans the whole chunk itself (lane l holds
    // tokens 4 l .. 4 l + 3; alpha 1 past the sequence), so that no barrier
    // between the warps sits on the chain; alpha is loaded a chunk ahead
    const uint32_t total = (uint32_t)(run.b - run.a);
    auto alpha4 = [&](uint32_t j) {
      float4 a = make_float4(1.f, 1.f, 1.f, 1.f);
      if (DECAY && j < total) {
        const long long gi = run.a + j;
        const int tok = (int)(gi % p.sp.NC) * C + 4 * lane;
        const float* ap = p.alpha + (size_t)(gi / p.sp.NC) * p.sp.N + tok;
        if (tok + 3 < p.sp.N && ((reinterpret_cast<uintptr_t>(ap) & 15) == 0)) {
          a = __ldg(reinterpret_cast<const float4*>(ap));
        } else {
          if (tok < p.sp.N) a.x = __ldg(ap);
          if (tok + 1 < p.sp.N) a.y = __ldg(ap + 1);
          if (tok + 2 < p.sp.N) a.z = __ldg(ap + 2);
          if (tok + 3 < p.sp.N) a.w = __ldg(ap + 3);
        }
      }
      return a;
    };
    float4 anext = alpha4(0);
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i)
      for (int c = 0; c < pc.nch; ++c, ++sj) {
        const int s = sj % NS;
        const int tok = pc.tok0 + c * C, valid = pc.tok1 - tok;
        float g = 0.f, tot = 0.f;
        if (DECAY) {  // g of this thread's row r, and of the chunk's last token
          const float4 acur = anext;
          anext = alpha4(sj + 1);
          const float l0 = __log2f(fmaxf(acur.x, 1e-30f)), l1 = __log2f(fmaxf(acur.y, 1e-30f));
          const float l2 = __log2f(fmaxf(acur.z, 1e-30f)), l3 = __log2f(fmaxf(acur.w, 1e-30f));
          const float p0 = l0, p1 = l0 + l1, p2 = p1 + l2, p3 = p2 + l3;
          float sc = p3;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xFFFFFFFFu, sc, off);
            if (lane >= off) sc += y;
          }
          const float ex = sc - p3;  // the sum over the lanes before this one
          tot = __shfl_sync(0xFFFFFFFFu, sc, 31);
          // row r's value from lane r / 4, element r % 4
          const float g0 = __shfl_sync(0xFFFFFFFFu, ex + p0, r >> 2);
          const float g1 = __shfl_sync(0xFFFFFFFFu, ex + p1, r >> 2);
          const float g2 = __shfl_sync(0xFFFFFFFFu, ex + p2, r >> 2);
          const float g3 = __shfl_sync(0xFFFFFFFFu, ex + p3, r >> 2);
          const int e = r & 3;
          g = e == 0 ? g0 : e == 1 ? g1 : e == 2 ? g2 : g3;
        }
        if (!waitb_warp(x, &B->full[s], (sj / NS) & 1)) continue;
        if (t == 0 && sj < 8) LA_TRACE(0, 2 + sj);
        phi_row<4>(smem + s * STAGE, r, c0, valid);
        if (DECAY) {
          const float w = exp2_ftz(tot - g);
          uint8_t* vt = smem + s * STAGE + BLK;
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // V's half row times w
            uint4 u = *reinterpret_cast<const uint4*>(vt + sw128_offset(r, c0 + q));
            uint32_t* e = &u.x;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              e[k] = pack_bf16x2(__uint_as_float(e[k] << 16) * w, __uint_as_float(e[k] & 0xFFFF0000u) * w);
            *reinterpret_cast<uint4*>(vt + sw128_offset(r, c0 + q)) = u;
          }
          if (c0 == 0) {
            *reinterpret_cast<uint4*>(vt + BLK + sw128_offset(r, 0)) = make_uint4(pack_bf16x2(w, 0.f), 0u, 0u, 0u);
            if (!*x.abort) p.G[(size_t)(run.a + sj) * C + r] = g;
          }
          if (t == 0) {  // the chunk's decay, for the prefix warps
            DB->gring[sj % 8] = exp2_ftz(tot);
            mbar_arrive(&DB->gready[sj % 8]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (t == 0 && sj < 8) LA_TRACE(0, 10 + sj);
        if (lane == 0) mbar_arrive(&B->xf[s]);
      }
  } else if (warp < 14) {
    // ---- the running prefix.  State lane `row` (0..64: quadrants 0..2) holds
    // slot row `row` in fp32.  Per chunk: the prefix before it as a bf16 tile,
    // staged and stored by TMA (thread 352); then the chunk's increment out of
    // TMEM added.  After a piece's last chunk its total R in fp32.
    const int quad = warp % 4, row = 32 * quad + lane, et = threadIdx.x - 320;
    const bool state_warp = quad <= 2;
    const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
    float acc[D];
    uint32_t sj = 0;
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i) {
      float gpiece = 1.f;  // decayed form: the decay from the piece's start to the current chunk
      // a piece that starts its head starts from S0, z0 (row `row` of S^T: column `row` of S0)
#pragma unroll
      for (int q = 0; q < D; ++q) acc[q] = 0.f;
      if (state_warp && pc.tok0 == 0) {
        if (row < D && p.S0) {
#pragma unroll
          for (int q = 0; q < D; ++q) acc[q] = __ldg(p.S0 + ((size_t)pc.h * D + q) * D + row);
        } else if (row == D && p.z0) {
#pragma unroll
          for (int q = 0; q < D; ++q) acc[q] = __ldg(p.z0 + (size_t)pc.h * D + q);
        }
      }
      for (int c = 0; c < pc.nch; ++c, ++sj) {
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
          if (quad == 2) {  // z -> rows 64 (hi) and 65 (lo), split by the whole warp
            __syncwarp();
            const float2 zz = reinterpret_cast<const float2*>(B->zbuf)[lane];  // z[2 lane], z[2 lane + 1]
            const uint32_t hi = pack_bf16x2(zz.x, zz.y);
            const uint32_t lo = pack_bf16x2(zz.x - __uint_as_float(hi << 16),
                                            zz.y - __uint_as_float(hi & 0xFFFF0000u));
            *reinterpret_cast<uint32_t*>(stg + sw128_offset(64, lane / 4) + (lane % 4) * 4) = hi;
            *reinterpret_cast<uint32_t*>(stg + sw128_offset(65, lane / 4) + (lane % 4) * 4) = lo;
            __syncwarp();  // zbuf is rewritten only after every lane has read it
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (et == 32 && !*x.abort && !p.totals_only) {
          tma_store_3d(&tm_p, stg, 0, 0, (int)(run.a + sj));
          bulk_commit();
          if (DECAY) p.gamc[run.a + sj] = gpiece;
        }
        const int b = sj % NB;
        const bool got = waitb_warp(x, &B->dsready[b], (sj / NB) & 1);
        float gC = 1.f;
        if (DECAY && waitb_warp(x, &DB->gready[sj % 8], (sj / 8) & 1)) gC = DB->gring[sj % 8];
        gpiece *= gC;
        if (state_warp) {
          if (got) {
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tl + 64 * b, r0);
            tmem_ld32(tl + 64 * b + 32, r1);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              acc[q] = DECAY ? fmaf(gC, acc[q], __uint_as_float(r0[q])) : acc[q] + __uint_as_float(r0[q]);
              acc[32 + q] = DECAY ? fmaf(gC, acc[32 + q], __uint_as_float(r1[q])) : acc[32 + q] + __uint_as_float(r1[q]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && got) mbar_arrive(&B->dsfree[b]);
        }
        if (row == 0 && sj < 8) LA_TRACE(0, 26 + sj);
      }
      if (state_warp && row <= D && !*x.abort) {  // the piece's total
        float4* dst = reinterpret_cast<float4*>(p.R + (size_t)pc.slot * SZ + row * D);
#pragma unroll
        for (int q = 0; q < 16; ++q)
          __stcg(dst + q, make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]));
      }
      if (DECAY && et == 32 && !*x.abort) p.gam[pc.slot] = gpiece;  // the decay over the whole piece
    }
    if (et == 32) bulk_wait_all();
  } else if (lane == 0) {  // ---- phi(K) -> workspace; the stage is released once read
    uint32_t sj = 0;
    Piece pc;
    for (int i = 0; run.piece(p.sp, i, &pc); ++i)
      for (int c = 0; c < pc.nch; ++c, ++sj) {
        const int s = sj % NS;
        if (!waitb(x, &B->xf[s], (sj / NS) & 1)) continue;
        if (!p.totals_only) {
          tma_store_3d(&tm_phik, smem + s * STAGE, 0, pc.tok0 + c * C, pc.h);
          bulk_commit();
          bulk_wait_read_all();
        }
        mbar_arrive(&B->empty[s]);
      }
    bulk_wait_all();
  }
  free_tmem(x, warp, kCols);
  if (threadIdx.x == 0) LA_TRACE(0, 39);
}

}  // namespace pfx

// ===========================================================================
// Outputs

namespace out {

constexpr int NS = 3;                              // Q | phi(K) | P | V stages
constexpr uint32_t OFF_K = BLK;
constexpr uint32_t OFF_P = 2 * BLK;                // P right after phi(K): one operand [phi(K) ; P]
constexpr uint32_t OFF_V = 2 * BLK + XT;
constexpr uint32_t OFF_G = 3 * BLK + XT;           // decayed form: g_t of the chunk's rows (128 floats)
template <bool DECAY>
struct Layout {
  static constexpr uint32_t STAGE = 3 * BLK + XT + (DECAY ? 1024 : 0);
  static constexpr uint32_t OFF_E = NS * STAGE;      // the first piece's entry state (bf16 tile)
  static constexpr uint32_t OFF_OUT = OFF_E + XT;    // output staging: two [128 x 32] fp32 boxes
  static constexpr uint32_t OFF_ONES = OFF_OUT + 2 * BLK;
  static constexpr uint32_t OFF_BAR = OFF_ONES + ONES;
  static constexpr uint32_t SMEM = OFF_BAR + 512 + 1024;
  static_assert(STAGE % 1024 == 0 && OFF_P % 1024 == 0 && OFF_V % 1024 == 0 && OFF_E % 1024 == 0 &&
                OFF_OUT % 1024 == 0 && OFF_ONES % 1024 == 0, "swizzled tile alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory per block");
};
constexpr uint32_t SMEM_PLAIN = Layout<false>::SMEM;
constexpr uint32_t SMEM_DECAY = Layout<true>::SMEM;
// 0 TMA, 1 MMA, 2-9 phi(Q) and the mask, 10-13 output epilogue; 2-14 build
// the entry state and store the final states first (14 then has nothing left
// to do)
constexpr int kWarps = 15;
constexpr uint32_t kCols = 512;
constexpr uint32_t TB = 208;   // buffer b at 208 b: scores then P (128 columns),
constexpr uint32_t TOO = 128;  //   then [num | den] (80 columns) at +128
constexpr uint32_t TQ = 416;   // phi(Q) of chunk j (bf16 pairs, 32 columns) at 416 + 32 (j % 3)

struct Bars {
  uint64_t qfull[NS];   // Q loaded                              (TMA -> phi warps)
  uint64_t full[NS];    // phi(K), P, V loaded                   (TMA -> MMA)
  uint64_t xf[NS];      // phi(Q) in TMEM: eight warps           (phi warps -> MMA)
  uint64_t empty[NS];   // the stage's products done             (MMA -> TMA)
  uint64_t accB[2];     // scores and state part in buffer b     (MMA -> mask)
  uint64_t pready[2];   // P in buffer b: eight warps            (mask -> MMA)
  uint64_t oready[2];   // num, den in buffer b                  (MMA -> epilogue)
  uint64_t ofree[2];    // num, den read: four warps             (epilogue -> MMA)
  uint64_t eready;      // entry-state tile written: 13 warps    (warps 2..14 -> MMA)
  uint64_t drain;
  uint64_t never;       // completed by nothing (the forced-timeout test hook)
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier area");

// The entry state E of the block's first piece: the sum, in order, of the
// totals of the head's earlier blocks (which already hold S0), as a bf16 tile
// in shared memory (left zero when there are none).  If that piece also ends
// its head, E plus the piece's own total is its final state, which goes to T
// ([64][65] fp32, transposed) and z_N.  Thread t of nthr, after the earlier
// launch's results are visible; each thread keeps up to fifteen loads in
// flight.  Returns whether T holds a final state.
// DECAY: `wts` holds w_k = prod_{k < k' < npred} Gamma_k' for the earlier
// slots k and, at [npred], the first piece's own decay: E = sum_k w_k R_k, and
// the final state is Gamma E + R.
template <bool DECAY>
__device__ __forceinline__ bool build_entry(const Params& p, const Run& run, uint8_t* et, float* T,
                                            int t, int nthr, const float* wts) {
  Piece pc;
  if (!run.piece(p.sp, 0, &pc)) return false;
  const int npred = run.idx0;
  const bool last = pc.tok1 == p.sp.N;
  if (npred == 0 && !last) return false;
  const float4* Rh = reinterpret_cast<const float4*>(p.R + (size_t)pc.h * p.sp.MPH * SZ);
  const int nsum = npred + (last ? 1 : 0);  // slots read: the earlier blocks, then the own total
  for (int f0 = t; f0 < SZ / 4; f0 += 3 * nthr) {  // float4 f: slot row f / 16, columns 4 (f % 16)..
    float4 e[3], fin[3];
#pragma unroll
    for (int u = 0; u < 3; ++u) e[u] = fin[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < nsum; k0 += 5) {
      float4 r[3][5];
#pragma unroll
      for (int u = 0; u < 3; ++u)
#pragma unroll
        for (int kk = 0; kk < 5; ++kk)
          r[u][kk] = (f0 + u * nthr < SZ / 4 && k0 + kk < nsum)
                         ? __ldcg(Rh + (size_t)(k0 + kk) * (SZ / 4) + f0 + u * nthr)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 3; ++u)
#pragma unroll
        for (int kk = 0; kk < 5; ++kk) {
          if (k0 + kk < npred) {
            if (DECAY) {
              const float wk = wts[k0 + kk];
              e[u].x = fmaf(wk, r[u][kk].x, e[u].x); e[u].y = fmaf(wk, r[u][kk].y, e[u].y);
              e[u].z = fmaf(wk, r[u][kk].z, e[u].z); e[u].w = fmaf(wk, r[u][kk].w, e[u].w);
            } else {
              e[u].x += r[u][kk].x; e[u].y += r[u][kk].y; e[u].z += r[u][kk].z; e[u].w += r[u][kk].w;
            }
          } else if (k0 + kk == npred) {  // the own total (only when the head ends here)
            fin[u] = r[u][kk];
          }
        }
    }
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      const int f = f0 + u * nthr;
      if (f >= SZ / 4) continue;
      const int row = f / 16, col = 4 * (f % 16);
      if (npred > 0) {
        uint2 hi;
        hi.x = pack_bf16x2(e[u].x, e[u].y);
        hi.y = pack_bf16x2(e[u].z, e[u].w);
        if (row < D) {
          *reinterpret_cast<uint2*>(et + sw128_offset(row, col / 8) + (col % 8) * 2) = hi;
        } else {  // z: hi in row 64, lo in row 65
          uint2 lo;
          lo.x = pack_bf16x2(e[u].x - __uint_as_float(hi.x << 16), e[u].y - __uint_as_float(hi.x & 0xFFFF0000u));
          lo.y = pack_bf16x2(e[u].z - __uint_as_float(hi.y << 16), e[u].w - __uint_as_float(hi.y & 0xFFFF0000u));
          *reinterpret_cast<uint2*>(et + sw128_offset(64, col / 8) + (col % 8) * 2) = hi;
          *reinterpret_cast<uint2*>(et + sw128_offset(65, col / 8) + (col % 8) * 2) = lo;
        }
      }
      if (last) {
        const float gw = DECAY ? wts[npred] : 1.f;
        const float4 v = make_float4(fmaf(gw, e[u].x, fin[u].x), fmaf(gw, e[u].y, fin[u].y),
                                     fmaf(gw, e[u].z, fin[u].z), fmaf(gw, e[u].w, fin[u].w));
        if (row < D) {
          T[(col + 0) * (D + 1) + row] = v.x;
          T[(col + 1) * (D + 1) + row] = v.y;
          T[(col + 2) * (D + 1) + row] = v.z;
          T[(col + 3) * (D + 1) + row] = v.w;
        } else {
          reinterpret_cast<float4*>(p.z_N + (size_t)pc.h * D)[col / 4] = v;
        }
      }
    }
  }
  return last;
}

// S_N of head h from T (written by the same nthr threads before a barrier).
__device__ __forceinline__ void store_S_from_T(const Params& p, int h, const float* T, int t, int nthr) {
  for (int g = t; g < D * D / 4; g += nthr) {  // S_N[i][4 g' ..], i = g / 16
    const int ii = g / 16, j0 = 4 * (g % 16);
    const float* src = T + ii * (D + 1) + j0;
    reinterpret_cast<float4*>(p.S_N + (size_t)h * D * D)[g] = make_float4(src[0], src[1], src[2], src[3]);
  }
}

// The final states of the heads that start and end in this block (pieces
// after the first): their own totals, through T like the first piece's.
// Threads t of nthr, a named barrier `bar` of them.
__device__ __forceinline__ void store_final_later(const Params& p, const Run& run, float* T, int t,
                                                  int nthr, int bar) {
  Piece pc;
  for (int i = 1; run.piece(p.sp, i, &pc); ++i) {
    if (pc.tok1 != p.sp.N) continue;
    const float4* Rs = reinterpret_cast<const float4*>(p.R + (size_t)pc.slot * SZ);
    for (int f = t; f < SZ / 4; f += nthr) {
      const float4 v = __ldcg(Rs + f);
      const int row = f / 16, col = 4 * (f % 16);
      if (row < D) {
        T[(col + 0) * (D + 1) + row] = v.x;
        T[(col + 1) * (D + 1) + row] = v.y;
        T[(col + 2) * (D + 1) + row] = v.z;
        T[(col + 3) * (D + 1) + row] = v.w;
      } else {
        reinterpret_cast<float4*>(p.z_N + (size_t)pc.h * D)[col / 4] = v;
      }
    }
    named_bar_sync(bar, nthr);
    store_S_from_T(p, pc.h, T, t, nthr);
    named_bar_sync(bar, nthr);  // T is free again
  }
}

// Q, phi(K), P, V and o are touched once here and go through TMA with the
// evict-first L2 policy.  BWD (the gradient's second launch): den goes to
// p.den, o out as bf16 (tm_o) and the entry-state tile to slot blockIdx.x of
// tm_e.  STRICT: read before write (token t reads the state before its own
// write: keys s < t inside the chunk).  DECAY: S_t = alpha_t S_{t-1} +
// phi(k_t) v_t^T; with g_t the inclusive sum of log2 alpha over the chunk
// (from the prefix kernel, with each stage's tiles) the state before the chunk
// enters token t as 2^g_t (P_c + Gamma_c E) (Gamma_c: the decay from the
// piece's start, applied to a copy of phi(Q) in shared memory for the E
// product) and key s <= t with weight 2^(g_t - g_s) <= 1: the mask warps
// weight the scores and scale the state part of the row by 2^g_t before
// P [V | 1] is added.
template <bool BWD, bool STRICT, bool DECAY>
__global__ void __launch_bounds__(32 * kWarps, 1)
output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_phik,
              const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_e,
              const Params p, const unsigned long long mbar_ns) {
  using OL = Layout<DECAY>;
  constexpr uint32_t STAGE = OL::STAGE, OFF_E = OL::OFF_E, OFF_OUT = OL::OFF_OUT, OFF_ONES = OL::OFF_ONES;
  constexpr uint32_t XB = 2 * BLK + XG + (DECAY ? C * 4 : 0);  // bytes of a stage's `full`
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* B = reinterpret_cast<Bars*>(smem + OL::OFF_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Run run(p.sp, blockIdx.x);
  const int total = (int)(run.b - run.a);
  Piece pc0;
  const bool have0 = run.piece(p.sp, 0, &pc0);
  const int nE = (have0 && run.idx0 > 0) ? pc0.nch : 0;  // chunks with a nonzero entry state
  if (threadIdx.x == 0) LA_TRACE(2, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&B->qfull[s], 1);
      mbar_init(&B->full[s], 1);
      mbar_init(&B->xf[s], 8);
      mbar_init(&B->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B->accB[b], 1);
      mbar_init(&B->pready[b], 8);
      mbar_init(&B->oready[b], 1);
      mbar_init(&B->ofree[b], 4);
    }
    mbar_init(&B->eready, kWarps - 2);
    mbar_init(&B->drain, 1);
    mbar_init(&B->never, 1);
    B->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_phik);
    tma_prefetch_desc(&tm_p);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
    if (BWD) tma_prefetch_desc(&tm_e);
  }
  // The first stages' Q and V (inputs of the call) go out before the earlier
  // launch has finished, so that phi(Q) of the first chunks is ready when it
  // is; each stage's `full` expects V, phi(K) and P, so phi(K) and P join it
  // once they may be read.
  int pre = 0;
  if (threadIdx.x == 0) {
    Piece pc;
    for (int i = 0; pre < NS && run.piece(p.sp, i, &pc); ++i)
      for (int c = 0; pre < NS && c < pc.nch; ++c, ++pre) {
        uint8_t* st = smem + pre * STAGE;
        const int tok = pc.tok0 + c * C;
        mbar_arrive_expect_tx(&B->qfull[pre], BLK);
        tma_load_3d_ef(st, &tm_q, 0, tok, pc.h, &B->qfull[pre]);
        mbar_arrive_expect_tx(&B->full[pre], XB);
        tma_load_3d_ef(st + OFF_V, &tm_v, 0, tok, pc.h, &B->full[pre]);
      }
  }
  // rows 66..79 of every stage's P tile and of the E tile: zero (read by the
  // MMAs, written by nothing); the E tile all zero until it is built
  for (int i = threadIdx.x; i < NS * (int)(XT - XG) / 16; i += 32 * kWarps) {
    const int s = i / ((XT - XG) / 16), k = i % ((XT - XG) / 16);
    reinterpret_cast<uint4*>(smem + s * STAGE + OFF_P + XG)[k] = make_uint4(0, 0, 0, 0);
  }
  for (int i = threadIdx.x; i < (int)(XT / 16); i += 32 * kWarps)
    reinterpret_cast<uint4*>(smem + OFF_E)[i] = make_uint4(0, 0, 0, 0);
  init_ones_atom(smem + OFF_ONES, threadIdx.x, 32 * kWarps);
  if (warp == 1) {
    tmem_alloc(&B->tmem_slot, kCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();  // a following launch may set up while this one runs
  const Ctx x{p.status, &B->abort, *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot), mbar_ns};

  // The entry-state tile, needed by the first products, and the final states:
  // warps 2..14, the phi warps once the first chunks' phi(Q) is in TMEM.
  auto entry_part = [&]() {
    pdl_wait();  // the piece totals of the earlier launch are complete
    const int t = threadIdx.x - 64, nthr = 32 * (kWarps - 2);
    if (t == 0) LA_TRACE(1, 0);
    float* T = reinterpret_cast<float*>(smem + OFF_OUT);  // the output staging, free until the epilogue
    float* wts = T + D * (D + 1);  // decayed form: the weights of the earlier totals, after T
    if (DECAY) {
      if (t == 0 && have0) {
        const int n = run.idx0;
        const float* gm = p.gam + (size_t)pc0.h * p.sp.MPH;
        float acc = 1.f;
        for (int k = n - 1; k >= 0; --k) {  // w_k = prod of the decays after slot k
          wts[k] = acc;
          acc *= __ldcg(gm + k);
        }
        wts[n] = __ldcg(gm + n);  // the first piece's own decay (for its final state)
      }
      named_bar_sync(6, nthr);
    }
    const bool last = build_entry<DECAY>(p, run, smem + OFF_E, T, t, nthr, wts);
    if (t == 0) LA_TRACE(1, 1);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&B->eready);
    if (last) {
      Piece pc;
      run.piece(p.sp, 0, &pc);
      named_bar_sync(6, nthr);
      store_S_from_T(p, pc.h, T, t, nthr);
      named_bar_sync(6, nthr);
    }
    store_final_later(p, run, T, t, nthr, 6);
  };

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      LA_TRACE(2, 1);
      pdl_wait();  // phi(K) and the prefix tiles of the earlier launch are complete
      LA_TRACE(2, 2);
      {
        Piece pc;
        int j = 0;
        for (int i = 0; j < pre && run.piece(p.sp, i, &pc); ++i)
          for (int c = 0; j < pre && c < pc.nch; ++c, ++j) {
            uint8_t* st = smem + j * STAGE;
            tma_load_3d_ef(st + OFF_K, &tm_phik, 0, pc.tok0 + c * C, pc.h, &B->full[j]);
            tma_load_3d_ef(st + OFF_P, &tm_p, 0, 0, (int)(run.a + j), &B->full[j]);
            if (DECAY) bulk_load(st + OFF_G, p.G + (size_t)(run.a + j) * C, C * 4, &B->full[j]);
          }
      }
      uint32_t sj = 0, issued = pre;
      Piece pc;
      for (int i = 0; run.piece(p.sp, i, &pc); ++i)
        for (int c = 0; c < pc.nch; ++c, ++sj) {
          const int s = sj % NS;
          if ((int)sj < pre) continue;
          if (!waitb(x, &B->empty[s], ((sj / NS) - 1) & 1)) break;
          uint8_t* st = smem + s * STAGE;
          const int tok = pc.tok0 + c * C;
          mbar_arrive_expect_tx(&B->qfull[s], BLK);
          tma_load_3d_ef(st, &tm_q, 0, tok, pc.h, &B->qfull[s]);
          mbar_arrive_expect_tx(&B->full[s], XB);
          tma_load_3d_ef(st + OFF_K, &tm_phik, 0, tok, pc.h, &B->full[s]);
          tma_load_3d_ef(st + OFF_P, &tm_p, 0, 0, (int)(run.a + sj), &B->full[s]);
          tma_load_3d_ef(st + OFF_V, &tm_v, 0, tok, pc.h, &B->full[s]);
          if (DECAY) bulk_load(st + OFF_G, p.G + (size_t)(run.a + sj) * C, C * 4, &B->full[s]);
          ++issued;
        }
      if (*x.abort) {
        drain_loads<NS>(B->qfull, issued, mbar_ns);
        drain_loads<NS>(B->full, issued, mbar_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issue
      // Per chunk a: [S | O] of buffer a % 2 = phi(Q) [phi(K) ; P_a]^T (N = 208),
      // O += phi(Q) E^T for the chunks of a first piece that has earlier
      // blocks, then O += P [V | 1].  Jobs in whichever order they become
      // ready (the products of chunk ap first): the first products of a need
      // phi(Q) of a, the stage's other tiles, and buffer a % 2 read by the
      // epilogue of a - 2 (which implies that the products of a - 2, the last
      // readers of that buffer's P, are done); the products need P of a.
      const uint32_t tm = x.tmem;
      const uint32_t aOnes = smem_u32(smem + OFF_ONES);
      const uint64_t e0 = sdesc_sw128(smem_u32(smem + OFF_E), 16, 1024);
      uint32_t as = 0, ap = 0, idle = 0;
      const uint32_t n = (uint32_t)total;
      bool ok = (!p.force_wait || waitb(x, &B->never, 0)) && (nE == 0 || waitb(x, &B->eready, 0));
      if (BWD && ok && nE > 0) {  // the entry-state tile, for the gradient's last launch
        tma_store_3d(&tm_e, smem + OFF_E, 0, 0, (int)blockIdx.x);
        bulk_commit();
      }
      uint64_t dl = globaltimer_ns() + mbar_ns;
      while (ok && ap < n) {
        if (*x.abort) break;
        bool did = false;
        if (ap < as && mbar_test_wait(&B->pready[ap % 2], (ap / 2) & 1)) {
          tc_fence_after();
          const uint32_t a = ap;
          if (a < 16) LA_TRACE(3, 16 + a);
          const uint32_t vt = smem_u32(smem + (a % NS) * STAGE + OFF_V);
          const uint32_t dO = tm + TB * (a % 2) + TOO, aP = tm + TB * (a % 2);
          const uint64_t v0 = sdesc_sw128(vt, aOnes - vt, 1024);
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks)  // P [V | 1], P from TMEM (keys 0..63, then 64..127)
            mma_bf16_ts(dO, aP + (ks < 4 ? 8 * ks : 64 + 8 * (ks - 4)), v0 + ks * kStepMN, ID_PV, 1u);
          if (a < 16) LA_TRACE(3, 48 + a);
          mma_commit(&B->oready[a % 2]);
          mma_commit(&B->empty[a % NS]);
          if (a < 6) LA_TRACE(2, 28 + a);
          ++ap;
          did = true;
        } else if (as < n && as < ap + 2 && mbar_test_wait(&B->xf[as % NS], (as / NS) & 1) &&
                   mbar_test_wait(&B->full[as % NS], (as / NS) & 1) &&
                   (as < 2 || mbar_test_wait(&B->ofree[as % 2], ((as / 2) - 1) & 1))) {
          tc_fence_after();
          const uint32_t a = as;
          if (a < 16) LA_TRACE(3, a);
          const uint32_t st = smem_u32(smem + (a % NS) * STAGE);
          const uint32_t dA = tm + TB * (a % 2), aQ = tm + TQ + 32 * (a % 3);
          const uint64_t b0 = sdesc_sw128(st + OFF_K, 16, 1024);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)  // phi(Q) from TMEM, [phi(K) ; P] from shared memory
            mma_bf16_ts(dA, aQ + 8 * ks, b0 + ks * kStepK16, ID_SX, ks > 0 ? 1u : 0u);
          if ((int)a < nE) {
            if (DECAY) {  // Gamma_c phi(Q), written over Q by the phi warps
              const uint64_t q0 = sdesc_sw128(st, 16, 1024);
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16_ss(dA + TOO, q0 + ks * kStepK16, e0 + ks * kStepK16, ID_X, 1u);
            } else {
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16_ts(dA + TOO, aQ + 8 * ks, e0 + ks * kStepK16, ID_X, 1u);
            }
          }
          if (a < 16) LA_TRACE(3, 32 + a);
          mma_commit(&B->accB[a % 2]);
          if (a < 6) LA_TRACE(2, 16 + a);
          ++as;
          did = true;
        }
        if (did) {  // the clock is read once per job and every 64 idle polls
          idle = 0;
          dl = globaltimer_ns() + mbar_ns;
        } else if ((++idle & 63) == 0 && globaltimer_ns() > dl) {
          *x.abort = 1;
          atomicOr(x.status, kStatusTimeout);
        }
      }
      if (*x.abort) {
        int never = 0;
        mma_commit(&B->drain);
        mbar_wait(&B->drain, 0, globaltimer_ns() + mbar_ns, &never);
      }
      if (BWD) bulk_wait_all();
    }
    __syncwarp();
  } else if (warp < 10) {
    // ---- two jobs per chunk, in whichever order they become ready (a mask
    // before a phi when both are), each mask after its chunk's phi:
    //   phi(j): phi(Q) into TMEM (buffer j % 3), the A operand of the chunk's
    //     first products: the two warps of a lane quadrant take half a row
    //     each (after mask(j - 3): the first products of j - 3, the last to
    //     read the buffer, are complete once their scores are);
    //   mask(j): the causal mask P of the scores, bf16, in place in TMEM.  The
    //     mask of a TMEM lane quadrant is split over its two warps (warp w
    //     reaches lanes 32 (w % 4)..+31): the warp of the first half builds key
    //     blocks 0 and 1 and packs them into columns 0..31, the other blocks 2
    //     and 3 into columns 64..95, each over scores it has read itself, so
    //     the two warps never wait for each other (the products read keys
    //     0..63 from columns 0..31 and keys 64..127 from columns 64..95).
    const int cw = warp - 2, quad = warp % 4, half = cw / 4;
    const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
    auto prep_step = [&](uint32_t j) {
      const int s = j % NS;
      if (!waitb_warp(x, &B->qfull[s], (j / NS) & 1)) return;
      const long long gc = run.a + j;
      const int valid = p.sp.N - (int)(gc % p.sp.NC) * C;
      if (cw == 0 && lane == 0 && j < 6) LA_TRACE(2, 4 + j);
      const int row = 32 * quad + lane;  // this lane's TMEM lane; elements 32 half .. 32 half + 31
      const uint8_t* qt = smem + s * STAGE;
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint4*>(qt + sw128_offset(row, 4 * half + i));
      const uint32_t keep = row < valid ? 0xFFFFFFFFu : 0u;
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        w[4 * i + 0] = phi2(v[i].x) & keep;
        w[4 * i + 1] = phi2(v[i].y) & keep;
        w[4 * i + 2] = phi2(v[i].z) & keep;
        w[4 * i + 3] = phi2(v[i].w) & keep;
      }
      tmem_st16(tl + TQ + 32 * (j % 3) + 16 * half, w);
      if (DECAY && (int)j < nE) {
        // a chunk with an entry state: Gamma_c phi(Q) over Q's half row (the
        // A operand of the E product), Gamma_c from the prefix kernel
        pdl_wait();
        const float gm = __ldcg(p.gamc + gc);
        uint8_t* qw = smem + s * STAGE;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 u;
          uint32_t* e = &u.x;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            e[k] = pack_bf16x2(__uint_as_float(w[4 * i + k] << 16) * gm,
                               __uint_as_float(w[4 * i + k] & 0xFFFF0000u) * gm);
          *reinterpret_cast<uint4*>(qw + sw128_offset(row, 4 * half + i)) = u;
        }
        fence_proxy_async_smem();
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (cw == 0 && lane == 0 && j < 6) LA_TRACE(2, 10 + j);
      if (lane == 0) mbar_arrive(&B->xf[s]);
    };
    auto mask_step = [&](uint32_t j) {
      const int b = j % 2;
      const bool got = waitb_warp(x, &B->accB[b], (j / 2) & 1);
      if (warp == 7 && lane == 0 && j < 6) LA_TRACE(2, 46 + j);
      const uint32_t base = tl + TB * b;
      const int q0 = 2 * half;  // this warp's key blocks: q0, q0 + 1
      uint32_t r0[32], r1[32];
      if (!got) return;
      tc_fence_after();
      // decayed form: the stage's g (loaded with its tiles; the phase of the
      // stage's `full` for chunk j is still current)
      const float* gs = reinterpret_cast<const float*>(smem + (j % NS) * STAGE + OFF_G);
      float gt = 0.f;
      if (DECAY) {
        waitb_warp(x, &B->full[j % NS], (j / NS) & 1);
        gt = gs[32 * quad + lane];
      }
      if (q0 <= quad) tmem_ld32(base + 32 * q0, r0);
      if (q0 + 1 <= quad) tmem_ld32(base + 32 * (q0 + 1), r1);
      tmem_ld_wait();
#pragma unroll 1
      for (int k = 0; k < 2; ++k) {
        const int q4 = q0 + k;
        uint32_t w[16];
        if (q4 > quad) {
#pragma unroll
          for (int t2 = 0; t2 < 16; ++t2) w[t2] = 0u;
        } else {
          const uint32_t* r = k ? r1 : r0;
          if (DECAY && q4 < quad) {  // 2^(g_t - g_s) <= 1
            const float* gk = gs + 32 * q4;
#pragma unroll
            for (int t2 = 0; t2 < 16; ++t2)
              w[t2] = pack_bf16x2(__uint_as_float(r[2 * t2]) * exp2_ftz(gt - gk[2 * t2]),
                                  __uint_as_float(r[2 * t2 + 1]) * exp2_ftz(gt - gk[2 * t2 + 1]));
          } else if (DECAY) {  // the diagonal block: 2^(g_t - g_s) for s <= t
            const float* gk = gs + 32 * q4;
#pragma unroll
            for (int t2 = 0; t2 < 16; ++t2)
              w[t2] = pack_bf16x2(2 * t2 <= lane ? __uint_as_float(r[2 * t2]) * exp2_ftz(gt - gk[2 * t2]) : 0.f,
                                  2 * t2 + 1 <= lane ? __uint_as_float(r[2 * t2 + 1]) * exp2_ftz(gt - gk[2 * t2 + 1])
                                                     : 0.f);
          } else if (q4 < quad) {
#pragma unroll
            for (int t2 = 0; t2 < 16; ++t2)
              w[t2] = pack_bf16x2(__uint_as_float(r[2 * t2]), __uint_as_float(r[2 * t2 + 1]));
          } else {
#pragma unroll
            for (int t2 = 0; t2 < 16; ++t2)
              w[t2] = pack_bf16x2((STRICT ? 2 * t2 < lane : 2 * t2 <= lane) ? __uint_as_float(r[2 * t2]) : 0.f,
                                  (STRICT ? 2 * t2 + 1 < lane : 2 * t2 + 1 <= lane)
                                      ? __uint_as_float(r[2 * t2 + 1]) : 0.f);
          }
        }
        tmem_st16(base + 64 * half + 16 * k, w);  // over this warp's own block q0's scores
      }
      if (DECAY) {  // the state part of the row, phi(Q) (P_c + Gamma_c E), times 2^g_t
        const float ga = exp2_ftz(gt);
        const uint32_t ob = base + TOO + 32 * half;  // columns 32 half .. +31, and 64..79 for half 0
        uint32_t o32[32];
        tmem_ld32(ob, o32);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t wq[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) wq[i] = __float_as_uint(__uint_as_float(o32[16 * q + i]) * ga);
          tmem_st16(ob + 16 * q, wq);
        }
        if (half == 0) {
          uint32_t o16[16];
          tmem_ld16(base + TOO + D, o16);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) o16[i] = __float_as_uint(__uint_as_float(o16[i]) * ga);
          tmem_st16(base + TOO + D, o16);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (warp == 7 && lane == 0 && j < 6) LA_TRACE(2, 22 + j);
      if (lane == 0) mbar_arrive(&B->pready[b]);
    };
    const uint32_t n = (uint32_t)total;
    uint32_t jp = 0, jm = 0, idle = 0;
    // phi(Q) of the first chunks (one per phi(Q) buffer) needs only Q: before
    // the earlier launch has finished
    for (; jp < n && jp < 3; ++jp) prep_step(jp);
    entry_part();
    uint64_t dl = globaltimer_ns() + x.mbar_ns;
    while (jp < n || jm < n) {
      if (*x.abort) break;  // given up
      bool did = false;
      if (jm < jp && __shfl_sync(0xFFFFFFFFu, (int)mbar_test_wait(&B->accB[jm % 2], (jm / 2) & 1), 0)) {
        mask_step(jm++);
        did = true;
      } else if (jp < n && jm + 2 >= jp &&  // mask(jp - 3) done: phi(Q) buffer jp % 3 is free
                 __shfl_sync(0xFFFFFFFFu, (int)mbar_test_wait(&B->qfull[jp % NS], (jp / NS) & 1), 0)) {
        prep_step(jp++);
        did = true;
      }
      if (did) {  // the clock is read once per job and every 64 idle polls
        idle = 0;
        dl = globaltimer_ns() + x.mbar_ns;
      } else if ((++idle & 63) == 0 && globaltimer_ns() > dl) {
        if (lane == 0 && !*x.abort) {
          *x.abort = 1;
          atomicOr(x.status, kStatusTimeout);
        }
        __syncwarp();
      }
    }
  } else {
    entry_part();
    // ---- the output epilogue (warps 10..13), o = num / (den + eps) (den =
    // the hi and lo columns of z plus the ones column), staged in shared
    // memory and stored by TMA (thread 352)
    if (warp < 14) {
      const int quad = warp % 4, row = 32 * quad + lane, et = threadIdx.x - 320;
      const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
      uint8_t* out = smem + OFF_OUT;
      uint32_t oj = 0;
      Piece pc;
      for (int i = 0; run.piece(p.sp, i, &pc); ++i)
        for (int c = 0; c < pc.nch; ++c, ++oj) {
          const int ob = oj % 2;
          waitb(x, &B->oready[ob], (oj / 2) & 1);  // on a timeout the rest runs on, storing nothing
          if (et == 32 && oj < 6) LA_TRACE(2, 34 + oj);
          tc_fence_after();
          const uint32_t base = tl + TB * ob + TOO;
          uint32_t n0[32], n1[32], d2[2];
          tmem_ld32(base, n0);
          tmem_ld32(base + 32, n1);
          tmem_ld2(base + D, d2);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&B->ofree[ob]);
          const float den = __uint_as_float(d2[0]) + __uint_as_float(d2[1]) + p.eps;
          const float inv = 1.f / den;
          if (BWD && row < pc.tok1 - (pc.tok0 + c * C) && !*x.abort)
            p.den[(size_t)pc.h * p.sp.N + pc.tok0 + c * C + row] = den;
          if (et == 32) bulk_wait_read_all();  // the previous chunk's store has read the staging
          named_bar_sync(5, 128);
          if (BWD) {  // o as bf16, one [128 x 64] tile
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              *reinterpret_cast<uint4*>(out + sw128_offset(row, cc)) =
                  make_uint4(pack_bf16x2(__uint_as_float(n0[8 * cc]) * inv, __uint_as_float(n0[8 * cc + 1]) * inv),
                             pack_bf16x2(__uint_as_float(n0[8 * cc + 2]) * inv, __uint_as_float(n0[8 * cc + 3]) * inv),
                             pack_bf16x2(__uint_as_float(n0[8 * cc + 4]) * inv, __uint_as_float(n0[8 * cc + 5]) * inv),
                             pack_bf16x2(__uint_as_float(n0[8 * cc + 6]) * inv, __uint_as_float(n0[8 * cc + 7]) * inv));
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              *reinterpret_cast<uint4*>(out + sw128_offset(row, 4 + cc)) =
                  make_uint4(pack_bf16x2(__uint_as_float(n1[8 * cc]) * inv, __uint_as_float(n1[8 * cc + 1]) * inv),
                             pack_bf16x2(__uint_as_float(n1[8 * cc + 2]) * inv, __uint_as_float(n1[8 * cc + 3]) * inv),
                             pack_bf16x2(__uint_as_float(n1[8 * cc + 4]) * inv, __uint_as_float(n1[8 * cc + 5]) * inv),
                             pack_bf16x2(__uint_as_float(n1[8 * cc + 6]) * inv, __uint_as_float(n1[8 * cc + 7]) * inv));
          } else {
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
          }
          fence_proxy_async_smem();
          named_bar_sync(5, 128);
          if (et == 32 && !*x.abort) {
            const int tok = pc.tok0 + c * C;
            if (BWD) {  // read again soon (the gradient's next launch)
              tma_store_3d(&tm_o, out, 0, tok, pc.h);
            } else {
              tma_store_3d_ef(&tm_o, out, 0, tok, pc.h);
              tma_store_3d_ef(&tm_o, out + BLK, 32, tok, pc.h);
            }
            bulk_commit();
            if (oj < 6) LA_TRACE(2, 40 + oj);
          }
        }
      if (et == 32) bulk_wait_all();
    }
  }
  free_tmem(x, warp, kCols);
  if (threadIdx.x == 0) LA_TRACE(2, 59);
}

}  // namespace out

}  // namespace

// Calls of at most this many chunks take this form: phi(K), the prefix tiles
// and V, read again by the output kernel, stay within L2 (40 KB per chunk).
constexpr long long kPrefixMaxChunks = 2048;

bool prefill_prefix64_chosen(int B, int H, int N) {
  const long long tc = (long long)B * H * ((N + C - 1) / C);
  return tc > 0 && tc <= kPrefixMaxChunks;
}

// piece totals, prefix tiles, then phi(K)
size_t prefill_prefix64_workspace_bytes(int B, int H, int N) {
  const Split s = make_split(B * H, N, sm_count());
  return (size_t)s.BH * s.MPH * SZ * sizeof(float) + (size_t)s.TC() * XG +
         (size_t)B * H * N * D * sizeof(__nv_bfloat16);
}

cudaError_t launch_prefix64_pair(const PrefillArgs& a, const Prefix64Buffers& b, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  Params p = {};
  p.sp = make_split(BH, a.N, sms);
  p.eps = a.eps;
  p.S0 = a.S0;
  p.z0 = a.z0;
  p.S_N = b.S_N;
  p.z_N = b.z_N;
  p.status = b.status;
  p.R = b.R;
  p.P = b.P;
  p.den = b.den;
  p.force_wait = b.force_wait;
  CUtensorMap mq, mk, mv, mo, mphik, mp, me;
  const bool bwd = b.den != nullptr;
  if ((bwd && !b.E) || (bwd && b.strict)) return cudaErrorInvalidValue;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !(bwd ? make_map(&mo, b.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C)
            : make_map(&mo, b.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C)) ||
      !make_map(&mphik, b.phik, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mp, p.P, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, XROWS, (int)p.sp.TC(), 64, XROWS) ||
      !make_map(&me, bwd ? b.E : p.P, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, XROWS,
                bwd ? p.sp.G : (int)p.sp.TC(), 64, XROWS))
    return cudaErrorInvalidValue;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);

  cudaError_t e = cudaFuncSetAttribute(pfx::prefix_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pfx::SMEM_PLAIN);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd ? out::output_kernel<true, false, false>
                             : b.strict ? out::output_kernel<false, true, false> : out::output_kernel<false, false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)out::SMEM_PLAIN);
  if (e != cudaSuccess) return e;
  // Both launches are programmatic dependents of what precedes them on the
  // stream: their blocks may start while the kernel before runs, and wait for
  // it (griddepcontrol.wait) before touching what it may write.
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(32 * pfx::kWarps);
  cfg.dynamicSmemBytes = pfx::SMEM_PLAIN;
  e = cudaLaunchKernelEx(&cfg, pfx::prefix_kernel<false>, mk, mv, mphik, mp, p, mbar_ns);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(32 * out::kWarps);
  cfg.dynamicSmemBytes = out::SMEM_PLAIN;
  if (bwd)
    return cudaLaunchKernelEx(&cfg, out::output_kernel<true, false, false>, mq, mphik, mp, mv, mo, me, p, mbar_ns);
  if (b.strict)
    return cudaLaunchKernelEx(&cfg, out::output_kernel<false, true, false>, mq, mphik, mp, mv, mo, me, p, mbar_ns);
  return cudaLaunchKernelEx(&cfg, out::output_kernel<false, false, false>, mq, mphik, mp, mv, mo, me, p, mbar_ns);
}

cudaError_t launch_prefix64_totals(const PrefillArgs& a, const Prefix64Buffers& b, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  Params p = {};
  p.sp = make_split(BH, a.N, sms);
  p.eps = a.eps;
  p.S0 = a.S0;
  p.z0 = a.z0;
  p.status = b.status;
  p.R = b.R;
  p.P = b.P;
  p.totals_only = 1;
  CUtensorMap mk, mv, mphik, mp;
  if (!make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mphik, b.phik, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mp, p.P, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, XROWS, (int)p.sp.TC(), 64, XROWS))
    return cudaErrorInvalidValue;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  cudaError_t e = cudaFuncSetAttribute(pfx::prefix_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pfx::SMEM_PLAIN);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(32 * pfx::kWarps);
  cfg.dynamicSmemBytes = pfx::SMEM_PLAIN;
  return cudaLaunchKernelEx(&cfg, pfx::prefix_kernel<false>, mk, mv, mphik, mp, p, mbar_ns);
}

cudaError_t launch_prefill_prefix64(const PrefillArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const Split sp = make_split(BH, a.N, sms);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  if (sizeof(WsHeader) + prefill_prefix64_workspace_bytes(a.B, a.H, a.N) > a.ws_bytes)
    return cudaErrorInvalidValue;
  Prefix64Buffers b = {};
  b.R = reinterpret_cast<float*>(ws + sizeof(WsHeader));
  b.P = reinterpret_cast<uint8_t*>(b.R + (size_t)BH * sp.MPH * SZ);
  b.phik = reinterpret_cast<__nv_bfloat16*>(b.P + (size_t)sp.TC() * XG);
  b.o = a.o;
  b.den = nullptr;
  b.E = nullptr;
  b.S_N = a.S_N;
  b.z_N = a.z_N;
  b.status = a.status ? a.status : &reinterpret_cast<WsHeader*>(ws)->status;
  b.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);
  return launch_prefix64_pair(a, b, stream);
}

cudaError_t launch_prefill_rbw64(const PrefillArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const Split sp = make_split(BH, a.N, sms);
  if (!a.workspace || prefill_prefix64_workspace_bytes(a.B, a.H, a.N) > a.ws_bytes)
    return cudaErrorInvalidValue;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  Prefix64Buffers b = {};
  b.R = reinterpret_cast<float*>(ws);
  b.P = reinterpret_cast<uint8_t*>(b.R + (size_t)BH * sp.MPH * SZ);
  b.phik = reinterpret_cast<__nv_bfloat16*>(b.P + (size_t)sp.TC() * XG);
  b.o = a.o;
  b.S_N = a.S_N;
  b.z_N = a.z_N;
  cudaError_t e = library_status_word(&b.status);
  if (e != cudaSuccess) return e;
  b.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);
  b.strict = 1;
  return launch_prefix64_pair(a, b, stream);
}


// Decayed form's workspace (no header): piece totals, prefix tiles, phi(K),
// then per chunk row g (fp32), per chunk the decay from its piece's start,
// per piece slot its decay.
struct DecayLayout {
  size_t R, P, phik, G, gamc, gam, total;
};
static DecayLayout decay_layout(int B, int H, int N) {
  const Split s = make_split(B * H, N, sm_count());
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  DecayLayout L;
  L.R = 0;
  L.P = up(L.R + (size_t)s.BH * s.MPH * SZ * sizeof(float));
  L.phik = up(L.P + (size_t)s.TC() * XG);
  L.G = up(L.phik + (size_t)s.BH * N * D * 2);
  L.gamc = up(L.G + (size_t)s.TC() * C * sizeof(float));
  L.gam = up(L.gamc + (size_t)s.TC() * sizeof(float));
  L.total = up(L.gam + (size_t)s.BH * s.MPH * sizeof(float));
  return L;
}

size_t prefill_prefix64_decay_workspace_bytes(int B, int H, int N) { return decay_layout(B, H, N).total; }

cudaError_t launch_prefill_prefix64_decay(const PrefillArgs& a, const float* alpha, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const DecayLayout L = decay_layout(a.B, a.H, a.N);
  if (!a.workspace || a.ws_bytes < L.total || !alpha) return cudaErrorInvalidValue;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  Params p = {};
  p.sp = make_split(BH, a.N, sms);
  p.eps = a.eps;
  p.S0 = a.S0;
  p.z0 = a.z0;
  p.S_N = a.S_N;
  p.z_N = a.z_N;
  cudaError_t e = library_status_word(&p.status);
  if (e != cudaSuccess) return e;
  p.R = reinterpret_cast<float*>(ws + L.R);
  p.P = ws + L.P;
  __nv_bfloat16* phik = reinterpret_cast<__nv_bfloat16*>(ws + L.phik);
  p.alpha = alpha;
  p.G = reinterpret_cast<float*>(ws + L.G);
  p.gamc = reinterpret_cast<float*>(ws + L.gamc);
  p.gam = reinterpret_cast<float*>(ws + L.gam);
  p.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);
  CUtensorMap mq, mk, mv, mo, mphik, mp;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mo, a.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C) ||
      !make_map(&mphik, phik, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mp, p.P, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, XROWS, (int)p.sp.TC(), 64, XROWS))
    return cudaErrorInvalidValue;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  e = cudaFuncSetAttribute(pfx::prefix_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)pfx::SMEM_DECAY);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(out::output_kernel<false, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)out::SMEM_DECAY);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(32 * pfx::kWarps);
  cfg.dynamicSmemBytes = pfx::SMEM_DECAY;
  e = cudaLaunchKernelEx(&cfg, pfx::prefix_kernel<true>, mk, mv, mphik, mp, p, mbar_ns);
  if (e != cudaSuccess) return e;
  cfg.blockDim = dim3(32 * out::kWarps);
  cfg.dynamicSmemBytes = out::SMEM_DECAY;
  return cudaLaunchKernelEx(&cfg, out::output_kernel<false, false, true>, mq, mphik, mp, mv, mo, mp, p, mbar_ns);
}

}  // namespace la
