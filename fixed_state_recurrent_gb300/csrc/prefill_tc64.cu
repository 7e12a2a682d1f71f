// prefill_tc64.cu -- pipelined chunked causal prefill for dk = dv = 64 on the
// sm_103a tensor cores.
//
// Operator (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03):
//   o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps),  S_t = S_{t-1} + phi(k_t) v_t^T,
//   z_t = z_{t-1} + phi(k_t),  phi = ELU + 1,  write before read.
// Chunkwise evaluation (page "线性注意力与SSM", section 3): inside a chunk of
// C = 128 tokens a masked phi(Q) phi(K)^T attention, across chunks the state.
//
// Work items are 512-token windows of one head (window-major, one persistent
// block per SM, cooperative launch), each processed in two phases:
//   A. for every chunk c of the item the tensor cores accumulate the
//      transposed state in one M = 128 product per 16 tokens,
//      R += [V_c | 1]^T phi(K_c), into a TMEM accumulator: lanes 0..63 hold
//      R^T (lane j = column j of R = sum phi(K)^T V), lane 64 holds the z part
//      (sum phi(K)^T 1).  After chunk c the epilogue warps snapshot the running
//      R_{c+1} to bf16 (R_0 = 0): the state each chunk of the item starts from,
//      relative to the item start.  The final R is the item's aggregate,
//      published for the look-back (workspace states are stored transposed,
//      one contiguous row per thread).
//   L. decoupled look-back (bounded waits) for the item's exclusive prefix E
//      (S0 and all earlier items of the head, always the same left fold so that
//      results are bit-identical from run to run); E is snapshotted to bf16.
//   B. for every chunk: scores A = phi(Q_c) phi(K_c)^T (tensor cores); the P
//      warps mask them causally (key <= query, diagonal kept), round to bf16
//      and write P back into the same TMEM columns; then
//        [num | den] = P [V_c | 1] + phi(Q_c) [E | z_E] + phi(Q_c) [R_c | z_R_c]
//      as three N = 80 tensor-core products (P read from TMEM; the state
//      snapshots are K-major B operands whose rows 0..63 are S^T and rows
//      64, 65 the bf16 hi / lo split of z), and o = num / (den + eps) is stored
//      through TMA.  Every denominator term rides in the numerator's products.
// Phase B has no serial dependence between chunks, and the look-back of an
// item overlaps with the scores and P of its first chunks.
//
// Warp roles (576 threads):
//   warp 0      TMA producer (3-stage ring of Q | K | V tiles, 48 KB each)
//   warp 1      TMEM owner; lane 0 issues every tcgen05.mma
//   warps 2-9   apply phi in shared memory (K in phase A, Q and K in phase B);
//               two threads per tile row, all loads issued before any math
//   warps 10-13 build P from the scores (one warp per TMEM lane quadrant)
//   warps 14-17 state epilogue (phase A), look-back, output epilogue (phase B)
// TMEM (512 columns): A[b] = cols 128b..128b+127 (scores, then P packed in
// place), b = 0, 1; O[ob] = cols 256 + 80 ob: 64 numerator columns, then the
// denominator in columns 64 (+ 65); R = cols 416..479 (phase-A running state).
#include "prefill_tc_common.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcp;

constexpr int D = 64;
constexpr int NS = 3;                       // stages in the TMA ring
constexpr int kWarps = 18;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxChunks = kItemTokens / C;  // 4
constexpr uint32_t BLK = 16384;             // [128 rows x 128 B] swizzled tile
constexpr uint32_t STAGE = 3 * BLK;         // Q | K | V
constexpr uint32_t SNAP = 80 * 128;        // K-major [80 rows x 64 dk] bf16: S^T, z hi, z lo, 0
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_ONES = NS * STAGE;                        // [128 x 64] MN-major, column 0 = 1
constexpr uint32_t OFF_ESNAP = OFF_ONES + BLK;                   // snapshot of E
constexpr uint32_t OFF_RSNAP = OFF_ESNAP + SNAP;                 // snapshots of R_c, c = 1..3
constexpr uint32_t OFF_BAR = OFF_RSNAP + (kMaxChunks - 1) * SNAP;
constexpr uint32_t SMEM = OFF_BAR + 512 + 1024;                  // + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TA = 0;
constexpr uint32_t TO = 256;
constexpr uint32_t TR = 416;
constexpr int SZ = D * D + D;

constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);   // phi(Q) phi(K)^T
constexpr uint32_t ID_PV = idesc_bf16_f32(128, D + 16, 0, 1); // P [V | 1]
constexpr uint32_t ID_QS = idesc_bf16_f32(128, D + 16, 0, 0); // phi(Q) [S | z]
constexpr uint32_t ID_DS = idesc_bf16_f32(128, D, 1, 1);    // [V | 1]^T phi(K)

struct Bars {
  uint64_t full[NS];    // TMA bytes landed              (producer -> phi warps)
  uint64_t xf[NS];      // phi applied (8 warps)         (phi warps -> MMA)
  uint64_t empty[NS];   // stage free                    (MMA / epilogue -> producer)
  uint64_t accA;        // R updated by a chunk          (MMA -> state epilogue)
  uint64_t rfree;       // R read: the MMA may update it (state epilogue -> MMA)
  uint64_t accB[2];     // scores ready in A[b]          (MMA -> P warps)
  uint64_t pready[2];   // P written into A[b]           (P warps -> MMA)
  uint64_t freeb[2];    // A[b] may be overwritten       (MMA -> MMA)
  uint64_t oready[2];   // num, den ready in O[ob]       (MMA -> epilogue)
  uint64_t ofree[2];    // O[ob] read                    (epilogue -> MMA)
  uint64_t eready;      // E and R_c snapshots written   (epilogue -> MMA)
  uint64_t snapfree;    // the item's last MMA reading snapshots is done (MMA -> epilogue)
  uint64_t drain;       // all MMAs done (abort path)
  uint32_t tmem_slot;
  int abort;
  int lb_start;
};

struct Ctx {
  const TcParams* p;
  uint8_t* smem;
  Bars* bars;
  uint32_t tmem;
  unsigned epoch;
  unsigned long long mbar_ns;
};

__device__ __forceinline__ void wait_bar(const Ctx& x, uint64_t* bar, uint32_t parity) {
  volatile int* ab = &x.bars->abort;
  if (*ab) return;
  if (!mbar_wait(bar, parity, globaltimer_ns() + x.mbar_ns, ab)) {
    *ab = 1;
    atomicOr(&x.p->hdr->status, kStatusTimeout);
  }
}

__device__ __forceinline__ uint8_t* stage_ptr(const Ctx& x, int s) {
  return x.smem + OFF_STAGE + s * STAGE;
}

// ---------------------------------------------------------------------------
// warp 0: TMA producer

__device__ void producer(const Ctx& x, const CUtensorMap* tq, const CUtensorMap* tk,
                         const CUtensorMap* tv) {
  const TcParams& p = *x.p;
  uint32_t sj = 0;
  for (int g = blockIdx.x; g < p.total_items; g += gridDim.x) {
    const Item it = item_of(p, g);
    for (int phase = 0; phase < 2; ++phase) {
      for (int c = 0; c < it.nch; ++c, ++sj) {
        const int s = sj % NS;
        if (sj >= NS) wait_bar(x, &x.bars->empty[s], ((sj / NS) - 1) & 1);
        uint8_t* st = stage_ptr(x, s);
        const int tok = it.tok0 + c * C;
        mbar_arrive_expect_tx(&x.bars->full[s], (phase == 0 ? 2 : 3) * BLK);
        if (phase == 1) tma_load_3d(st, tq, 0, tok, it.h, &x.bars->full[s]);
        tma_load_3d(st + BLK, tk, 0, tok, it.h, &x.bars->full[s]);
        tma_load_3d(st + 2 * BLK, tv, 0, tok, it.h, &x.bars->full[s]);
      }
    }
  }
  if (x.bars->abort) {  // let the last loads of every stage land before exiting
    int never = 0;
    const uint64_t dl = globaltimer_ns() + x.mbar_ns;
    for (uint32_t j = (sj > NS ? sj - NS : 0); j < sj; ++j)
      mbar_wait(&x.bars->full[j % NS], (j / NS) & 1, dl, &never);
  }
}

// ---------------------------------------------------------------------------
// warps 2-5: phi in place on the swizzled tiles

// phi on two bf16: exp(min(u,0)) + max(u,0) with the min, max and the final
// add done on the pair (bf16 arithmetic rounds once, so the result equals
// rounding u + 1, resp. exp(u), to bf16) and the exponentials in fp32.
__device__ __forceinline__ uint32_t phi_bf16x2_packed(uint32_t x) {
  const __nv_bfloat162 u = *reinterpret_cast<const __nv_bfloat162*>(&x);
  const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
  const __nv_bfloat162 m = __hmin2(u, zero);
  const __nv_bfloat162 M = __hmax2(u, zero);
  const uint32_t mb = *reinterpret_cast<const uint32_t*>(&m);
  const uint32_t e = pack_bf16x2(__expf(__uint_as_float(mb << 16)),
                                 __expf(__uint_as_float(mb & 0xFFFF0000u)));
  const __nv_bfloat162 r = __hadd2(*reinterpret_cast<const __nv_bfloat162*>(&e), M);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// phi on chunks [4 part, 4 part + 4) of row r of one tile, or of both the Q
// and K tiles; all shared-memory loads are issued before any arithmetic.
template <int NT>
__device__ __forceinline__ void phi_rows(uint8_t* const (&tiles)[NT], int r, int part,
                                         int valid) {
  uint4 v[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      v[t][i] = *reinterpret_cast<const uint4*>(tiles[t] + sw128_offset(r, 4 * part + i));
  const bool keep = r < valid;
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 u = v[t][i];
      u.x = keep ? phi_bf16x2_packed(u.x) : 0u;
      u.y = keep ? phi_bf16x2_packed(u.y) : 0u;
      u.z = keep ? phi_bf16x2_packed(u.z) : 0u;
      u.w = keep ? phi_bf16x2_packed(u.w) : 0u;
      v[t][i] = u;
    }
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<uint4*>(tiles[t] + sw128_offset(r, 4 * part + i)) = v[t][i];
}

__device__ void transformer(const Ctx& x, int et, int lane) {
  const int r = et % C, part = et / C;  // 256 threads: row r, half `part` of it
  const TcParams& p = *x.p;
  uint32_t sj = 0;
  for (int g = blockIdx.x; g < p.total_items; g += gridDim.x) {
    const Item it = item_of(p, g);
    for (int phase = 0; phase < 2; ++phase) {
      for (int c = 0; c < it.nch; ++c, ++sj) {
        const int s = sj % NS;
        wait_bar(x, &x.bars->full[s], (sj / NS) & 1);
        uint8_t* st = stage_ptr(x, s);
        const int valid = it.tok1 - (it.tok0 + c * C);
        if (phase == 1) {
          uint8_t* const t2[2] = {st, st + BLK};
          phi_rows<2>(t2, r, part, valid);
        } else {
          uint8_t* const t1[1] = {st + BLK};
          phi_rows<1>(t1, r, part, valid);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&x.bars->xf[s]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// warp 1 lane 0: MMA issue

__device__ void mma_issuer(const Ctx& x) {
  const TcParams& p = *x.p;
  Bars* B = x.bars;
  const uint32_t tm = x.tmem;
  const uint32_t aOnes = smem_u32(x.smem + OFF_ONES);
  const uint32_t aE = smem_u32(x.smem + OFF_ESNAP);
  const uint32_t aR = smem_u32(x.smem + OFF_RSNAP);
  uint32_t sj = 0, aj = 0, oj = 0, itn = 0;
  uint32_t npr[2] = {0, 0};  // uses of pready[b]
  uint32_t nrf = 0;          // R updates issued (each but the very first waits for rfree)

  // wait for the stage of job `j` to be transformed and for A[b] of job `a` to be free
  auto acquire = [&](uint32_t j, uint32_t a) {
    wait_bar(x, &B->xf[j % NS], (j / NS) & 1);
    if (a >= 2) wait_bar(x, &B->freeb[a % 2], ((a / 2) - 1) & 1);
    tc_fence_after();
  };
  auto scores = [&](uint32_t j, uint32_t a) {  // A[b] = phi(Q) phi(K)^T
    const uint32_t st = smem_u32(stage_ptr(x, j % NS));
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
      mma_bf16_ss(tm + TA + 128 * (a % 2), sdesc_sw128(st + ks * 32, 16, 1024),
                  sdesc_sw128(st + BLK + ks * 32, 16, 1024), ID_S, ks > 0 ? 1u : 0u);
    mma_commit(&B->accB[a % 2]);
  };

  for (int g = blockIdx.x; g < p.total_items; g += gridDim.x) {
    const Item it = item_of(p, g);
    // ---- phase A: R (+)= [V_c | 1]^T phi(K_c), chunk by chunk
    for (int c = 0; c < it.nch; ++c, ++sj) {
      wait_bar(x, &B->xf[sj % NS], (sj / NS) & 1);
      if (nrf > 0) wait_bar(x, &B->rfree, (nrf - 1) & 1);  // previous R read / item done
      ++nrf;
      tc_fence_after();
      const uint32_t st = smem_u32(stage_ptr(x, sj % NS));
      const uint32_t vt = st + 2 * BLK;
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) {
        // A = [V | 1]^T, MN-major: M rows 0..63 from the V tile, rows 64..127
        // from the ones tile (row 64 all ones); B = phi(K), MN-major (N = dk).
        const uint64_t a = sdesc_sw128(vt + ks * 2048, aOnes - vt, 1024);
        const uint64_t b = sdesc_sw128(st + BLK + ks * 2048, BLK, 1024);
        mma_bf16_ss(tm + TR, a, b, ID_DS, (c > 0 || ks > 0) ? 1u : 0u);
      }
      mma_commit(&B->accA);
      mma_commit(&B->empty[sj % NS]);
    }
    // ---- phase B
    const uint32_t sj0 = sj, aj0 = aj;
    acquire(sj0, aj0);
    scores(sj0, aj0);
    for (int c = 0; c < it.nch; ++c) {
      const uint32_t j = sj0 + c, a = aj0 + c;
      if (c + 1 < it.nch) {  // scores of the next chunk run while P of this one is built
        acquire(j + 1, a + 1);
        scores(j + 1, a + 1);
      }
      const int b = a % 2;
      wait_bar(x, &B->pready[b], npr[b] & 1);
      ++npr[b];
      if (c == 0) wait_bar(x, &B->eready, itn & 1);
      const int ob = oj % 2;
      if (oj >= 2) wait_bar(x, &B->ofree[ob], ((oj / 2) - 1) & 1);
      tc_fence_after();
      const uint32_t st = smem_u32(stage_ptr(x, j % NS));
      const uint32_t dO = tm + TO + 80 * ob;
      const uint32_t aP = tm + TA + 128 * b;
      const uint32_t vt = st + 2 * BLK;
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)  // P [V | 1], P from TMEM (8 columns per 16 keys)
        mma_bf16_ts(dO, aP + 8 * ks, sdesc_sw128(vt + ks * 2048, aOnes - vt, 1024), ID_PV,
                    ks > 0 ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {  // phi(Q) [E | z_E] + phi(Q) [R_c | z_R_c]
        const uint64_t aq = sdesc_sw128(st + ks * 32, 16, 1024);
        mma_bf16_ss(dO, aq, sdesc_sw128(aE + ks * 32, 16, 1024), ID_QS, 1u);
        if (c > 0)
          mma_bf16_ss(dO, aq, sdesc_sw128(aR + (c - 1) * SNAP + ks * 32, 16, 1024), ID_QS, 1u);
      }
      mma_commit(&B->oready[ob]);
      mma_commit(&B->freeb[b]);
      ++oj;
    }
    mma_commit(&B->snapfree);
    sj = sj0 + it.nch;
    aj = aj0 + it.nch;
    ++itn;
  }
  if (B->abort) {  // every issued MMA completes before TMEM is released
    int never = 0;
    mma_commit(&B->drain);
    mbar_wait(&B->drain, 0, globaltimer_ns() + x.mbar_ns, &never);
  }
}

// ---------------------------------------------------------------------------
// warps 6-9: P = causal mask of the scores, bf16, packed in place in TMEM

__device__ void p_builder(const Ctx& x, int quad, int lane) {
  const TcParams& p = *x.p;
  const int row = 32 * quad + lane;  // query row of the chunk
  const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
  uint32_t aj = 0;
  uint32_t nb[2] = {0, 0};  // uses of accB[b]
  for (int g = blockIdx.x; g < p.total_items; g += gridDim.x) {
    const Item it = item_of(p, g);
    for (int c = 0; c < it.nch; ++c, ++aj) {
      const int b = aj % 2;
      wait_bar(x, &x.bars->accB[b], nb[b] & 1);
      ++nb[b];
      tc_fence_after();
      const uint32_t base = tl + TA + 128 * b;
      // Keys in blocks of 32: this warp's rows are 32 quad .. 32 quad + 31, so
      // blocks before `quad` are fully visible, block `quad` holds the
      // diagonal, later blocks are fully masked (written as zeros, not read).
      // Packed keys 32 q4 .. +31 go to columns 16 q4 .. +15; in increasing q4
      // order those columns have always been read already.
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t w[16];
        if (q4 > quad) {
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = 0u;
        } else {
          uint32_t r[32];
          tmem_ld32(base + 32 * q4, r);
          tmem_ld_wait();
          if (q4 < quad) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j0 = 2 * i;  // key index within the block; the row's is `lane`
              w[i] = pack_bf16x2(j0 <= lane ? __uint_as_float(r[2 * i]) : 0.f,
                                 j0 + 1 <= lane ? __uint_as_float(r[2 * i + 1]) : 0.f);
            }
          }
        }
        tmem_st16(base + 16 * q4, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&x.bars->pready[b]);
    }
  }
}

// ---------------------------------------------------------------------------
// warps 10-13: state epilogue, look-back, output epilogue

// Row `n` of a K-major snapshot from 64 fp32 values (eight values per 16-byte chunk).
__device__ __forceinline__ void store_snap_row(uint8_t* snap, int n, const float* v /*64*/) {
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * cc + 0], v[8 * cc + 1]);
    u.y = pack_bf16x2(v[8 * cc + 2], v[8 * cc + 3]);
    u.z = pack_bf16x2(v[8 * cc + 4], v[8 * cc + 5]);
    u.w = pack_bf16x2(v[8 * cc + 6], v[8 * cc + 7]);
    *reinterpret_cast<uint4*>(snap + sw128_offset(n, cc)) = u;
  }
}

// Rows 64 (hi) and 65 (lo) of a snapshot from the 64 fp32 values of z:
// hi = bf16(z), lo = bf16(z - hi), so hi + lo carries about 16 bits of z.
__device__ __forceinline__ void store_snap_z(uint8_t* snap, const float* z /*64*/) {
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    float hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      hi[i] = __bfloat162float(__float2bfloat16_rn(z[8 * cc + i]));
      lo[i] = z[8 * cc + i] - hi[i];
    }
    uint4 h, l;
    h.x = pack_bf16x2(hi[0], hi[1]); h.y = pack_bf16x2(hi[2], hi[3]);
    h.z = pack_bf16x2(hi[4], hi[5]); h.w = pack_bf16x2(hi[6], hi[7]);
    l.x = pack_bf16x2(lo[0], lo[1]); l.y = pack_bf16x2(lo[2], lo[3]);
    l.z = pack_bf16x2(lo[4], lo[5]); l.w = pack_bf16x2(lo[6], lo[7]);
    *reinterpret_cast<uint4*>(snap + sw128_offset(64, cc)) = h;
    *reinterpret_cast<uint4*>(snap + sw128_offset(65, cc)) = l;
  }
}

// The state threads are TMEM lanes 0..64 of the running state R: lane j < 64
// holds row j of R^T (column j of S), lane 64 holds z.  Workspace states use
// that transposed layout -- thread `row` owns floats [64 row, 64 row + 64) of
// a slot, z last -- so every thread moves one contiguous 256-byte row.  S0 and
// S_N keep the API layout [dk][dv]: there lane j < 64 touches S[i][j], i.e.
// element i * 64 + j (coalesced across the warp), and lane 64 touches z[i].
__device__ __forceinline__ const float* api_elem(const float* S, const float* z, int row, int i) {
  return row < D ? S + i * D + row : z + i;
}
__device__ __forceinline__ float* api_elem(float* S, float* z, int row, int i) {
  return row < D ? S + i * D + row : z + i;
}

// 32 fp32 columns [32 half, 32 half + 32) of this lane's row of R from TMEM.
__device__ __forceinline__ void load_r_half(uint32_t tl, int half, float* out /*32*/) {
  uint32_t r[32];
  tmem_ld32(tl + TR + 32 * half, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = __uint_as_float(r[i]);
}

// 32 values of a row into chunks [4 half, 4 half + 4) of snapshot row n.
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

// A state lane's 32 values into a snapshot: S^T row `row`, or for the z lane
// rows 64 (hi = bf16(z)) and 65 (lo = bf16(z - hi)), about 16 bits of z.
__device__ __forceinline__ void snap_half(uint8_t* snap, int row, int half, const float* v) {
  if (row < D) {
    store_snap_half(snap, row, half, v);
  } else {
    float hi[32], lo[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      hi[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
      lo[i] = v[i] - hi[i];
    }
    store_snap_half(snap, 64, half, hi);
    store_snap_half(snap, 65, half, lo);
  }
}

__device__ void epilogue(const Ctx& x, int quad, int lane, int et, const CUtensorMap* to) {
  const TcParams& p = *x.p;
  Bars* B = x.bars;
  const int row = 32 * quad + lane;
  const bool state_warp = quad <= 2;        // TMEM lanes 0..95 (loads are warp-wide)
  const bool state_row = row <= D;          // lanes 0..64 carry R^T and z
  const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
  uint8_t* sE = x.smem + OFF_ESNAP;
  uint8_t* sR = x.smem + OFF_RSNAP;
  uint32_t oj = 0, sj = 0, itn = 0, nacc = 0;

  for (int g = blockIdx.x; g < p.total_items; g += gridDim.x) {
    const Item it = item_of(p, g);
    // the previous item's last MMA has read every snapshot we are about to overwrite
    if (itn > 0) wait_bar(x, &B->snapfree, (itn - 1) & 1);

    // ---- phase A: snapshots R_1..R_{n-1} of the running state
    for (int c = 0; c < it.nch; ++c, ++sj) {
      wait_bar(x, &B->accA, nacc & 1);
      ++nacc;
      if (c + 1 < it.nch) {
        tc_fence_after();
        if (state_warp) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[32];
            load_r_half(tl, half, v);
            if (state_row) snap_half(sR + c * SNAP, row, half, v);
          }
        }
        tc_fence_before();
        named_bar_sync(1, 128);
        if (et == 0) mbar_arrive(&B->rfree);
      }
    }
    tc_fence_after();

    // ---- publish the aggregate, look back, publish the inclusive prefix.
    // Publication: every thread stores, the named barrier orders the stores
    // before thread 0's release store of the flag (thread 0 issues no bulk
    // copies).  Window 0 has no earlier item: it publishes S0 + R directly.
    float* my_agg = p.agg + (size_t)g * SZ + row * D;
    float* my_inc = p.inc + (size_t)g * SZ + row * D;
    const bool last = it.w == p.items_per_head - 1;
    if (it.w > 0) {
      if (state_warp) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          load_r_half(tl, half, v);
          if (state_row) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              __stcg(reinterpret_cast<float4*>(my_agg + 32 * half) + i,
                     make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
          }
        }
      }
      named_bar_sync(1, 128);
      if (et == 0) st_release_gpu(&p.flags[g], (x.epoch << 2) | kFlagAggregate);
    }
    if (et == 0) B->lb_start = lookback_start(p, it, x.epoch);  // -1 for window 0
    named_bar_sync(1, 128);
    const int start = *reinterpret_cast<volatile int*>(&B->lb_start);
    if (state_warp) {
      // E = left fold S0 + agg_0 + ... + agg_{w-1}, starting from the nearest
      // published inclusive prefix; inclusive = E + R is published, E goes to
      // the bf16 snapshot.  Every load of a step is issued before its sums.
      const float* S0h = p.S0 ? p.S0 + (size_t)it.h * D * D : nullptr;
      const float* z0h = p.z0 ? p.z0 + (size_t)it.h * D : nullptr;
      const bool base_api = start < 0;
      const bool has_base = !base_api || (row < D ? S0h != nullptr : z0h != nullptr);
      const float* base_slot = p.inc + (size_t)(start < 0 ? 0 : start * p.BH + it.h) * SZ + row * D;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float e[32];
        if (!state_row || !has_base) {
#pragma unroll
          for (int i = 0; i < 32; ++i) e[i] = 0.f;
        } else if (base_api) {
#pragma unroll
          for (int i = 0; i < 32; ++i) e[i] = __ldcg(api_elem(S0h, z0h, row, 32 * half + i));
        } else {
          float4 u[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) u[i] = __ldcg(reinterpret_cast<const float4*>(base_slot + 32 * half) + i);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            e[4 * i] = u[i].x; e[4 * i + 1] = u[i].y; e[4 * i + 2] = u[i].z; e[4 * i + 3] = u[i].w;
          }
        }
        if (state_row) {
          for (int ww = start + 1; ww < it.w; ++ww) {
            const float* src = p.agg + (size_t)(ww * p.BH + it.h) * SZ + row * D + 32 * half;
            float4 u[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) u[i] = __ldcg(reinterpret_cast<const float4*>(src) + i);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              e[4 * i] += u[i].x; e[4 * i + 1] += u[i].y; e[4 * i + 2] += u[i].z; e[4 * i + 3] += u[i].w;
            }
          }
        }
        float r[32];
        load_r_half(tl, half, r);
        if (state_row) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 v = make_float4(e[4 * i] + r[4 * i], e[4 * i + 1] + r[4 * i + 1],
                                         e[4 * i + 2] + r[4 * i + 2], e[4 * i + 3] + r[4 * i + 3]);
            __stcg(reinterpret_cast<float4*>(my_inc + 32 * half) + i, v);
            if (last) {
              float* SN = p.S_N + (size_t)it.h * D * D;
              float* zN = p.z_N + (size_t)it.h * D;
              *api_elem(SN, zN, row, 32 * half + 4 * i) = v.x;
              *api_elem(SN, zN, row, 32 * half + 4 * i + 1) = v.y;
              *api_elem(SN, zN, row, 32 * half + 4 * i + 2) = v.z;
              *api_elem(SN, zN, row, 32 * half + 4 * i + 3) = v.w;
            }
          }
          snap_half(sE, row, half, e);
        }
      }
    }
    tc_fence_before();
    named_bar_sync(1, 128);
    if (et == 0) {
      st_release_gpu(&p.flags[g], (x.epoch << 2) | kFlagInclusive);
      mbar_arrive(&B->rfree);  // R may be overwritten by the next item
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&B->eready);

    // ---- phase B: o = num / (den + eps), stored through TMA from the stage's Q|K area
    for (int c = 0; c < it.nch; ++c, ++oj, ++sj) {
      const int ob = oj % 2;
      wait_bar(x, &B->oready[ob], (oj / 2) & 1);
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
      uint8_t* st = stage_ptr(x, sj % NS);  // Q | K area: two [128 x 32 fp32] blocks
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<float4*>(st + sw128_offset(row, cc)) =
            make_float4(__uint_as_float(n0[4 * cc]) * inv, __uint_as_float(n0[4 * cc + 1]) * inv,
                        __uint_as_float(n0[4 * cc + 2]) * inv, __uint_as_float(n0[4 * cc + 3]) * inv);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<float4*>(st + BLK + sw128_offset(row, cc)) =
            make_float4(__uint_as_float(n1[4 * cc]) * inv, __uint_as_float(n1[4 * cc + 1]) * inv,
                        __uint_as_float(n1[4 * cc + 2]) * inv, __uint_as_float(n1[4 * cc + 3]) * inv);
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (et == 32) {  // the bulk-store thread (never publishes flags)
        const int tok = it.tok0 + c * C;
        tma_store_3d(to, st, 0, tok, it.h);
        tma_store_3d(to, st + BLK, 32, tok, it.h);
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(&B->empty[sj % NS]);
      }
    }
    ++itn;
  }
  if (et == 32) bulk_wait_all();
}

// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const TcParams p, const unsigned long long mbar_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const unsigned epoch = *reinterpret_cast<volatile unsigned*>(&p.hdr->epoch) & 0x3FFFFFFFu;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->xf[s], 8);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->accB[b], 1);
      mbar_init(&bars->pready[b], 4);
      mbar_init(&bars->freeb[b], 1);
      mbar_init(&bars->oready[b], 1);
      mbar_init(&bars->ofree[b], 4);
    }
    mbar_init(&bars->accA, 1);
    mbar_init(&bars->rfree, 1);
    mbar_init(&bars->eready, 4);
    mbar_init(&bars->snapfree, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  // constant operand data: the ones tile (column 0 = 1 in every token row,
  // MN-major 128-byte swizzle) and the snapshots' zero rows 66..79
  for (int i = threadIdx.x; i < (int)(BLK / 16); i += kThreads)
    reinterpret_cast<uint4*>(smem + OFF_ONES)[i] = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < (int)(kMaxChunks * SNAP / 16); i += kThreads)
    reinterpret_cast<uint4*>(smem + OFF_ESNAP)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (threadIdx.x < C) {  // token row t: logical chunk 0 sits at physical chunk t % 8
    const int t = threadIdx.x;
    *reinterpret_cast<uint16_t*>(smem + OFF_ONES + sw128_offset(t, 0)) = 0x3F80u;  // bf16 1.0
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  Ctx x{&p, smem, bars, *reinterpret_cast<volatile uint32_t*>(&bars->tmem_slot), epoch, mbar_ns};
  if (warp == 0) {
    if (lane == 0) producer(x, &tm_q, &tm_k, &tm_v);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) mma_issuer(x);
    __syncwarp();
  } else if (warp < 10) {
    transformer(x, threadIdx.x - 64, lane);
  } else if (warp < 14) {
    p_builder(x, warp % 4, lane);
  } else {
    epilogue(x, warp % 4, lane, threadIdx.x - 448, &tm_o);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(x.tmem, kTmemCols);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(&p.hdr->done, 1u);
    if (prev == gridDim.x - 1) {  // last block: reset for the next launch
      p.hdr->done = 0;
      atomicAdd(&p.hdr->epoch, 1u);
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t launch_prefill_tc64(const PrefillArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mo, a.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(prefill_tc64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM);
  if (e != cudaSuccess) return e;
  TcParams p = make_params(a, D);
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  const int grid = p.total_items < sms ? p.total_items : sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc64_kernel, mq, mk, mv, mo, p, mbar_ns);
}

}  // namespace la
