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
//   A. for every chunk c of the item: dS_c = phi(K_c)^T V_c, dz_c = phi(K_c)^T 1
//      (tensor cores, fresh accumulator per chunk).  The epilogue warps add the
//      dS_c up in fp32 registers and, after chunk c, snapshot the running sum
//      R_{c+1} = dS_0 + ... + dS_c to bf16 (R_0 = 0): the state each chunk of
//      the item starts from, relative to the item start.  The total R is the
//      item's aggregate, published for the look-back.
//   L. decoupled look-back (bounded waits) for the item's exclusive prefix E
//      (S0 and all earlier items of the head, always the same left fold so that
//      results are bit-identical from run to run); E is snapshotted to bf16.
//   B. for every chunk: scores A = phi(Q_c) phi(K_c)^T (tensor cores); the P
//      warps mask them causally (key <= query, diagonal kept), round to bf16
//      and write P back into the same TMEM columns; then
//        num = P V_c + phi(Q_c) E + phi(Q_c) R_c
//        den = P 1  + phi(Q_c) z_E + phi(Q_c) z_R_c        (z split hi + lo)
//      as tensor-core products with P read from TMEM, and o = num / (den + eps)
//      is stored through TMA.
// Phase B has no serial dependence between chunks, and the look-back of an
// item overlaps with the scores and P of its first chunks.
//
// Warp roles (448 threads):
//   warp 0      TMA producer (3-stage ring of Q | K | V tiles, 48 KB each)
//   warp 1      TMEM owner; lane 0 issues every tcgen05.mma
//   warps 2-5   apply phi in shared memory (K in phase A, Q and K in phase B)
//   warps 6-9   build P from the scores (one warp per TMEM lane quadrant)
//   warps 10-13 state epilogue (phase A), look-back, output epilogue (phase B)
// TMEM (512 columns): A[b] = cols 128b..128b+127 (scores, then P packed in
// place; dS_c | dz_c in phase A), b = 0, 1; O[ob] = cols 256 + 80 ob: 64
// numerator columns, then 16 denominator columns.
#include "prefill_tc_common.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcp;

constexpr int D = 64;
constexpr int NS = 3;                       // stages in the TMA ring
constexpr int kWarps = 14;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxChunks = kItemTokens / C;  // 4
constexpr uint32_t BLK = 16384;             // [128 rows x 128 B] swizzled tile
constexpr uint32_t STAGE = 3 * BLK;         // Q | K | V
constexpr uint32_t SNAP = 8192;             // [64 dk rows x 64 dv] bf16, MN-major B operand
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_ESNAP = NS * STAGE;                       // bf16(E)
constexpr uint32_t OFF_RSNAP = OFF_ESNAP + SNAP;                 // bf16(R_c), c = 1..3
constexpr uint32_t OFF_BZ = OFF_RSNAP + (kMaxChunks - 1) * SNAP; // z hi/lo: E, R_1..R_3
constexpr uint32_t OFF_B1 = OFF_BZ + kMaxChunks * 2048;          // ones in row 0 (2 blocks)
constexpr uint32_t OFF_BAR = OFF_B1 + 4096;
constexpr uint32_t SMEM = OFF_BAR + 512 + 1024;                  // + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TA = 0;
constexpr uint32_t TO = 256;
constexpr int SZ = D * D + D;

constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);  // phi(Q) phi(K)^T
constexpr uint32_t ID_PV = idesc_bf16_f32(128, D, 0, 1);   // x [*, dv] MN-major B
constexpr uint32_t ID_N16 = idesc_bf16_f32(128, 16, 0, 0); // x [16, *] K-major B
constexpr uint32_t ID_SU = idesc_bf16_f32(128, D, 1, 1);   // phi(K)^T V
constexpr uint32_t ID_ZU = idesc_bf16_f32(128, 16, 1, 0);  // phi(K)^T 1

struct Bars {
  uint64_t full[NS];    // TMA bytes landed              (producer -> phi warps)
  uint64_t xf[NS];      // phi applied                   (phi warps -> MMA)
  uint64_t empty[NS];   // stage free                    (MMA / epilogue -> producer)
  uint64_t accA[2];     // dS_c ready in A[b]            (MMA -> state epilogue)
  uint64_t accB[2];     // scores ready in A[b]          (MMA -> P warps)
  uint64_t pready[2];   // P written into A[b]           (P warps -> MMA)
  uint64_t freeb[2];    // A[b] may be overwritten       (epilogue / MMA -> MMA)
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

__device__ __forceinline__ void phi_tile(uint8_t* tile, int r, int valid) {
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    uint4* ptr = reinterpret_cast<uint4*>(tile + sw128_offset(r, cc));
    uint4 v = *ptr;
    if (r < valid) {
      v.x = phi_bf16x2(v.x);
      v.y = phi_bf16x2(v.y);
      v.z = phi_bf16x2(v.z);
      v.w = phi_bf16x2(v.w);
    } else {
      v = make_uint4(0, 0, 0, 0);
    }
    *ptr = v;
  }
}

__device__ void transformer(const Ctx& x, int r, int lane) {
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
        if (phase == 1) phi_tile(st, r, valid);
        phi_tile(st + BLK, r, valid);
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
  const uint32_t aB1 = smem_u32(x.smem + OFF_B1);
  const uint32_t aE = smem_u32(x.smem + OFF_ESNAP);
  const uint32_t aR = smem_u32(x.smem + OFF_RSNAP);
  const uint32_t aBz = smem_u32(x.smem + OFF_BZ);
  uint32_t sj = 0, aj = 0, oj = 0, itn = 0;
  uint32_t npr[2] = {0, 0};  // uses of pready[b]

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
    // ---- phase A: dS_c, dz_c per chunk, each into a fresh accumulator
    for (int c = 0; c < it.nch; ++c, ++sj, ++aj) {
      acquire(sj, aj);
      const uint32_t st = smem_u32(stage_ptr(x, sj % NS));
      const uint32_t d = tm + TA + 128 * (aj % 2);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) {
        // A = phi(K)^T, MN-major; its second 64-row block (rows 64..127 of the
        // M = 128 product) reads the V tile and is ignored.
        const uint64_t a = sdesc_sw128(st + BLK + ks * 2048, BLK, 1024);
        mma_bf16_ss(d, a, sdesc_sw128(st + 2 * BLK + ks * 2048, BLK, 1024), ID_SU,
                    ks > 0 ? 1u : 0u);
        mma_bf16_ss(d + D, a, sdesc_sw128(aB1 + (ks / 4) * 2048 + (ks % 4) * 32, 16, 1024),
                    ID_ZU, ks > 0 ? 1u : 0u);
      }
      mma_commit(&B->accA[aj % 2]);
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
      const uint32_t dO = tm + TO + 80 * ob, dD = dO + D;
      const uint32_t aP = tm + TA + 128 * b;
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) {  // P V and P 1, P from TMEM (8 columns per 16 keys)
        mma_bf16_ts(dO, aP + 8 * ks, sdesc_sw128(st + 2 * BLK + ks * 2048, BLK, 1024), ID_PV,
                    ks > 0 ? 1u : 0u);
        mma_bf16_ts(dD, aP + 8 * ks, sdesc_sw128(aB1 + (ks / 4) * 2048 + (ks % 4) * 32, 16, 1024),
                    ID_N16, ks > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {  // phi(Q) (E + R_c), phi(Q) (z_E + z_R_c)
        const uint64_t aq = sdesc_sw128(st + ks * 32, 16, 1024);
        mma_bf16_ss(dO, aq, sdesc_sw128(aE + ks * 2048, SNAP, 1024), ID_PV, 1u);
        mma_bf16_ss(dD, aq, sdesc_sw128(aBz + ks * 32, 16, 1024), ID_N16, 1u);
        if (c > 0) {
          mma_bf16_ss(dO, aq, sdesc_sw128(aR + (c - 1) * SNAP + ks * 2048, SNAP, 1024), ID_PV, 1u);
          mma_bf16_ss(dD, aq, sdesc_sw128(aBz + c * 2048 + ks * 32, 16, 1024), ID_N16, 1u);
        }
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
    aj += it.nch;  // phase-A jobs use the A buffers without the P warps
    for (int c = 0; c < it.nch; ++c, ++aj) {
      const int b = aj % 2;
      wait_bar(x, &x.bars->accB[b], nb[b] & 1);
      ++nb[b];
      tc_fence_after();
      const uint32_t base = tl + TA + 128 * b;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {  // keys 32 q4 .. 32 q4 + 31
        uint32_t r[32];
        tmem_ld32(base + 32 * q4, r);
        tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j0 = 32 * q4 + 2 * i;
          const float lo = (j0 <= row) ? __uint_as_float(r[2 * i]) : 0.f;
          const float hi = (j0 + 1 <= row) ? __uint_as_float(r[2 * i + 1]) : 0.f;
          w[i] = pack_bf16x2(lo, hi);
        }
        // packed keys 32 q4 .. +31 go to columns 16 q4 .. +15, already read
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

__device__ __forceinline__ void store_snap_row(uint8_t* snap, int row, const float* v /*64*/) {
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * cc + 0], v[8 * cc + 1]);
    u.y = pack_bf16x2(v[8 * cc + 2], v[8 * cc + 3]);
    u.z = pack_bf16x2(v[8 * cc + 4], v[8 * cc + 5]);
    u.w = pack_bf16x2(v[8 * cc + 6], v[8 * cc + 7]);
    *reinterpret_cast<uint4*>(snap + sw128_offset(row, cc)) = u;
  }
}

// Bz operand (K-major [16 rows][dk]): row 0 = bf16(z), row 1 = bf16(z - row 0).
__device__ __forceinline__ void store_bz(uint8_t* bz, int i, float z) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(z);
  const __nv_bfloat16 lo = __float2bfloat16_rn(z - __bfloat162float(hi));
  const int c8 = i / 8, e = i % 8;
  *reinterpret_cast<__nv_bfloat16*>(bz + sw128_offset(0, c8) + 2 * e) = hi;
  *reinterpret_cast<__nv_bfloat16*>(bz + sw128_offset(1, c8) + 2 * e) = lo;
}

__device__ void epilogue(const Ctx& x, int quad, int lane, int et, const CUtensorMap* to) {
  const TcParams& p = *x.p;
  Bars* B = x.bars;
  const int row = 32 * quad + lane;
  const bool state_row = row < D;  // S / z rows live in TMEM lanes 0..63
  const uint32_t tl = x.tmem + ((uint32_t)(32 * quad) << 16);
  uint8_t* sE = x.smem + OFF_ESNAP;
  uint8_t* sR = x.smem + OFF_RSNAP;
  uint8_t* sBz = x.smem + OFF_BZ;
  uint32_t aj = 0, oj = 0, sj = 0, itn = 0;
  uint32_t na[2] = {0, 0};  // uses of accA[b]

  for (int g = blockIdx.x; g < p.total_items; g += gridDim.x) {
    const Item it = item_of(p, g);
    // the previous item's last MMA has read every snapshot we are about to overwrite
    if (itn > 0) wait_bar(x, &B->snapfree, (itn - 1) & 1);

    // ---- phase A: running sum R of dS_c, dz_c; snapshots R_1..R_{n-1}
    float R[D];
    float Rz = 0.f;
#pragma unroll
    for (int i = 0; i < D; ++i) R[i] = 0.f;
    for (int c = 0; c < it.nch; ++c, ++aj, ++sj) {
      const int b = aj % 2;
      wait_bar(x, &B->accA[b], na[b] & 1);
      ++na[b];
      tc_fence_after();
      if (state_row) {
        const uint32_t base = tl + TA + 128 * b;
        uint32_t r[32];
        tmem_ld32(base, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) R[i] += __uint_as_float(r[i]);
        tmem_ld32(base + 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) R[32 + i] += __uint_as_float(r[i]);
        uint32_t z2[2];
        tmem_ld2(base + D, z2);
        tmem_ld_wait();
        Rz += __uint_as_float(z2[0]);
      }
      tc_fence_before();
      named_bar_sync(1, 128);
      if (et == 0) mbar_arrive(&B->freeb[b]);
      if (c + 1 < it.nch && state_row) {
        store_snap_row(sR + c * SNAP, row, R);
        store_bz(sBz + (c + 1) * 2048, row, Rz);
      }
    }

    // ---- publish the aggregate, look back, publish the inclusive prefix
    float* my_agg = p.agg + (size_t)g * SZ;
    if (state_row) {
#pragma unroll
      for (int i = 0; i < D; i += 4)
        __stcg(reinterpret_cast<float4*>(my_agg + row * D + i),
               make_float4(R[i], R[i + 1], R[i + 2], R[i + 3]));
      __stcg(my_agg + D * D + row, Rz);
    }
    __threadfence();
    named_bar_sync(1, 128);
    if (et == 0) {
      st_release_gpu(&p.flags[g], (x.epoch << 2) | kFlagAggregate);
      B->lb_start = lookback_start(p, it, x.epoch);
    }
    named_bar_sync(1, 128);
    const int start = *reinterpret_cast<volatile int*>(&B->lb_start);
    if (state_row) {
      // E = left fold S0 + agg_0 + ... + agg_{w-1}, eight columns at a time;
      // inclusive = E + R is published, E goes to the bf16 snapshot
      const float* base_src = start >= 0 ? p.inc + (size_t)(start * p.BH + it.h) * SZ
                                         : (p.S0 ? p.S0 + (size_t)it.h * D * D : nullptr);
      float* my_inc = p.inc + (size_t)g * SZ;
      const bool last = it.w == p.items_per_head - 1;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float e[8];
        if (base_src) {
          const float4 u0 = __ldcg(reinterpret_cast<const float4*>(base_src + row * D + 8 * cc));
          const float4 u1 = __ldcg(reinterpret_cast<const float4*>(base_src + row * D + 8 * cc + 4));
          e[0] = u0.x; e[1] = u0.y; e[2] = u0.z; e[3] = u0.w;
          e[4] = u1.x; e[5] = u1.y; e[6] = u1.z; e[7] = u1.w;
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) e[i] = 0.f;
        }
        for (int ww = start + 1; ww < it.w; ++ww) {
          const float* src = p.agg + (size_t)(ww * p.BH + it.h) * SZ + row * D + 8 * cc;
          const float4 u0 = __ldcg(reinterpret_cast<const float4*>(src));
          const float4 u1 = __ldcg(reinterpret_cast<const float4*>(src + 4));
          e[0] += u0.x; e[1] += u0.y; e[2] += u0.z; e[3] += u0.w;
          e[4] += u1.x; e[5] += u1.y; e[6] += u1.z; e[7] += u1.w;
        }
        const float4 i0 = make_float4(e[0] + R[8 * cc + 0], e[1] + R[8 * cc + 1],
                                      e[2] + R[8 * cc + 2], e[3] + R[8 * cc + 3]);
        const float4 i1 = make_float4(e[4] + R[8 * cc + 4], e[5] + R[8 * cc + 5],
                                      e[6] + R[8 * cc + 6], e[7] + R[8 * cc + 7]);
        __stcg(reinterpret_cast<float4*>(my_inc + row * D + 8 * cc), i0);
        __stcg(reinterpret_cast<float4*>(my_inc + row * D + 8 * cc + 4), i1);
        if (last) {
          float* sn = p.S_N + (size_t)it.h * D * D + row * D + 8 * cc;
          *reinterpret_cast<float4*>(sn) = i0;
          *reinterpret_cast<float4*>(sn + 4) = i1;
        }
        uint4 u;
        u.x = pack_bf16x2(e[0], e[1]);
        u.y = pack_bf16x2(e[2], e[3]);
        u.z = pack_bf16x2(e[4], e[5]);
        u.w = pack_bf16x2(e[6], e[7]);
        *reinterpret_cast<uint4*>(sE + sw128_offset(row, cc)) = u;
      }
      float ez = 0.f;
      if (start >= 0) ez = __ldcg(p.inc + (size_t)(start * p.BH + it.h) * SZ + D * D + row);
      else if (p.z0) ez = __ldcg(p.z0 + (size_t)it.h * D + row);
      for (int ww = start + 1; ww < it.w; ++ww)
        ez += __ldcg(p.agg + (size_t)(ww * p.BH + it.h) * SZ + D * D + row);
      __stcg(my_inc + D * D + row, ez + Rz);
      if (last) p.z_N[(size_t)it.h * D + row] = ez + Rz;
      store_bz(sBz, row, ez);
    }
    __threadfence();
    named_bar_sync(1, 128);
    if (et == 0) st_release_gpu(&p.flags[g], (x.epoch << 2) | kFlagInclusive);
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
      if (et == 0) {
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
  if (et == 0) bulk_wait_all();
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
      mbar_init(&bars->xf[s], 4);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->accA[b], 1);
      mbar_init(&bars->accB[b], 1);
      mbar_init(&bars->pready[b], 4);
      mbar_init(&bars->freeb[b], 1);
      mbar_init(&bars->oready[b], 1);
      mbar_init(&bars->ofree[b], 4);
    }
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
  // constant B operands: B1 (row 0 ones, 2 blocks), Bz rows 2..15 zero
  for (int i = threadIdx.x; i < (kMaxChunks * 2048 + 4096) / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + OFF_BZ)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (threadIdx.x < 16) {
    const uint32_t one2 = 0x3F803F80u;  // two bf16 1.0
    reinterpret_cast<uint4*>(smem + OFF_B1 + (threadIdx.x / 8) * 2048)[threadIdx.x % 8] =
        make_uint4(one2, one2, one2, one2);
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
  } else if (warp < 6) {
    transformer(x, threadIdx.x - 64, lane);
  } else if (warp < 10) {
    p_builder(x, warp % 4, lane);
  } else {
    epilogue(x, warp % 4, lane, threadIdx.x - 320, &tm_o);
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
