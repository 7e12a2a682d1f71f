// prefill_tc.cu -- chunked causal prefill on the sm_103a tensor cores.
//
// Operator (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03):
//   o_t = (phi(q_t)^T S_t) / (phi(q_t)^T z_t + eps),  S_t = S_{t-1} + phi(k_t) v_t^T,
//   z_t = z_{t-1} + phi(k_t),  phi = ELU + 1,  write before read.
// Chunkwise evaluation (page "线性注意力与SSM", section 3: a small masked
// phi(Q) phi(K)^T attention inside each chunk, a recurrence across chunks that
// hands over only the state): for a chunk of C = 128 tokens entering with
// state (S_prev, z_prev),
//   P   = phi(Q) phi(K)^T with everything above the diagonal set to 0
//   num = P V + phi(Q) S_prev,  den = P 1 + phi(Q) z_prev + eps,  o = num / den
//   S_prev += phi(K)^T V,  z_prev += phi(K)^T 1.
// Every product is a tcgen05.mma (bf16 operands in shared memory, fp32
// accumulators in TMEM).  The chunk-entry state is snapshotted to bf16 for
// the phi(Q) S_prev product; z_prev is split into two bf16 halves (hi + lo)
// so the dominant denominator term keeps ~16 bits.
//
// Work decomposition.  Each (batch, head) sequence is cut into items of 512
// tokens; items are ordered window-major (all heads' first items, then all
// heads' second items, ...) and dealt round-robin to one persistent block
// per SM.  An item is processed in two phases:
//   A. stream K, V through the tensor cores to get the item's aggregate
//      (dS, dz) = (phi(K)^T V, phi(K)^T 1) and publish it;
//   B. obtain the exclusive prefix state E (S0 plus every earlier item of the
//      same head) and stream Q, K, V again (K, V mostly from L2) to produce o.
// The prefix comes from a decoupled look-back over earlier items' published
// flags.  To keep results bit-identical from run to run the sum is always the
// same left fold, S0 + agg_0 + agg_1 + ...: the look-back finds the nearest
// item with a published inclusive prefix (itself such a left fold) and adds
// the aggregates after it in increasing order.  Every inter-block wait is
// bounded; a wait that gives up records LA_ERR_TIMEOUT in the workspace header
// and the kernel finishes with unspecified outputs.  The launch is
// cooperative, so all blocks are co-resident and a block only ever waits on
// items with smaller indices.
//
// Roles: warp 0 lane 0 issues TMA loads and MMAs; warps 1..8 (two per TMEM
// lane quadrant) apply phi, build the masked P tile, run the normalisation
// epilogue (TMA stores of o), the state snapshots and the look-back.
#include "prefill_tc_common.cuh"

namespace la {


namespace {

using namespace tc;
using namespace tcp;

constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (1 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Cfg {
  static constexpr int DB = D / 64;                    // 128-byte column blocks per row
  static constexpr uint32_t TILE = (uint32_t)C * 128 * DB;
  static constexpr uint32_t BLK = (uint32_t)C * 128;   // one column block of a tile
  // TMEM columns (fp32)
  static constexpr uint32_t T_A = 0;                   // scores, 128
  static constexpr uint32_t T_O = 128;                 // numerator, D
  static constexpr uint32_t T_DEN = 128 + D;           // denominator, 16
  static constexpr uint32_t T_S = 128 + D + 16;        // state, D
  static constexpr uint32_t T_Z = 128 + 2 * D + 16;    // normalizer, 16
  static_assert(T_Z + 16 <= kTmemCols, "TMEM budget");
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = TILE;
  static constexpr uint32_t OFF_V = 2 * TILE;
  static constexpr uint32_t OFF_P = 3 * TILE;          // 2 blocks, 32 KB
  static constexpr uint32_t OFF_SNAP = OFF_P + 2 * BLK;
  static constexpr uint32_t SNAP_BLK = (uint32_t)D * 128;  // [dk rows x 64 dv]
  static constexpr uint32_t OFF_B1 = OFF_SNAP + DB * SNAP_BLK;
  static constexpr uint32_t OFF_BZ = OFF_B1 + 2 * 2048;
  static constexpr uint32_t OFF_BAR = OFF_BZ + DB * 2048;
  static constexpr uint32_t USED = OFF_BAR + 128;
  // request more than half of the SM's shared memory: one block per SM, so a
  // block never waits for TMEM held by a co-resident block
  static constexpr uint32_t SMEM = (USED + 1024 > 120 * 1024 ? USED + 1024 : 120 * 1024);
  static constexpr int SZ = D * D + D;                 // floats per published state
  // instruction descriptors
  static constexpr uint32_t ID_SCORES = idesc_bf16_f32(128, 128, 0, 0);
  static constexpr uint32_t ID_PV = idesc_bf16_f32(128, D, 0, 1);
  static constexpr uint32_t ID_N16 = idesc_bf16_f32(128, 16, 0, 0);
  static constexpr uint32_t ID_SU = idesc_bf16_f32(128, D, 1, 1);
  static constexpr uint32_t ID_ZU = idesc_bf16_f32(128, 16, 1, 0);
};

struct Sync {
  uint64_t* ld;
  uint64_t* x;
  uint64_t* mma;
  volatile int* abort;
  WsHeader* hdr;
  unsigned long long mbar_ns;
};

// Bounded mbarrier wait; on failure record a timeout and raise the block's
// abort flag so that every later wait returns at once.
__device__ __forceinline__ void wait_bar(const Sync& s, uint64_t* bar, uint32_t parity) {
  if (*s.abort) return;
  if (!mbar_wait(bar, parity, globaltimer_ns() + s.mbar_ns, s.abort)) {
    *s.abort = 1;
    atomicOr(&s.hdr->status, kStatusTimeout);
  }
}

// ---------------------------------------------------------------------------
// MMA issue (one thread)

template <int D>
__device__ __forceinline__ void issue_state_update(uint32_t tmem, uint32_t sK, uint32_t sV,
                                                   uint32_t sB1, bool accumulate) {
  using Cf = Cfg<D>;
#pragma unroll
  for (int ks = 0; ks < C / 16; ++ks) {
    // A = phi(K)^T: MN-major (M = dk contiguous, K = token rows)
    const uint64_t a = sdesc_sw128(sK + ks * 2048, Cf::BLK, 1024);
    const uint64_t b = sdesc_sw128(sV + ks * 2048, Cf::BLK, 1024);
    const uint64_t bz = sdesc_sw128(sB1 + (ks / 4) * 2048 + (ks % 4) * 32, 16, 1024);
    const uint32_t acc = (accumulate || ks > 0) ? 1u : 0u;
    mma_bf16_ss(tmem + Cf::T_S, a, b, Cf::ID_SU, acc);
    mma_bf16_ss(tmem + Cf::T_Z, a, bz, Cf::ID_ZU, acc);
  }
}

template <int D>
__device__ __forceinline__ void issue_scores(uint32_t tmem, uint32_t sQ, uint32_t sK) {
  using Cf = Cfg<D>;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = (ks / 4) * Cf::BLK + (ks % 4) * 32;
    mma_bf16_ss(tmem + Cf::T_A, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024),
                Cf::ID_SCORES, ks > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void issue_output(uint32_t tmem, uint32_t sQ, uint32_t sV, uint32_t sP,
                                             uint32_t sSnap, uint32_t sB1, uint32_t sBz) {
  using Cf = Cfg<D>;
#pragma unroll
  for (int ks = 0; ks < C / 16; ++ks) {  // P V and P 1 over the chunk's keys
    const uint64_t a = sdesc_sw128(sP + (ks / 4) * Cf::BLK + (ks % 4) * 32, 16, 1024);
    mma_bf16_ss(tmem + Cf::T_O, a, sdesc_sw128(sV + ks * 2048, Cf::BLK, 1024), Cf::ID_PV,
                ks > 0 ? 1u : 0u);
    mma_bf16_ss(tmem + Cf::T_DEN, a,
                sdesc_sw128(sB1 + (ks / 4) * 2048 + (ks % 4) * 32, 16, 1024), Cf::ID_N16,
                ks > 0 ? 1u : 0u);
  }
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {  // phi(Q) S_prev and phi(Q) (z_hi, z_lo)
    const uint64_t a = sdesc_sw128(sQ + (ks / 4) * Cf::BLK + (ks % 4) * 32, 16, 1024);
    mma_bf16_ss(tmem + Cf::T_O, a, sdesc_sw128(sSnap + ks * 2048, Cf::SNAP_BLK, 1024), Cf::ID_PV,
                1u);
    mma_bf16_ss(tmem + Cf::T_DEN, a,
                sdesc_sw128(sBz + (ks / 4) * 2048 + (ks % 4) * 32, 16, 1024), Cf::ID_N16, 1u);
  }
}

template <int D>
__device__ void ctrl_loop(const TcParams& p, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                          const CUtensorMap* tm_v, uint8_t* smem, uint32_t tmem, const Sync& s) {
  using Cf = Cfg<D>;
  uint8_t* sQ = smem + Cf::OFF_Q;
  uint8_t* sK = smem + Cf::OFF_K;
  uint8_t* sV = smem + Cf::OFF_V;
  const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
  const uint32_t aP = smem_u32(smem + Cf::OFF_P), aSnap = smem_u32(smem + Cf::OFF_SNAP);
  const uint32_t aB1 = smem_u32(smem + Cf::OFF_B1), aBz = smem_u32(smem + Cf::OFF_BZ);
  uint32_t n_ld = 0, n_x = 0, n_mma = 0;
  bool mma_pending = false;

  for (int g = blockIdx.x; g < p.total_items; g += gridDim.x) {
    const Item it = item_of(p, g);
    // ---- phase A: aggregate of the item
    for (int c = 0; c < it.nch; ++c) {
      if (mma_pending) {  // K, V buffers are free once the last MMA batch is done
        wait_bar(s, s.mma, (n_mma - 1) & 1);
        mma_pending = false;
      }
      const int tok = it.tok0 + c * C;
      mbar_arrive_expect_tx(s.ld, 2 * Cf::TILE);
      ++n_ld;
#pragma unroll
      for (int db = 0; db < Cf::DB; ++db) {
        tma_load_3d(sK + db * Cf::BLK, tm_k, 64 * db, tok, it.h, s.ld);
        tma_load_3d(sV + db * Cf::BLK, tm_v, 64 * db, tok, it.h, s.ld);
      }
      wait_bar(s, s.x, n_x & 1);  // phi(K) in place
      ++n_x;
      tc_fence_after();
      issue_state_update<D>(tmem, aK, aV, aB1, c > 0);
      mma_commit(s.mma);
      ++n_mma;
      mma_pending = true;
    }
    wait_bar(s, s.x, n_x & 1);  // prefix state in TMEM and in the snapshot
    ++n_x;
    mma_pending = false;  // the epilogue waited for it before arriving
    // ---- phase B: outputs
    for (int c = 0; c < it.nch; ++c) {
      const int tok = it.tok0 + c * C;
      mbar_arrive_expect_tx(s.ld, 3 * Cf::TILE);
      ++n_ld;
#pragma unroll
      for (int db = 0; db < Cf::DB; ++db) {
        tma_load_3d(sQ + db * Cf::BLK, tm_q, 64 * db, tok, it.h, s.ld);
        tma_load_3d(sK + db * Cf::BLK, tm_k, 64 * db, tok, it.h, s.ld);
        tma_load_3d(sV + db * Cf::BLK, tm_v, 64 * db, tok, it.h, s.ld);
      }
      wait_bar(s, s.x, n_x & 1);  // phi(Q), phi(K)
      ++n_x;
      tc_fence_after();
      issue_scores<D>(tmem, aQ, aK);
      mma_commit(s.mma);
      ++n_mma;
      wait_bar(s, s.x, n_x & 1);  // masked P
      ++n_x;
      tc_fence_after();
      issue_output<D>(tmem, aQ, aV, aP, aSnap, aB1, aBz);
      issue_state_update<D>(tmem, aK, aV, aB1, true);
      mma_commit(s.mma);
      ++n_mma;
      wait_bar(s, s.x, n_x & 1);  // o stored, next snapshot written
      ++n_x;
    }
  }
  if (mma_pending) wait_bar(s, s.mma, (n_mma - 1) & 1);
  if (*s.abort) {
    // a wait gave up: before the block exits, give the last TMA batch and the
    // last MMA batch a bounded chance to land
    int never = 0;
    const uint64_t dl = globaltimer_ns() + s.mbar_ns;
    if (n_ld) mbar_wait(s.ld, (n_ld - 1) & 1, dl, &never);
    if (n_mma) mbar_wait(s.mma, (n_mma - 1) & 1, dl, &never);
  }
}

// ---------------------------------------------------------------------------
// epilogue warps

template <int D>
__device__ __forceinline__ void transform_tile(uint8_t* tile, int et, int valid) {
  using Cf = Cfg<D>;
  const int r = et % C;
  const int part = et / C;
  constexpr int kPer = 4 * Cf::DB;  // 16-byte chunks per thread
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int cc = part * kPer + i;
    uint8_t* ptr = tile + (cc / 8) * Cf::BLK + sw128_offset(r, cc % 8);
    uint4 x = *reinterpret_cast<uint4*>(ptr);
    if (r < valid) {
      x.x = phi_bf16x2(x.x);
      x.y = phi_bf16x2(x.y);
      x.z = phi_bf16x2(x.z);
      x.w = phi_bf16x2(x.w);
    } else {
      x = make_uint4(0, 0, 0, 0);
    }
    *reinterpret_cast<uint4*>(ptr) = x;
  }
}

// Epilogue hand-off to the control thread: make this warp's shared-memory and
// TMEM writes visible to the async proxy / tensor core, then one arrive.
__device__ __forceinline__ void epi_arrive(uint64_t* bar, int lane) {
  fence_proxy_async_smem();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

template <int D>
__device__ __forceinline__ void write_snapshot_row(uint8_t* snap, int row, int col0,
                                                   const float* vals /*D/2*/) {
  // Snap: MN-major B operand [dk rows][dv], blocks of 64 dv columns.
#pragma unroll
  for (int c = 0; c < D / 2; c += 8) {
    const int j = col0 + c;
    uint4 v;
    v.x = pack_bf16x2(vals[c + 0], vals[c + 1]);
    v.y = pack_bf16x2(vals[c + 2], vals[c + 3]);
    v.z = pack_bf16x2(vals[c + 4], vals[c + 5]);
    v.w = pack_bf16x2(vals[c + 6], vals[c + 7]);
    *reinterpret_cast<uint4*>(snap + (j / 64) * Cfg<D>::SNAP_BLK +
                              sw128_offset(row, (j % 64) / 8)) = v;
  }
}

template <int D>
__device__ __forceinline__ void write_bz(uint8_t* bz, int i, float z) {
  // Bz: K-major B operand [16 rows][dk]; row 0 = bf16(z), row 1 = bf16(z - row 0)
  const __nv_bfloat16 hi = __float2bfloat16_rn(z);
  const __nv_bfloat16 lo = __float2bfloat16_rn(z - __bfloat162float(hi));
  const int blk = i / 64, c8 = (i % 64) / 8, e = i % 8;
  *reinterpret_cast<__nv_bfloat16*>(bz + blk * 2048 + sw128_offset(0, c8) + 2 * e) = hi;
  *reinterpret_cast<__nv_bfloat16*>(bz + blk * 2048 + sw128_offset(1, c8) + 2 * e) = lo;
}

template <int D>
__device__ __forceinline__ void tmem_load_half(uint32_t taddr, float* out /*D/2*/) {
#pragma unroll
  for (int c = 0; c < D / 2; c += 16) {
    uint32_t r[16];
    tmem_ld16(taddr + c, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) out[c + i] = __uint_as_float(r[i]);
  }
}

template <int D>
__device__ void epi_loop(const TcParams& p, const CUtensorMap* tm_o, uint8_t* smem, uint32_t tmem,
                         const Sync& s, unsigned epoch, int* lb_start) {
  using Cf = Cfg<D>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int et = threadIdx.x - 32;        // 0..255
  const int quad = warp % 4;              // TMEM lane quadrant of this warp
  const int hf = (warp - 1) / 4;          // column half
  const int row = 32 * quad + lane;       // TMEM lane = tile row
  const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16);
  const bool state_row = row < D;         // rows of S / z
  const int col0 = hf * (D / 2);
  uint8_t* sQ = smem + Cf::OFF_Q;
  uint8_t* sK = smem + Cf::OFF_K;
  uint8_t* sP = smem + Cf::OFF_P;
  uint8_t* sSnap = smem + Cf::OFF_SNAP;
  uint8_t* sBz = smem + Cf::OFF_BZ;
  uint32_t n_ld = 0, n_mma = 0;

  for (int g = blockIdx.x; g < p.total_items; g += gridDim.x) {
    const Item it = item_of(p, g);
    // ---- phase A: phi(K) for each chunk
    for (int c = 0; c < it.nch; ++c) {
      wait_bar(s, s.ld, n_ld & 1);
      ++n_ld;
      transform_tile<D>(sK, et, it.tok1 - (it.tok0 + c * C));
      epi_arrive(s.x, lane);
      ++n_mma;
    }
    wait_bar(s, s.mma, (n_mma - 1) & 1);
    tc_fence_after();

    // ---- aggregate -> workspace
    float a[D / 2];
    float az = 0.f;
    if (state_row) {
      tmem_load_half<D>(tl + Cf::T_S + col0, a);
      if (hf == 0) {
        uint32_t r2[2];
        tmem_ld2(tl + Cf::T_Z, r2);
        tmem_ld_wait();
        az = __uint_as_float(r2[0]);
      }
    }
    float* my_agg = p.agg + (size_t)g * Cf::SZ;
    if (state_row) {
#pragma unroll
      for (int c = 0; c < D / 2; c += 4)
        __stcg(reinterpret_cast<float4*>(my_agg + row * D + col0 + c),
               make_float4(a[c], a[c + 1], a[c + 2], a[c + 3]));
      if (hf == 0) __stcg(my_agg + D * D + row, az);
    }
    __threadfence();
    named_bar_sync(1, 32 * kEpiWarps);
    if (et == 0) st_release_gpu(&p.flags[g], (epoch << 2) | 1u);

    // ---- look-back: nearest earlier item of this head with an inclusive prefix
    if (et == 0) *lb_start = lookback_start(p, it, epoch);
    named_bar_sync(1, 32 * kEpiWarps);
    const int start = *reinterpret_cast<volatile int*>(lb_start);

    float e[D / 2];
    float ez = 0.f;
    if (state_row) {
      // exclusive prefix = left fold S0 + agg_0 + ... + agg_{w-1}
      if (start >= 0) {
        const float* src = p.inc + (size_t)(start * p.BH + it.h) * Cf::SZ;
#pragma unroll
        for (int c = 0; c < D / 2; c += 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + row * D + col0 + c));
          e[c] = v.x; e[c + 1] = v.y; e[c + 2] = v.z; e[c + 3] = v.w;
        }
        ez = __ldcg(src + D * D + row);
      } else {
#pragma unroll
        for (int c = 0; c < D / 2; ++c) e[c] = 0.f;
        if (p.S0) {
          const float* src = p.S0 + (size_t)it.h * D * D;
#pragma unroll
          for (int c = 0; c < D / 2; c += 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(src + row * D + col0 + c));
            e[c] = v.x; e[c + 1] = v.y; e[c + 2] = v.z; e[c + 3] = v.w;
          }
        }
        if (p.z0) ez = __ldcg(p.z0 + (size_t)it.h * D + row);
      }
      for (int ww = start + 1; ww < it.w; ++ww) {
        const float* src = p.agg + (size_t)(ww * p.BH + it.h) * Cf::SZ;
#pragma unroll
        for (int c = 0; c < D / 2; c += 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + row * D + col0 + c));
          e[c] += v.x; e[c + 1] += v.y; e[c + 2] += v.z; e[c + 3] += v.w;
        }
        ez += __ldcg(src + D * D + row);
      }
      // inclusive = exclusive + own aggregate
      float* my_inc = p.inc + (size_t)g * Cf::SZ;
      const bool last = it.w == p.items_per_head - 1;
#pragma unroll
      for (int c = 0; c < D / 2; c += 4) {
        const float4 v = make_float4(e[c] + a[c], e[c + 1] + a[c + 1], e[c + 2] + a[c + 2],
                                     e[c + 3] + a[c + 3]);
        __stcg(reinterpret_cast<float4*>(my_inc + row * D + col0 + c), v);
        if (last)
          *reinterpret_cast<float4*>(p.S_N + (size_t)it.h * D * D + row * D + col0 + c) = v;
      }
      if (hf == 0) {
        __stcg(my_inc + D * D + row, ez + az);
        if (last) p.z_N[(size_t)it.h * D + row] = ez + az;
      }
    }
    __threadfence();
    named_bar_sync(1, 32 * kEpiWarps);
    if (et == 0) st_release_gpu(&p.flags[g], (epoch << 2) | 2u);

    // ---- phase-B entry state: TMEM S, Z <- exclusive prefix; bf16 snapshot
    if (state_row) {
#pragma unroll
      for (int c = 0; c < D / 2; c += 16) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(e[c + i]);
        tmem_st16(tl + Cf::T_S + col0 + c, r);
      }
      if (hf == 0) {
        uint32_t r[16];
        r[0] = __float_as_uint(ez);
#pragma unroll
        for (int i = 1; i < 16; ++i) r[i] = 0u;
        tmem_st16(tl + Cf::T_Z, r);
        write_bz<D>(sBz, row, ez);
      }
      tmem_st_wait();
      write_snapshot_row<D>(sSnap, row, col0, e);
    }
    epi_arrive(s.x, lane);

    // ---- phase B
    for (int c = 0; c < it.nch; ++c) {
      const int tok = it.tok0 + c * C;
      const int valid = it.tok1 - tok;
      wait_bar(s, s.ld, n_ld & 1);
      ++n_ld;
      transform_tile<D>(sQ, et, valid);
      transform_tile<D>(sK, et, valid);
      epi_arrive(s.x, lane);

      // masked scores -> P (bf16, K-major, 2 blocks of 64 keys)
      wait_bar(s, s.mma, n_mma & 1);
      ++n_mma;
      tc_fence_after();
#pragma unroll
      for (int cb = 0; cb < 64; cb += 16) {
        uint32_t r[16];
        tmem_ld16(tl + Cf::T_A + hf * 64 + cb, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; i += 8) {
          float f[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int j = hf * 64 + cb + i + k;
            f[k] = (j <= row) ? __uint_as_float(r[i + k]) : 0.f;
          }
          uint4 v;
          v.x = pack_bf16x2(f[0], f[1]);
          v.y = pack_bf16x2(f[2], f[3]);
          v.z = pack_bf16x2(f[4], f[5]);
          v.w = pack_bf16x2(f[6], f[7]);
          *reinterpret_cast<uint4*>(sP + hf * Cf::BLK + sw128_offset(row, (cb + i) / 8)) = v;
        }
      }
      epi_arrive(s.x, lane);

      // o = num / den -> staging (fp32, 128-byte swizzled blocks of 32 columns)
      wait_bar(s, s.mma, n_mma & 1);
      ++n_mma;
      tc_fence_after();
      {
        uint32_t d2[2];
        tmem_ld2(tl + Cf::T_DEN, d2);
        tmem_ld_wait();
        const float inv = 1.f / (__uint_as_float(d2[0]) + __uint_as_float(d2[1]) + p.eps);
#pragma unroll
        for (int cb = 0; cb < D / 2; cb += 16) {
          uint32_t r[16];
          tmem_ld16(tl + Cf::T_O + col0 + cb, r);
          tmem_ld_wait();
          const int j0 = col0 + cb;  // first output column of these 16
          const int blk = j0 / 32;
          uint8_t* st = (blk < 2) ? sP + blk * Cf::BLK : sQ + (blk - 2) * Cf::BLK;
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 v = make_float4(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv,
                                         __uint_as_float(r[i + 2]) * inv,
                                         __uint_as_float(r[i + 3]) * inv);
            *reinterpret_cast<float4*>(st + sw128_offset(row, ((j0 % 32) + i) / 4)) = v;
          }
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(2 + hf, 128);
      if (et == hf * 128) {
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          const int blk = hf * (D / 64) + b;
          const uint8_t* st = (blk < 2) ? sP + blk * Cf::BLK : sQ + (blk - 2) * Cf::BLK;
          tma_store_3d(tm_o, st, 32 * blk, tok, it.h);
        }
        bulk_commit();
        bulk_wait_read_all();
      }
      // state snapshot for the next chunk
      if (c + 1 < it.nch && state_row) {
        float sv[D / 2];
        tmem_load_half<D>(tl + Cf::T_S + col0, sv);
        write_snapshot_row<D>(sSnap, row, col0, sv);
        if (hf == 0) {
          uint32_t r2[2];
          tmem_ld2(tl + Cf::T_Z, r2);
          tmem_ld_wait();
          write_bz<D>(sBz, row, __uint_as_float(r2[0]));
        }
      }
      epi_arrive(s.x, lane);
    }
  }
  // every TMA store of this block has completed before the block exits
  if (et == 0 || et == 128) bulk_wait_all();
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const TcParams p, const unsigned long long mbar_ns) {
  using Cf = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array by pointer
  // arithmetic so that accesses through it stay shared-space accesses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cf::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 5);
  int* lb_start = reinterpret_cast<int*>(bars + 6);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // the flag generation of this launch (advanced by the last block to finish);
  // a flag word is (generation << 2) | state, so 30 bits of it are compared
  const unsigned epoch = *reinterpret_cast<volatile unsigned*>(&p.hdr->epoch) & 0x3FFFFFFFu;

  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);          // TMA loads
    mbar_init(&bars[1], kEpiWarps);  // epilogue -> control
    mbar_init(&bars[2], 1);          // MMA completion
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  if (warp >= 1) {
    // constant B operands: B1 (row 0 = ones, 2 blocks), Bz (rows 2..15 zero)
    const int et = threadIdx.x - 32;
    uint8_t* b1 = smem + Cf::OFF_B1;
    for (int i = et; i < (4096 + Cf::DB * 2048) / 16; i += 32 * kEpiWarps)
      reinterpret_cast<uint4*>(b1)[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (warp >= 1) {
    const int et = threadIdx.x - 32;
    if (et < 16) {  // row 0 of both B1 blocks: 64 ones each
      const uint32_t one2 = 0x3F803F80u;  // two bf16 1.0
      reinterpret_cast<uint4*>(smem + Cf::OFF_B1 + (et / 8) * 2048)[et % 8] =
          make_uint4(one2, one2, one2, one2);
    }
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  Sync s{&bars[0], &bars[1], &bars[2], abort_flag, p.hdr, mbar_ns};
  if (warp == 0) {
    if (lane == 0) ctrl_loop<D>(p, &tm_q, &tm_k, &tm_v, smem, tmem, s);
    __syncwarp();
  } else {
    epi_loop<D>(p, &tm_o, smem, tmem, s, epoch, lb_start);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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

// ---------------------------------------------------------------------------
// host side

template <int D>
cudaError_t launch_d(const PrefillArgs& a, cudaStream_t stream) {
  using Cf = Cfg<D>;
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
    e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Cf::SMEM);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prefill_tc_kernel<D>, kThreads,
                                                    Cf::SMEM);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;

  TcParams p = make_params(a, D);
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);

  const int grid = p.total_items < sms ? p.total_items : sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cf::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D>, mq, mk, mv, mo, p, mbar_ns);
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs& a) {
  return a.bf16 && a.dk == a.dv && (a.dk == 64 || a.dk == 128) && a.chunk == C && a.N > 0 &&
         get_encode() != nullptr;
}

size_t prefill_tc_workspace_bytes(int B, int H, int N, int d, int /*chunk*/) {
  if (d == 64) return prefill_chunked64_workspace_bytes(B, H, N);
  return prefill_chunked128_workspace_bytes(B, H, N);
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream) {
  if (a.dk == 64) return launch_prefill_chunked64(a, stream);
  return launch_prefill_chunked128(a, stream);
}

}  // namespace la
