// delta_chunked128.cu -- the delta-rule memory on the sm_103a tensor cores,
// chunkwise, for bf16 keys and values with dk = dv = 128.
//
// Recurrence (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03
// "从累加改成纠错", and page "sequence-models" practice notes, "Delta-rule fast
// weight"): read_t = S_{t-1}^T k_t, then S_t = S_{t-1} + beta_t k_t (v_t - read_t)^T.
//
// Chunkwise form (the LinearMem page names a chunked delta rule as the way to
// train it fast; the steps below follow from the recurrence).  For a chunk of
// C tokens with keys K [C x dk], values V [C x dv], beta, and the state S at
// the chunk's start, let u_t = beta_t (v_t - read_t) and L = strictly lower
// part of K K^T (L[t][s] = k_t . k_s for s < t).  Then
//   read_t = S^T k_t + sum_{s<t} L[t][s] u_s,  i.e.  R = K S + L U,
//   (I + diag(beta) L) U = diag(beta) (V - K S),  i.e.  U = T diag(beta) (V - K S)
//   with T = (I + diag(beta) L)^-1 (unit lower triangular), and
//   S_new = S + K^T U.
// In exact arithmetic this equals the token recurrence; only the order of the
// sums and the operand roundings differ.
//
// Gated form (the LinearMem page, section 03: D = alpha_t S_{t-1}, then the
// correction against D).  With g_t = sum_{r <= t} log2 alpha_r inside the
// chunk, gamma_t = 2^g_t and L~[t][s] = 2^(g_t - g_s) k_t . k_s (s < t), the
// recurrence unrolls to
//   R = diag(gamma) K S + L~ U,   U = T~ diag(beta) (V - diag(gamma) K S),
//   T~ = (I + diag(beta) L~)^-1,  S_new = gamma_C S + K^T diag(gamma_C / gamma) U,
// so the same products run with L~ in place of L; the state warps scale K S by
// gamma_t (in X and, written back, in the reads), keep a second bf16 copy of
// U scaled by gamma_C / gamma_t for the state product, and scale S by gamma_C
// once per chunk.  The decay ratios are taken as 2^(g_t - g_s) <= 1 (a zero
// alpha is clamped to 1e-30), never as quotients.
//
// One block per head, chunks of C = 64 tokens taken in pairs (128 tokens per
// TMA stage, so that the Gram matrix of a pair is one M = 128 product).  The
// state and every product live transposed, TMEM lanes = value columns j:
//   ST  S^T (fp32)                         SB  S^T as packed bf16 (A operand)
//   KR  (K S)^T, then R^T = (K S + L U)^T  UU  U^T (fp32)
//       (KR and UU swap their two 64-column regions from chunk to chunk, so
//       a chunk's reads can leave TMEM while the next chunk runs)
//   XB  (V - K S)^T, packed bf16 (A operand)
//   UB  U^T, packed bf16 (A operand)       LL  K2 K2^T of the pair (lanes = tokens)
// Products per chunk (tcgen05, bf16 operands, fp32 accumulation):
//   KR = SB  x K_c^T    (M 128, N 64, K 128)   UU = XB x (T_c B_c)^T (M 128, N 64, K 64)
//   ST += UB x K_c      (M 128, N 128, K 64)   KR += UB x L_c^T      (M 128, N 64, K 64)
// with B_c = diag(beta) folded into the T operand.  T is computed per chunk
// by 64 threads from A = diag(beta) L (fp32, in shared memory) by block
// recursion: the four 16 x 16 diagonal blocks of (I + A)^-1 by forward
// substitution on CUDA cores, then the off-diagonal blocks from
//   T_ij = -T_ii A_ij T_jj      (lower block row i over block column j)
// first at 16 x 16 and then at 32 x 32 granularity, as small products on the
// warp-level tensor-core instruction (tf32 operands, fp32 accumulation).  A
// column-per-thread substitution over all 64 rows would have every thread
// load the whole of A from shared memory; the products take their operands
// from registers instead.
//
// Schedule: the chunks form one dependent chain (SB -> KR -> XB -> UU -> UB ->
// ST -> SB; the reads' product KR += UB L^T comes after ST's, off the chain).  Off that chain run the TMA loads (K in a ring of three pair
// stages, V in a ring of two chunk slots), the Gram product and T of the NEXT
// pair (its Gram is issued after the current pair's first K S product, once
// the T builders have copied the previous Gram out of TMEM: issuing tensor
// instructions stalls while the tensor queue is full, so it goes where the
// chain waits on the epilogue anyway; T and L operand tiles are double-
// buffered by pair parity), and the global stores of each chunk's reads.
#include "prefill_tc_common.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcp;

namespace dc {

constexpr int D = 128;    // dk = dv
constexpr int CH = 64;    // tokens per chunk
constexpr int PT = 128;   // tokens per pair
constexpr int NK = 3;     // K stages (pairs)
constexpr int NV = 2;     // V slots (chunks)
constexpr uint32_t HALF = PT * 128;          // one 64-element column block of a pair's K: 16 KB
constexpr uint32_t KSTAGE = 2 * HALF;        // K of a pair: 32 KB
constexpr uint32_t VHALF = CH * 128;         // one 64-element column block of a chunk's V: 8 KB
constexpr uint32_t VSLOT = 2 * VHALF;        // V of a chunk: 16 KB
constexpr uint32_t CT = CH * 128;            // a [64 x 64] bf16 operand tile: 8 KB
constexpr uint32_t OFF_V = NK * KSTAGE;      // V slots
constexpr uint32_t OFF_T = OFF_V + NV * VSLOT;  // (T B)_c tiles, [pair parity][chunk]
constexpr uint32_t OFF_L = OFF_T + 4 * CT;   // L_c tiles, [pair parity][chunk]
constexpr uint32_t OFF_LC = OFF_L + 4 * CT;  // fp32 A, then T, of both chunks (2 x 16 KB)
constexpr uint32_t OFF_BETA = OFF_LC + 2 * CH * CH * 4;  // beta of the chunks being solved
constexpr uint32_t OFF_GAM = OFF_BETA + PT * 4;  // gated: [pair parity][chunk] gamma[64], ratio[64]
constexpr uint32_t OFF_BAR = OFF_GAM + 2 * 2 * 2 * CH * 4;
// The dynamic shared window starts 1024-byte aligned (the kernel checks it
// and does no work, with kStatusLayout, otherwise), so no slack is reserved.
constexpr uint32_t SMEM = OFF_BAR + 256;
static_assert(SMEM <= 227 * 1024, "shared memory per block");

constexpr int kWarps = 11;  // 0 TMA of K, 1 MMA, 2-5 T builders, 6-9 state epilogue, 10 TMA of V
constexpr uint32_t kCols = 512;
constexpr uint32_t ST = 0, LL = 128, KRUU = 256, SB = 384, XB = 448, UB = 480;
// (K S)^T / R^T of chunk ch in KRUU + 64 (ch & 1), U^T in the other region
__device__ __forceinline__ uint32_t kr_cols(uint32_t ch) { return KRUU + 64 * (ch & 1); }
__device__ __forceinline__ uint32_t uu_cols(uint32_t ch) { return KRUU + 64 * ((ch + 1) & 1); }

constexpr uint32_t ID_LL = idesc_bf16_f32(128, 128, 0, 0);  // K2 K2^T
constexpr uint32_t ID_KS = idesc_bf16_f32(128, CH, 0, 0);   // SB x K_c^T (B K-major)
constexpr uint32_t ID_U = idesc_bf16_f32(128, CH, 0, 0);    // XB x (T B)_c^T (B K-major)
constexpr uint32_t ID_R = idesc_bf16_f32(128, CH, 0, 0);    // UB x L_c^T (B K-major)
constexpr uint32_t ID_S = idesc_bf16_f32(128, D, 0, 1);     // UB x K_c   (B MN-major)

struct Params {
  int BH, N;
  const float* beta;
  const float* alpha;  // gated form: per-token forgetting (kernel instantiated with GATED)
  const float* S0;
  float* reads;
  float* S_N;
  unsigned* status;
  int force_wait;  // test hook: the MMA thread waits once on a barrier nothing completes
};

struct Bars {
  uint64_t kfull[NK], kempty[NK];  // K ring                 (TMA <-> MMA)
  uint64_t vfull[NV], vfree[NV];   // V ring                 (TMA <-> epilogue)
  uint64_t lready;   // Gram product of a pair in LL        (MMA -> T)
  uint64_t llfree;   // LL copied out by the T builders     (T -> MMA)
  uint64_t tready[2];  // T and L tiles, by pair parity    (T -> MMA)
  uint64_t sbready;  // S^T packed into SB                  (epilogue -> MMA)
  uint64_t krready;  // (K S)^T in KR                       (MMA -> epilogue)
  uint64_t xready;   // X^T packed into XB                  (epilogue -> MMA)
  uint64_t uready;   // U^T in UU                           (MMA -> epilogue)
  uint64_t ubready;  // U^T packed into UB                  (epilogue -> MMA)
  uint64_t sready;   // S^T advanced past the chunk         (MMA -> epilogue)
  uint64_t rready;   // R^T of the chunk in its KR region   (MMA -> epilogue)
  uint64_t drain, drain2;  // completion of the MMA and Gram threads' products on abort
  uint64_t never;          // completed by nothing (the forced-timeout test hook)
  uint32_t tmem_slot;
  int abort;
};

static_assert(sizeof(Bars) <= 256, "barrier block");

struct Ctx {
  const Params* p;
  volatile int* abort;
  unsigned long long ns;
};

__device__ __forceinline__ bool waitd(const Ctx& x, uint64_t* bar, uint32_t parity) {
  if (*x.abort) return false;
  if (mbar_try_wait(bar, parity)) return true;
  if (mbar_wait(bar, parity, globaltimer_ns() + x.ns, x.abort)) return true;
  *x.abort = 1;
  atomicOr(x.p->status, kStatusTimeout);
  return false;
}

__device__ __forceinline__ bool waitd_warp(const Ctx& x, uint64_t* bar, uint32_t parity) {
  return __all_sync(0xFFFFFFFFu, waitd(x, bar, parity));
}

// Element (row, col) of a 128-byte-swizzled bf16 tile with 64 elements per row.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + (col & 7) * 2;
}

__device__ __forceinline__ uint16_t bf16_bits(float f) {
  const __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<const uint16_t*>(&b);
}

// ---- T = (I + A)^-1 of one chunk, A strictly lower 64 x 64 ----------------
// Scratch layout: fp32 row-major, 64 floats per row, 4-float groups permuted
// per row (column c of row r sits at c ^ sw(r)) so that row-wise 16-byte
// stores, column-wise loads and the mma fragment loads below all spread over
// the 32 banks.
__device__ __forceinline__ int sw(int r) { return ((r & 3) << 3) | (((r >> 2) & 1) << 2); }
__device__ __forceinline__ int sidx(int r, int c) { return r * CH + (c ^ sw(r)); }

__device__ __forceinline__ uint32_t to_tf32(float f) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
  return r;
}

// d += a b for one 16 x 8 x 8 tile (warp-level; tf32 operands, fp32 accumulate)
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Fragment of the 16 x 8 left operand whose (m, k) is scratch[r0 + m][k0 + k]:
// lane (g = lane / 4, t = lane % 4) holds (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4).
__device__ __forceinline__ void frag_a(const float* s, int r0, int k0, int lane, uint32_t (&a)[4]) {
  const int g = lane >> 2, t = lane & 3;
  a[0] = to_tf32(s[sidx(r0 + g, k0 + t)]);
  a[1] = to_tf32(s[sidx(r0 + g + 8, k0 + t)]);
  a[2] = to_tf32(s[sidx(r0 + g, k0 + t + 4)]);
  a[3] = to_tf32(s[sidx(r0 + g + 8, k0 + t + 4)]);
}

// Fragment of the 8 x 8 right operand whose (k, n) is scratch[k0 + k][n0 + n]:
// lane holds (t, g) and (t + 4, g).
__device__ __forceinline__ void frag_b(const float* s, int k0, int n0, int lane, uint32_t (&b)[2]) {
  const int g = lane >> 2, t = lane & 3;
  b[0] = to_tf32(s[sidx(k0 + t, n0 + g)]);
  b[1] = to_tf32(s[sidx(k0 + t + 4, n0 + g)]);
}

// scratch[r0 + m][n0 + n] = scale * d(m, n); lane holds (g, 2t), (g, 2t + 1),
// (g + 8, 2t), (g + 8, 2t + 1).
__device__ __forceinline__ void store_d(float* s, int r0, int n0, int lane, const float (&d)[4], float scale) {
  const int g = lane >> 2, t = lane & 3;
  *reinterpret_cast<float2*>(s + sidx(r0 + g, n0 + 2 * t)) = make_float2(scale * d[0], scale * d[1]);
  *reinterpret_cast<float2*>(s + sidx(r0 + g + 8, n0 + 2 * t)) = make_float2(scale * d[2], scale * d[3]);
}

// (T diag(beta))[r][c0], [r][c0 + 1] as one packed bf16 pair of the operand tile
__device__ __forceinline__ void store_tb_pair(uint8_t* ttile, int r, int c0, float v0, float v1) {
  *reinterpret_cast<uint32_t*>(ttile + swz(r, c0)) = pack_bf16x2(v0, v1);
}

// Fragment tile (16 x 8 at rows r0, cols n0) of T, scaled by -1, into the bf16
// (T diag(beta)) operand tile; bs = beta of the chunk's tokens.
__device__ __forceinline__ void store_tb_tile(uint8_t* ttile, const float* bs, int r0, int n0, int lane,
                                              const float (&d)[4]) {
  const int g = lane >> 2, t = lane & 3, c = n0 + 2 * t;
  const float b0 = bs[c], b1 = bs[c + 1];
  store_tb_pair(ttile, r0 + g, c, -d[0] * b0, -d[1] * b1);
  store_tb_pair(ttile, r0 + g + 8, c, -d[2] * b0, -d[3] * b1);
}

// T = (I + A)^-1 for one chunk, and the bf16 operand tile T diag(beta).  The
// scratch holds A (strictly lower, zero elsewhere) on entry; the blocks of T
// that later steps read replace the blocks of A they no longer need, and the
// strict-upper blocks take the intermediate products.  64 threads (two
// warps) of one chunk, tid in [0, 64).  The strictly upper 16 x 16 blocks of
// the bf16 tile are not written (they are zero from the start).  Within each
// step every load comes before every store: the scratch is read and written
// through the same array, so the compiler keeps their program order.
__device__ __forceinline__ void solve_t(float* S, const float* bs, uint8_t* ttile, int tid, int bar_id) {
  const int lane = tid & 31, w = tid >> 5;
  {  // (1) T_qq = (I + A_qq)^-1, q = tid / 16, column tid % 16, axpy order
    const int q = tid >> 4, cc = tid & 15, o = 16 * q;
    float y[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) y[r] = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float xk = (k == cc ? 1.f : 0.f) - y[k];
      y[k] = xk;
#pragma unroll
      for (int r = k + 1; r < 16; ++r) y[r] = fmaf(S[sidx(o + r, o + k)], xk, y[r]);
    }
    __syncwarp();  // the blocks of a warp's threads are read by that warp only
    const float bc = bs[o + cc];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      S[sidx(o + r, o + cc)] = y[r];
      *reinterpret_cast<uint16_t*>(ttile + swz(o + r, o + cc)) = bf16_bits(y[r] * bc);
    }
    __syncwarp();
  }
  {  // (2) warp w, 32-block at O = 32 w: T_10 = -T_11 (A_10 T_00); P = A_10 T_00
     //     goes to the free strict-upper block (rows O.., cols O + 16..)
    const int O = 32 * w;
    uint32_t a0[4], a1[4], b[4][2];
    frag_a(S, O + 16, O, lane, a0);
    frag_a(S, O + 16, O + 8, lane, a1);
    frag_b(S, O, O, lane, b[0]);
    frag_b(S, O + 8, O, lane, b[1]);
    frag_b(S, O, O + 8, lane, b[2]);
    frag_b(S, O + 8, O + 8, lane, b[3]);
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
    mma_tf32(d0, a0, b[0]);
    mma_tf32(d0, a1, b[1]);
    mma_tf32(d1, a0, b[2]);
    mma_tf32(d1, a1, b[3]);
    store_d(S, O, O + 16, lane, d0, 1.f);
    store_d(S, O, O + 24, lane, d1, 1.f);
    __syncwarp();
    frag_a(S, O + 16, O + 16, lane, a0);  // T_11
    frag_a(S, O + 16, O + 24, lane, a1);
    frag_b(S, O, O + 16, lane, b[0]);     // P
    frag_b(S, O + 8, O + 16, lane, b[1]);
    frag_b(S, O, O + 24, lane, b[2]);
    frag_b(S, O + 8, O + 24, lane, b[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) d0[i] = d1[i] = 0.f;
    mma_tf32(d0, a0, b[0]);
    mma_tf32(d0, a1, b[1]);
    mma_tf32(d1, a0, b[2]);
    mma_tf32(d1, a1, b[3]);
    store_d(S, O + 16, O, lane, d0, -1.f);  // over A_10, read above by this warp only
    store_d(S, O + 16, O + 8, lane, d1, -1.f);
    store_tb_tile(ttile, bs, O + 16, O, lane, d0);
    store_tb_tile(ttile, bs, O + 16, O + 8, lane, d1);
  }
  named_bar_sync(bar_id, 64);
  {  // (3) lower-left 32 x 32: T_(23,01) = -T_(23,23) (A_(23,01) T_(01,01)); warp w
     //     on rows r0 = 32 + 16 w; P2 goes to the free block rows 0..31, cols 32..63
    const int r0 = 32 + 16 * w;
    uint32_t a[4][4];
    float d[4][4];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) frag_a(S, r0, 8 * ks, lane, a[ks]);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) d[nt][i] = 0.f;
      // T_(01,01) is lower: columns 16.. have rows 16.. only (rows 0..15 of
      // those columns hold the warp-0 temporary)
#pragma unroll
      for (int ks = (nt < 2 ? 0 : 2); ks < 4; ++ks) {
        uint32_t bb[2];
        frag_b(S, 8 * ks, 8 * nt, lane, bb);
        mma_tf32(d[nt], a[ks], bb);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) store_d(S, 16 * w, 32 + 8 * nt, lane, d[nt], 1.f);
    named_bar_sync(bar_id, 64);
    // -T_(23,23) P2, warp w on columns 16 w .. 16 w + 15 of both row tiles
    // (12 products each).  T_(23,23) rows 32..47 use columns 32..47 only
    // (48.. hold the warp-1 temporary); rows 48..63 use 32..63.
    uint32_t ta[6][4];
    frag_a(S, 32, 32, lane, ta[0]);
    frag_a(S, 32, 40, lane, ta[1]);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) frag_a(S, 48, 32 + 8 * ks, lane, ta[2 + ks]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int n0 = 16 * w + 8 * nt;
      uint32_t bb[4][2];
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) frag_b(S, 8 * ks, 32 + n0, lane, bb[ks]);
#pragma unroll
      for (int i = 0; i < 4; ++i) d[nt][i] = d[2 + nt][i] = 0.f;
      mma_tf32(d[nt], ta[0], bb[0]);
      mma_tf32(d[nt], ta[1], bb[1]);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) mma_tf32(d[2 + nt], ta[2 + ks], bb[ks]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      store_tb_tile(ttile, bs, 32, 16 * w + 8 * nt, lane, d[nt]);
      store_tb_tile(ttile, bs, 48, 16 * w + 8 * nt, lane, d[2 + nt]);
    }
  }
}

// DW: dk = dv of the call (64, 96 or 128, a compile-time stride for the
// stores); the kernel works at 128 with the key and value columns past DW zero.
template <bool GATED, int DW>
__global__ void __launch_bounds__(32 * kWarps, 1)
delta_chunked_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const Params p, const unsigned long long mbar_ns) {
  extern __shared__ uint8_t smem_raw[];
  // The base is offset by a zero the compiler cannot see through: with the
  // base a known constant the kernel measured ~15 % slower.  The swizzled
  // tiles need it 1024-byte aligned, which the dynamic window is; if it were
  // not, the launch does no work and reports kStatusLayout (the layout is
  // never shifted: no slack is reserved).
  uint32_t zero;
  asm volatile("mov.u32 %0, 0;" : "=r"(zero));
  uint8_t* smem = smem_raw + zero;
  const bool aligned = (smem_u32(smem_raw) & 1023u) == 0;
  if (!aligned && threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
  Bars* B = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int head = blockIdx.x;
  const int npairs = aligned ? (p.N + PT - 1) / PT : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NK; ++s) {
      mbar_init(&B->kfull[s], 1);
      mbar_init(&B->kempty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&B->vfull[s], 1);
      mbar_init(&B->vfree[s], 4);
    }
    mbar_init(&B->lready, 1);
    mbar_init(&B->llfree, 4);
    mbar_init(&B->tready[0], 4);
    mbar_init(&B->tready[1], 4);
    mbar_init(&B->sbready, 4);
    mbar_init(&B->krready, 1);
    mbar_init(&B->xready, 4);
    mbar_init(&B->uready, 1);
    mbar_init(&B->ubready, 4);
    mbar_init(&B->sready, 1);
    mbar_init(&B->rready, 1);
    mbar_init(&B->drain, 1);
    mbar_init(&B->drain2, 1);
    mbar_init(&B->never, 1);
    B->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&B->tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot);
  const Ctx x{&p, &B->abort, mbar_ns};

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer of K, one pair (two 64-column halves) per stage
      uint32_t issued = 0;
      for (int pr = 0; pr < npairs; ++pr) {
        const int s = pr % NK;
        if (pr >= NK && !waitd(x, &B->kempty[s], ((pr / NK) - 1) & 1)) break;
        uint8_t* st = smem + s * KSTAGE;
        mbar_arrive_expect_tx(&B->kfull[s], KSTAGE);
        for (int h = 0; h < 2; ++h) tma_load_3d(st + h * HALF, &tm_k, 64 * h, pr * PT, head, &B->kfull[s]);
        ++issued;
      }
      if (*x.abort) {
        int never = 0;
        const uint64_t dl = globaltimer_ns() + mbar_ns;
        for (uint32_t q = (issued > NK ? issued - NK : 0); q < issued; ++q)
          mbar_wait(&B->kfull[q % NK], (q / NK) & 1, dl, &never);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issue
      uint32_t nch = 0;  // chunks done
      bool ok = !p.force_wait || waitd(x, &B->never, 0);
      for (int pr = 0; ok && pr < npairs; ++pr) {
        const int s = pr % NK;
        const uint32_t kb = smem_u32(smem + s * KSTAGE);
        const uint32_t aT = smem_u32(smem + OFF_T + (pr & 1) * 2 * CT);
        const uint32_t aL = smem_u32(smem + OFF_L + (pr & 1) * 2 * CT);
        if (!(ok = waitd(x, &B->tready[pr & 1], (pr >> 1) & 1))) break;
        for (int c = 0; ok && c < 2; ++c, ++nch) {
          const uint32_t kc = kb + c * CT;  // the chunk's 64 rows inside each half
          const uint32_t tc_ = aT + c * CT, lc = aL + c * CT;
          const uint32_t kr = kr_cols(nch), uu = uu_cols(nch);
          if (!(ok = waitd(x, &B->sbready, nch & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)  // KR = SB x K_c^T
            mma_bf16_ts(tmem + kr, tmem + SB + 8 * ks,
                        sdesc_sw128(kc + (ks / 4) * HALF + (ks % 4) * 32, 16, 1024), ID_KS, ks > 0 ? 1u : 0u);
          mma_commit(&B->krready);
          if (!(ok = waitd(x, &B->xready, nch & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < CH / 16; ++ks)  // UU = XB x (T B)_c^T
            mma_bf16_ts(tmem + uu, tmem + XB + 8 * ks, sdesc_sw128(tc_ + ks * 32, 16, 1024), ID_U,
                        ks > 0 ? 1u : 0u);
          mma_commit(&B->uready);
          if (!(ok = waitd(x, &B->ubready, nch & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < CH / 16; ++ks)  // ST += UB x K_c (K rows = tokens, B MN-major);
                                                // gated: the gamma_C / gamma_t scaled copy (in XB)
            mma_bf16_ts(tmem + ST, tmem + (GATED ? XB : UB) + 8 * ks, sdesc_sw128(kc + ks * 2048, HALF, 1024),
                        ID_S, 1u);
          mma_commit(&B->sready);
#pragma unroll
          for (int ks = 0; ks < CH / 16; ++ks)  // KR += UB x L_c^T: the chunk's reads
            mma_bf16_ts(tmem + kr, tmem + UB + 8 * ks, sdesc_sw128(lc + ks * 32, 16, 1024), ID_R, 1u);
          mma_commit(&B->rready);
        }
        if (ok) mma_commit(&B->kempty[s]);
      }
      if (*x.abort) {
        int never = 0;
        mma_commit(&B->drain);
        mbar_wait(&B->drain, 0, globaltimer_ns() + mbar_ns, &never);
      }
    }
    __syncwarp();
  } else if (warp == 10) {
    if (lane == 0) {  // ---- TMA producer of V, one chunk per slot
      uint32_t issued = 0;
      for (int ch = 0; ch < 2 * npairs; ++ch) {
        const int s = ch % NV;
        if (ch >= NV && !waitd(x, &B->vfree[s], ((ch / NV) - 1) & 1)) break;
        uint8_t* st = smem + OFF_V + s * VSLOT;
        mbar_arrive_expect_tx(&B->vfull[s], VSLOT);
        for (int h = 0; h < 2; ++h) tma_load_3d(st + h * VHALF, &tm_v, 64 * h, ch * CH, head, &B->vfull[s]);
        ++issued;
      }
      if (*x.abort) {
        int never = 0;
        const uint64_t dl = globaltimer_ns() + mbar_ns;
        for (uint32_t q = (issued > NV ? issued - NV : 0); q < issued; ++q)
          mbar_wait(&B->vfull[q % NV], (q / NV) & 1, dl, &never);
      }
    }
    __syncwarp();
  } else if (warp < 6) {  // ---- T builders: L and (T B) operand tiles of each pair
    // TMEM lane quadrant = warp % 4: warps 4, 5 hold pair tokens 0..63 (chunk 0),
    // warps 2, 3 pair tokens 64..127 (chunk 1).  Thread ct of a chunk is Gram
    // row ct while copying and T column ct while solving.
    const int quad = warp % 4, c = quad >> 1, ct = 32 * (quad & 1) + lane;
    const int bar_id = 2 + c;  // named barrier of the chunk's 64 threads
    const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16);
    float* sa = reinterpret_cast<float*>(smem + OFF_LC) + c * CH * CH;
    float* bs = reinterpret_cast<float*>(smem + OFF_BETA) + c * CH;
    // The strictly upper 16 x 16 blocks of the (T B) tiles are never written
    // by the solve: zero both pair-parity tiles of this chunk once (the first
    // chunk barrier below orders this before any solve writes).
    for (int e = ct; e < 2 * (int)CT / 16; e += 64) {
      const int par = e / (CT / 16), off = e % (CT / 16);
      *reinterpret_cast<uint4*>(smem + OFF_T + (par * 2 + c) * CT + off * 16) = make_uint4(0, 0, 0, 0);
    }
    const float* beta_h = p.beta + (size_t)head * p.N;
    // beta (and, gated, alpha) of this thread's token, loaded one pair ahead
    float bnext = (c * CH + ct < p.N) ? beta_h[c * CH + ct] : 0.f;
    const float* alpha_h = GATED ? p.alpha + (size_t)head * p.N : nullptr;
    float anext = 1.f;
    if (GATED) anext = (c * CH + ct < p.N) ? alpha_h[c * CH + ct] : 1.f;
    // Gram product of pair q, LL = K2 K2^T (A and B both the pair's K tile,
    // K-major), issued by one T-builder thread: for pair 0 here, for pair
    // q + 1 as soon as T of pair q is done, so that the Gram products run
    // ahead of the state chain instead of on its issue thread.
    const bool gram_thread = warp == 2 && lane == 0;
    auto gram = [&](int q) -> bool {
      const int s = q % NK;
      if (!waitd(x, &B->kfull[s], (q / NK) & 1)) return false;
      tc_fence_after();
      const uint32_t kb = smem_u32(smem + s * KSTAGE);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t a = kb + (ks / 4) * HALF + (ks % 4) * 32;
        mma_bf16_ss(tmem + LL, sdesc_sw128(a, 16, 1024), sdesc_sw128(a, 16, 1024), ID_LL, ks > 0 ? 1u : 0u);
      }
      mma_commit(&B->lready);
      return true;
    };
    bool gram_ok = !gram_thread || npairs == 0 || gram(0);
    __syncwarp();
    for (int pr = 0; pr < npairs; ++pr) {
      // The T and L tiles of this pair parity were last read by the products
      // of pair pr - 2: wait for their completion (the commit of that pair's
      // K stage) before overwriting them.
      bool got = gram_ok && waitd(x, &B->lready, pr & 1);
      if (pr >= 2) got = got && waitd(x, &B->kempty[(pr - 2) % NK], ((pr - 2) / NK) & 1);
      // the chunk's threads agree (barriers follow); this also keeps the copy
      // below from overwriting sa before every thread is done with it
      if (!named_bar_and(bar_id, 64, got)) continue;
      __syncwarp();  // (re)converged for the warp-wide TMEM loads and mma below
      tc_fence_after();
      const float brow = bnext;  // beta of token ct: Gram row ct, T column ct
      bs[ct] = brow;
      const int tok_next = (pr + 1) * PT + c * CH + ct;
      bnext = tok_next < p.N ? beta_h[tok_next] : 0.f;
      // gated: g_ct = sum_{r <= ct} log2 alpha_r over the chunk (inclusive scan
      // over the chunk's 64 threads), kept in this pair parity's gamma array
      float* gam = reinterpret_cast<float*>(smem + OFF_GAM) + ((pr & 1) * 2 + c) * 2 * CH;
      float grow = 0.f, g63 = 0.f;
      if (GATED) {
        const float arow = anext;
        anext = tok_next < p.N ? alpha_h[tok_next] : 1.f;
        grow = log2f(fmaxf(arow, 1e-30f));
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float o = __shfl_up_sync(0xFFFFFFFFu, grow, off);
          if (lane >= off) grow += o;
        }
        gam[ct] = grow;
        named_bar_sync(bar_id, 64);
        if (ct >= 32) {
          grow += gam[31];
          gam[ct] = grow;
        }
        named_bar_sync(bar_id, 64);
        g63 = gam[CH - 1];
      }
      uint8_t* ltile = smem + OFF_L + ((pr & 1) * 2 + c) * CT;
      uint8_t* ttile = smem + OFF_T + ((pr & 1) * 2 + c) * CT;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t g[32];
        tmem_ld32(tl + LL + 64 * c + 32 * h, g);
        tmem_ld_wait();
        float l[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) l[q] = (32 * h + q < ct) ? __uint_as_float(g[q]) : 0.f;
        if (GATED) {  // L~[ct][s] = 2^(g_ct - g_s) k_ct . k_s
#pragma unroll
          for (int q = 0; q < 32; ++q) l[q] *= exp2f(fminf(grow - gam[32 * h + q], 0.f));
        }
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4)  // A row ct = beta_ct L row ct, fp32
          *reinterpret_cast<float4*>(sa + sidx(ct, 32 * h + 4 * g4)) =
              make_float4(brow * l[4 * g4], brow * l[4 * g4 + 1], brow * l[4 * g4 + 2], brow * l[4 * g4 + 3]);
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {  // L row ct, bf16 operand tile
          uint4 w;
          w.x = pack_bf16x2(l[8 * g8 + 0], l[8 * g8 + 1]);
          w.y = pack_bf16x2(l[8 * g8 + 2], l[8 * g8 + 3]);
          w.z = pack_bf16x2(l[8 * g8 + 4], l[8 * g8 + 5]);
          w.w = pack_bf16x2(l[8 * g8 + 6], l[8 * g8 + 7]);
          *reinterpret_cast<uint4*>(ltile + swz(ct, 32 * h + 8 * g8)) = w;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->llfree);  // LL may take the next Gram product
      named_bar_sync(bar_id, 64);
      if (GATED) {  // per-token factors for the state warps: gamma_t and gamma_C / gamma_t
        gam[ct] = exp2f(grow);
        gam[CH + ct] = exp2f(fminf(g63 - grow, 0.f));
      }
      solve_t(sa, bs, ttile, ct, bar_id);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->tready[pr & 1]);
      // the next Gram product, once every T builder has copied this pair's
      // out of LL
      if (gram_thread && pr + 1 < npairs)
        gram_ok = waitd(x, &B->llfree, pr & 1) && gram(pr + 1);
      __syncwarp();
    }
    if (gram_thread && *x.abort) {  // Gram products still in flight finish before TMEM is freed
      int never = 0;
      mma_commit(&B->drain2);
      mbar_wait(&B->drain2, 0, globaltimer_ns() + mbar_ns, &never);
    }
  } else {  // ---- state epilogue: lane j of S^T, one TMEM quadrant per warp
    const int quad = warp % 4, j = 32 * quad + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16);
    // S^T = S0^T
    for (int h = 0; h < 8; ++h) {
      uint32_t w[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        w[q] = __float_as_uint(p.S0 && 16 * h + q < DW && j < DW
                                   ? p.S0[((size_t)head * DW + 16 * h + q) * DW + j] : 0.f);
      tmem_st16(tl + ST + 16 * h, w);
    }
    tmem_st_wait();
    const uint32_t nchunks = 2u * (uint32_t)npairs;
    // value column j of the reads (lanes j >= d hold the zero columns of a
    // narrower call and store nothing)
    const bool jout = j < DW;
    float* reads_j = p.reads + (size_t)head * p.N * DW + (jout ? j : 0);
    for (uint32_t ch = 0; ch < nchunks; ++ch) {
      const uint8_t* vt = smem + OFF_V + (ch % NV) * VSLOT;
      // gated: the pair's gamma factors are published with its T (tready)
      const float* gam = reinterpret_cast<const float*>(smem + OFF_GAM) + (((ch / 2) & 1) * 2 + (ch & 1)) * 2 * CH;
      if (GATED && (ch & 1) == 0) waitd_warp(x, &B->tready[(ch / 2) & 1], ((ch / 2) >> 1) & 1);
      // SB = bf16(S^T) once S has advanced past chunk ch - 1; gated: in the
      // same pass S <- gamma_C S for this chunk's state product (issued after
      // ubready), while SB keeps S itself for K S
      if (ch > 0) waitd_warp(x, &B->sready, (ch - 1) & 1);
      tc_fence_after();
      const float gc = GATED ? gam[CH - 1] : 1.f;
#pragma unroll 1
      for (int h = 0; h < 4; ++h) {
        uint32_t f[32], w[16];
        tmem_ld32(tl + ST + 32 * h, f);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 16; ++q) w[q] = pack_bf16x2(__uint_as_float(f[2 * q]), __uint_as_float(f[2 * q + 1]));
        tmem_st16(tl + SB + 16 * h, w);
        if (GATED) {
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            w0[q] = __float_as_uint(gc * __uint_as_float(f[q]));
            w1[q] = __float_as_uint(gc * __uint_as_float(f[16 + q]));
          }
          tmem_st16(tl + ST + 32 * h, w0);
          tmem_st16(tl + ST + 32 * h + 16, w1);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->sbready);
      // reads of chunk ch - 1 (R^T in its KR region, which this chunk's U^T
      // overwrites only after xready below)
      if (ch > 0) {
        waitd_warp(x, &B->rready, (ch - 1) & 1);
        tc_fence_after();
        const int t0 = (int)(ch - 1) * CH;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t f[32];
          tmem_ld32(tl + kr_cols(ch - 1) + 32 * h, f);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 32; ++q)
            if (jout && t0 + 32 * h + q < p.N) reads_j[(size_t)(t0 + 32 * h + q) * DW] = __uint_as_float(f[q]);
        }
      }
      // V of the chunk, column j, into registers (token pairs packed)
      waitd_warp(x, &B->vfull[ch % NV], (ch / NV) & 1);
      uint32_t vv[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const uint32_t lo = *reinterpret_cast<const uint16_t*>(vt + (j / 64) * VHALF + swz(2 * q, j % 64));
        const uint32_t hi = *reinterpret_cast<const uint16_t*>(vt + (j / 64) * VHALF + swz(2 * q + 1, j % 64));
        vv[q] = lo | (hi << 16);
      }
      // X^T = V^T - (K S)^T, packed over token pairs
      waitd_warp(x, &B->krready, ch & 1);
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t f[32], w[16];
        tmem_ld32(tl + kr_cols(ch) + 32 * h, f);
        tmem_ld_wait();
        if (GATED) {  // (K S)^T -> diag(gamma) (K S)^T, kept for the reads
          uint32_t y0[16], y1[16];
#pragma unroll
          for (int q = 0; q < 32; ++q) f[q] = __float_as_uint(gam[32 * h + q] * __uint_as_float(f[q]));
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            y0[q] = f[q];
            y1[q] = f[16 + q];
          }
          tmem_st16(tl + kr_cols(ch) + 32 * h, y0);
          tmem_st16(tl + kr_cols(ch) + 32 * h + 16, y1);
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const uint32_t v2 = vv[16 * h + q];
          w[q] = pack_bf16x2(__uint_as_float(v2 << 16) - __uint_as_float(f[2 * q]),
                             __uint_as_float(v2 & 0xFFFF0000u) - __uint_as_float(f[2 * q + 1]));
        }
        tmem_st16(tl + XB + 16 * h, w);
      }
      tmem_st_wait();
      tc_fence_before();
      // The V slot goes back to the TMA producer only now that its values
      // have been consumed, and after a proxy fence: these generic-proxy reads
      // must be ordered before the async-proxy (TMA) write that refills the
      // slot.  (Releasing it right after the loads let the refill overtake
      // some of them.)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&B->xready);
        mbar_arrive(&B->vfree[ch % NV]);
      }
      // UB = bf16(U^T)
      waitd_warp(x, &B->uready, ch & 1);
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t f[32], w[16];
        tmem_ld32(tl + uu_cols(ch) + 32 * h, f);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 16; ++q) w[q] = pack_bf16x2(__uint_as_float(f[2 * q]), __uint_as_float(f[2 * q + 1]));
        tmem_st16(tl + UB + 16 * h, w);
        if (GATED) {  // the copy scaled by gamma_C / gamma_t for the state product (XB is free)
          const float* ratio = gam + CH + 32 * h;
#pragma unroll
          for (int q = 0; q < 16; ++q)
            w[q] = pack_bf16x2(ratio[2 * q] * __uint_as_float(f[2 * q]),
                               ratio[2 * q + 1] * __uint_as_float(f[2 * q + 1]));
          tmem_st16(tl + XB + 16 * h, w);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->ubready);
    }
    // the last chunk's reads and S_N = S^T transposed back
    if (nchunks > 0) {
      waitd_warp(x, &B->rready, (nchunks - 1) & 1);
      tc_fence_after();
      const int t0 = (int)(nchunks - 1) * CH;
      for (int h = 0; h < 2; ++h) {
        uint32_t f[32];
        tmem_ld32(tl + kr_cols(nchunks - 1) + 32 * h, f);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q)
          if (jout && t0 + 32 * h + q < p.N) reads_j[(size_t)(t0 + 32 * h + q) * DW] = __uint_as_float(f[q]);
      }
      waitd_warp(x, &B->sready, (nchunks - 1) & 1);
      tc_fence_after();
    }
    for (int h = 0; h < 4; ++h) {
      uint32_t f[32];
      tmem_ld32(tl + ST + 32 * h, f);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 32; ++q)
        if (jout && 32 * h + q < DW) p.S_N[((size_t)head * DW + 32 * h + q) * DW + j] = __uint_as_float(f[q]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// Bounded-wait timeouts of the kernels whose calls take no workspace (this
// kernel, and the decayed tensor-core prefill of la_prefill_variant).
__device__ unsigned g_delta_status;

}  // namespace dc
}  // namespace

// dk = dv = 64 and 96 run the same kernel: the K and V maps are as wide as the
// call, so the column blocks past it load as zeros (TMA fills what lies
// outside a tensor), and with zero key and value columns the state's rows and
// columns past d stay exactly zero; only the first d columns are stored.
bool delta_chunked_supported(bool bf16, int dk, int dv) {
  return bf16 && dk == dv && (dk == 64 || dk == 96 || dk == 128);
}

cudaError_t launch_delta_chunked(const void* k, const void* v, const float* beta, const float* alpha,
                                 int B, int H, int N, int d, const float* S0, float* reads, float* S_N,
                                 cudaStream_t stream) {
  using namespace dc;
  if (!delta_chunked_supported(true, d, d)) return cudaErrorInvalidValue;
  unsigned* status = nullptr;
  cudaError_t se = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_delta_status);
  if (se != cudaSuccess) return se;
  const int BH = B * H;
  CUtensorMap mk, mv;
  if (!make_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64, PT) ||
      !make_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64, CH))
    return cudaErrorInvalidValue;
  Params p;
  p.BH = BH;
  p.N = N;
  p.beta = beta;
  p.alpha = alpha;
  p.S0 = S0;
  p.reads = reads;
  p.S_N = S_N;
  p.status = status;
  p.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
    if (e != cudaSuccess) return e;
    kern<<<BH, 32 * kWarps, SMEM, stream>>>(mk, mv, p, mbar_ns);
    return cudaGetLastError();
  };
  if (d == 64) return alpha ? go(delta_chunked_kernel<true, 64>) : go(delta_chunked_kernel<false, 64>);
  if (d == 96) return alpha ? go(delta_chunked_kernel<true, 96>) : go(delta_chunked_kernel<false, 96>);
  return alpha ? go(delta_chunked_kernel<true, 128>) : go(delta_chunked_kernel<false, 128>);
}

cudaError_t library_status_word(unsigned** out) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(out), dc::g_delta_status);
}

cudaError_t delta_status_take(unsigned* out) {
  using namespace dc;
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_delta_status, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_delta_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *out = v;
  return cudaSuccess;
}

}  // namespace la
