// prefill_noncausal.cu -- the non-causal read order of la_prefill_variant on
// the sm_103a tensor cores, for bf16 inputs at dk = dv = 64 and 128.
//
// Operator (the linear-attention explainer, section 线性化核心): every query
// reads the state over the whole sequence,
//   o_t = phi(q_t)^T S_N / (phi(q_t)^T z_N + eps),
//   S_N = S0 + sum_t phi(k_t) v_t^T,  z_N = z0 + sum_t phi(k_t).
// Three launches over splits of prefill_tc_common.cuh:
//   1. the piece totals R: at d = 64, for calls of at most 2048 chunks, the
//      prefill's prefix kernel (prefill_prefix64.cu), whose totals carry S0 in
//      a piece that starts its head; otherwise the aggregate kernel of the
//      three-launch prefill at that width (prefill_chunked64.cu,
//      prefill_chunked128.cu), whose totals do not;
//   2. the fold of prefill_scan.cuh, once per head: S_N = S0 (unless the
//      totals carry it) + the totals in slot order, stored as S_N, z_N and as
//      the head's bf16 operand tile (StateTile, z as hi + lo rows);
//   3. nc_kernel<D>: per piece of the block's run, its head's tile by one bulk
//      copy; per chunk phi(Q) in place, then [num | den] = phi(Q) [S_N | z_N]^T
//      as one product of N_S = D + 16 columns, o = num / (den + eps) staged
//      for TMA stores.
// At d = 64 a block takes 77 KB of shared memory and the split has two blocks
// per SM; at d = 128 it takes 133 KB and one.  Every wait is bounded; one that
// gives up records a timeout in the library status word and the kernel
// finishes with unspecified outputs.
#include "prefill_scan.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcp;

constexpr uint32_t BLK = 16384;   // [128 rows x 128 B] swizzled block: 64 bf16 or 32 fp32 columns
constexpr int kThreads = 128;     // one thread per chunk row / TMEM lane

template <int D>
struct Nc {
  static constexpr int NS = StateTile<D>::NS;                 // state operand rows (N of the product)
  static constexpr uint32_t QT = (D / 64) * BLK;              // a Q tile: D / 64 column blocks
  static constexpr uint32_t XA = StateTile<D>::XA;            // one K-atom of the state operand
  static constexpr uint32_t XT = StateTile<D>::BYTES;         // the state operand
  static constexpr uint32_t COLS = D == 64 ? 128 : 256;       // TMEM columns allocated
  static constexpr uint32_t OFF_S = 2 * QT;                   // after the two Q stages
  static constexpr uint32_t OFF_OUT = OFF_S + XT;             // output staging: two [128 x 32] fp32 boxes
  static constexpr uint32_t OFF_BAR = OFF_OUT + 2 * BLK;
  static constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;
  static constexpr uint32_t ID = idesc_bf16_f32(128, NS, 0, 0);  // phi(Q) [S | z]^T, both K-major
  static constexpr int SPLIT = D == 64 ? 2 : 1;                  // blocks per SM
  static_assert(OFF_S % 1024 == 0 && OFF_OUT % 1024 == 0, "swizzled tile alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory per block");
  static_assert(NS <= (int)COLS, "TMEM columns");
};

struct Params {
  Split sp;           // this kernel's runs
  Split sr;           // the split of the launch whose slots hold the piece totals
  float eps;
  const uint8_t* tiles;  // [BH] operand tiles of S_N, z_N (StateTile), from the fold
  unsigned* status;
  int force_wait;     // test hook: the first product waits once on a barrier that nothing completes
};

struct Bars {
  uint64_t full[2];
  uint64_t tile;  // a piece's state tile landed (bulk copy)
  uint64_t mma;
  uint64_t never;
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};

struct Ctx {
  unsigned* status;
  volatile int* abort;
  unsigned long long mbar_ns;
};

__device__ __forceinline__ bool waitb(const Ctx& x, uint64_t* bar, uint32_t parity) {
  if (*x.abort) return false;
  if (mbar_try_wait(bar, parity)) return true;
  if (mbar_wait(bar, parity, globaltimer_ns() + x.mbar_ns, x.abort)) return true;
  *x.abort = 1;
  atomicOr(x.status, kStatusTimeout);
  return false;
}

// bytes from global memory into shared memory with one bulk copy, completing
// on `bar` (both addresses 16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void bulk_copy_in(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// One [128 x 32] fp32 box of o: columns 32 b .. 32 b + 31 of this thread's row.
__device__ __forceinline__ void stage_box(uint8_t* box, int t, const uint32_t* n, float inv) {
#pragma unroll
  for (int cc = 0; cc < 8; ++cc)
    *reinterpret_cast<float4*>(box + sw128_offset(t, cc)) =
        make_float4(__uint_as_float(n[4 * cc]) * inv, __uint_as_float(n[4 * cc + 1]) * inv,
                    __uint_as_float(n[4 * cc + 2]) * inv, __uint_as_float(n[4 * cc + 3]) * inv);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
nc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
          const Params p, const unsigned long long mbar_ns) {
  using L = Nc<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* B = reinterpret_cast<Bars*>(smem + L::OFF_BAR);
  uint8_t* stile = smem + L::OFF_S;
  uint8_t* out = smem + L::OFF_OUT;
  const int t = threadIdx.x, warp = t / 32;
  const Split& sp = p.sp;
  const int NC = sp.NC;
  const Run run(sp, blockIdx.x);
  const uint32_t total = (uint32_t)(run.b - run.a);
  if (t == 0) {
    mbar_init(&B->full[0], 1);
    mbar_init(&B->full[1], 1);
    mbar_init(&B->tile, 1);
    mbar_init(&B->mma, 1);
    mbar_init(&B->never, 1);
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_o);
  }
  for (int i = t; i < (int)(L::XT / 16); i += kThreads)  // rows D + 2 .. N_S - 1 stay zero
    reinterpret_cast<uint4*>(stile)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    tmem_alloc(&B->tmem_slot, L::COLS);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *reinterpret_cast<volatile uint32_t*>(&B->tmem_slot);
  const uint32_t tl = tm + ((uint32_t)(32 * warp) << 16);  // this thread's TMEM lane (row t)
  const Ctx x{p.status, &B->abort, mbar_ns};
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&B->abort) != 0; };
  pdl_launch_dependents();
  pdl_wait();  // the piece totals are complete

  uint32_t nload = 0;
  auto load = [&](uint32_t j) {  // thread 0: Q of the run's chunk j into stage j % 2
    const long long gi = run.a + j;
    const int h = (int)(gi / NC), tok = (int)(gi % NC) * C;
    uint8_t* dst = smem + (j % 2) * L::QT;
    mbar_arrive_expect_tx(&B->full[j % 2], L::QT);
#pragma unroll
    for (int b = 0; b < D / 64; ++b) tma_load_3d_ef(dst + b * BLK, &tm_q, 64 * b, tok, h, &B->full[j % 2]);
    ++nload;
  };
  if (t == 0 && total > 0) load(0);

  uint32_t j = 0, nmma = 0;
  Piece pc;
  for (int i = 0; run.piece(sp, i, &pc); ++i) {
    const int h = pc.h;
    // the head's tile, folded once per head by the launch before
    if (t == 0 && !aborted()) {
      mbar_arrive_expect_tx(&B->tile, L::XT);
      bulk_copy_in(stile, p.tiles + (size_t)h * L::XT, L::XT, &B->tile);
    }
    waitb(x, &B->tile, i & 1);
    fence_proxy_async_smem();
    __syncthreads();

    for (int c = 0; c < pc.nch; ++c, ++j) {
      const int s = j % 2;
      uint8_t* qt = smem + s * L::QT;
      const int tok = pc.tok0 + c * C;
      if (t == 0 && j + 1 < total && !aborted()) load(j + 1);
      waitb(x, &B->full[s], (j / 2) & 1);
#pragma unroll
      for (int b = 0; b < D / 64; ++b) phi_row<8>(qt + b * BLK, t, 0, pc.tok1 - tok);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (t == 0) {
        if ((!p.force_wait || j > 0 || waitb(x, &B->never, 0)) && !aborted()) {
          tc_fence_after();
          const uint32_t qa = smem_u32(qt), sa = smem_u32(stile);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16_ss(tm, sdesc_sw128(qa + (ks / 4) * BLK + (ks % 4) * 32, 16, 1024),
                        sdesc_sw128(sa + (ks / 4) * L::XA + (ks % 4) * 32, 16, 1024), L::ID,
                        ks > 0 ? 1u : 0u);
        }
        mma_commit(&B->mma);
      }
      waitb(x, &B->mma, nmma & 1);
      ++nmma;
      tc_fence_after();
      uint32_t d2[2];
      tmem_ld2(tl + D, d2);
      tmem_ld_wait();
      const float inv = 1.f / (__uint_as_float(d2[0]) + __uint_as_float(d2[1]) + p.eps);
#pragma unroll 1
      for (int r = 0; r < D / 64; ++r) {  // two boxes (64 columns of o) per round
        uint32_t n0[32], n1[32];
        tmem_ld32(tl + 64 * r, n0);
        tmem_ld32(tl + 64 * r + 32, n1);
        tmem_ld_wait();
        if (t == 0) bulk_wait_read_all();  // the previous boxes' stores have read the staging
        tc_fence_before();
        __syncthreads();
        stage_box(out, t, n0, inv);
        stage_box(out + BLK, t, n1, inv);
        fence_proxy_async_smem();
        __syncthreads();
        if (t == 0 && !aborted()) {  // rows past the sequence are not stored
          tma_store_3d_ef(&tm_o, out, 64 * r, tok, h);
          tma_store_3d_ef(&tm_o, out + BLK, 64 * r + 32, tok, h);
          bulk_commit();
        }
      }
    }
    __syncthreads();  // every product that read this piece's state tile is done before the next
  }
  if (t == 0) {
    bulk_wait_all();
    if (aborted()) {  // MMAs and loads in flight end first
      int never = 0;
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, globaltimer_ns() + mbar_ns, &never);
      const uint64_t dl = globaltimer_ns() + mbar_ns;
      for (uint32_t q = (nload > 2 ? nload - 2 : 0); q < nload; ++q)
        mbar_wait(&B->full[q % 2], (q / 2) & 1, dl, &never);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, L::COLS);
  }
}

// Per head: S_N = S0 + the piece totals in slot order, stored as S_N, z_N and
// as the head's operand tile (in place: S_N may be S0).
template <int D>
__global__ void __launch_bounds__(kScanThreads) fold_kernel(const Split sr, const float* R, const float* S0,
                                                            const float* z0, float* S_N, float* z_N,
                                                            uint8_t* tiles) {
  pdl_launch_dependents();  // the reads may be scheduled now; they wait for this grid
  pdl_wait();               // the totals are complete
  scan_fold<D, false>(sr, R, nullptr, nullptr, S0, z0, S_N, z_N, tiles);
}

// The launch of the reads, a programmatic dependent of the one before.
template <int D>
cudaError_t launch_nc_kernel(const PrefillArgs& a, const Params& p, cudaStream_t stream) {
  using L = Nc<D>;
  const int BH = a.B * a.H;
  CUtensorMap mq, mo;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mo, a.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C))
    return cudaErrorInvalidValue;
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  cudaError_t e = cudaFuncSetAttribute(nc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.sp.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::SMEM;
  return cudaLaunchKernelEx(&cfg, nc_kernel<D>, mq, mo, p, mbar_ns);
}

}  // namespace

size_t prefill_nc64_workspace_bytes(int B, int H, int N) {
  return prefill_prefix64_workspace_bytes(B, H, N) + (size_t)B * H * StateTile<64>::BYTES;
}

cudaError_t launch_prefill_nc64(const PrefillArgs& a, cudaStream_t stream) {
  constexpr int D = 64;
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const Split sr = make_split(BH, a.N, sms);
  if (!a.workspace || prefill_nc64_workspace_bytes(a.B, a.H, a.N) > a.ws_bytes) return cudaErrorInvalidValue;
  // the prefill's workspace layout (piece totals, prefix tiles, phi(K); only
  // the totals are written), then one state tile per head
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  Prefix64Buffers b = {};
  b.R = reinterpret_cast<float*>(ws);
  b.P = reinterpret_cast<uint8_t*>(b.R + (size_t)BH * sr.MPH * (D * D + D));  // slots of D D + D floats
  b.phik = reinterpret_cast<__nv_bfloat16*>(b.P + (size_t)sr.TC() * 66 * 128);
  uint8_t* tiles = ws + prefill_prefix64_workspace_bytes(a.B, a.H, a.N);
  cudaError_t e = library_status_word(&b.status);
  if (e != cudaSuccess) return e;
  e = launch_prefix64_totals(a, b, stream);
  if (e != cudaSuccess) return e;
  // the fold (S0 is in the totals already), a programmatic dependent
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kScanThreads);
  cfg.gridDim = dim3(scan_blocks_per_head<D>(), BH);
  e = cudaLaunchKernelEx(&cfg, fold_kernel<D>, sr, (const float*)b.R, (const float*)nullptr,
                         (const float*)nullptr, a.S_N, a.z_N, tiles);
  if (e != cudaSuccess) return e;
  Params p = {};
  p.sp = make_split(BH, a.N, Nc<D>::SPLIT * sms);
  p.sr = sr;
  p.eps = a.eps;
  p.tiles = tiles;
  p.status = b.status;
  p.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);
  return launch_nc_kernel<D>(a, p, stream);
}

size_t prefill_nc_workspace_bytes(int B, int H, int N, int d) {
  const size_t heads = (size_t)B * H;
  if (d == 64) return aggregate64_totals_bytes(B, H, N) + heads * StateTile<64>::BYTES;
  return aggregate128_totals_bytes(B, H, N) + heads * StateTile<128>::BYTES;
}

cudaError_t launch_prefill_nc(const PrefillArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int d = a.dk;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  if ((d != 64 && d != 128) || !a.workspace || prefill_nc_workspace_bytes(a.B, a.H, a.N, d) > a.ws_bytes)
    return cudaErrorInvalidValue;
  // workspace: the piece totals, then one state tile per head
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  float* R = reinterpret_cast<float*>(ws);
  uint8_t* tiles = ws + (d == 64 ? aggregate64_totals_bytes(a.B, a.H, a.N) : aggregate128_totals_bytes(a.B, a.H, a.N));
  Params p = {};
  p.tiles = tiles;
  p.sr = make_split(BH, a.N, sms);
  p.eps = a.eps;
  p.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);
  cudaError_t e = library_status_word(&p.status);
  if (e == cudaSuccess)
    e = d == 64 ? launch_aggregate64_totals(a, R, p.status, stream)
                : launch_aggregate128_totals(a, R, p.status, stream);
  if (e != cudaSuccess) return e;
  // the fold, a programmatic dependent of the aggregate launch
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kScanThreads);
  if (d == 64) {
    cfg.gridDim = dim3(scan_blocks_per_head<64>(), BH);
    e = cudaLaunchKernelEx(&cfg, fold_kernel<64>, p.sr, (const float*)R, a.S0, a.z0, a.S_N, a.z_N, tiles);
    if (e != cudaSuccess) return e;
    p.sp = make_split(BH, a.N, Nc<64>::SPLIT * sms);
    return launch_nc_kernel<64>(a, p, stream);
  }
  cfg.gridDim = dim3(scan_blocks_per_head<128>(), BH);
  e = cudaLaunchKernelEx(&cfg, fold_kernel<128>, p.sr, (const float*)R, a.S0, a.z0, a.S_N, a.z_N, tiles);
  if (e != cudaSuccess) return e;
  p.sp = make_split(BH, a.N, Nc<128>::SPLIT * sms);
  return launch_nc_kernel<128>(a, p, stream);
}

}  // namespace la
