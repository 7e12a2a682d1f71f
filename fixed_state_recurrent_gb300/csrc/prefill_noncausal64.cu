// prefill_noncausal64.cu -- the non-causal read order of la_prefill_variant on
// the sm_103a tensor cores, for bf16 inputs at dk = dv = 64.
//
// Operator (the linear-attention explainer, section 线性化核心): every query
// reads the state over the whole sequence,
//   o_t = phi(q_t)^T S_N / (phi(q_t)^T z_N + eps),
//   S_N = S0 + sum_t phi(k_t) v_t^T,  z_N = z0 + sum_t phi(k_t).
// Two launches over splits of prefill_tc_common.cuh:
//   1. the prefill's prefix kernel (prefill_prefix64.cu): the piece totals R
//      (with S0 for a piece that starts its head);
//   2. nc_kernel (two blocks per SM, over a split of twice as many runs): per
//      piece of the block's run, S_N of its head as the sum of the head's
//      totals from the first launch (fp32, in slot order), a bf16 operand tile (z as
//      hi + lo rows); per chunk [num | den] = phi(Q) [S_N | z_N]^T as one
//      N = 80 product, o = num / (den + eps) staged for TMA.  The block that
//      holds a head's last chunk writes S_N, z_N.
// Every wait is bounded; one that gives up records a timeout in the library
// status word and the kernel finishes with unspecified outputs.
#include "prefill_tc_common.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcp;

constexpr int D = 64;
constexpr int SZ = D * D + D;         // floats per state slot (S^T rows, then z)
constexpr uint32_t BLK = 16384;       // [128 rows x 128 B] swizzled tile
constexpr uint32_t XT = 80 * 128;     // the state operand: [80 x 64] bf16, rows 66..79 zero

constexpr int kThreads = 128;         // one thread per chunk row / TMEM lane
constexpr uint32_t kCols = 128;
constexpr uint32_t OFF_S = 2 * BLK;   // after the two Q stages
constexpr uint32_t OFF_OUT = OFF_S + XT;  // output staging: two [128 x 32] fp32 boxes
constexpr uint32_t OFF_BAR = OFF_OUT + 2 * BLK;
constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;
static_assert(OFF_S % 1024 == 0 && OFF_OUT % 1024 == 0, "swizzled tile alignment");
static_assert(SMEM <= 227 * 1024, "shared memory per block");

constexpr uint32_t ID_N80 = idesc_bf16_f32(128, D + 16, 0, 0);  // phi(Q) [S | z]^T, both K-major

struct Params {
  Split sp;         // this kernel's runs (two blocks per SM)
  Split sr;         // the prefix kernel's split, whose slots hold the piece totals
  float eps;
  const float* R;   // [BH * sr.MPH][SZ] piece totals (slot layout)
  float* S_N;
  float* z_N;
  unsigned* status;
  int force_wait;   // test hook: the first product waits once on a barrier that nothing completes
};

struct Bars {
  uint64_t full[2];
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

__global__ void __launch_bounds__(kThreads, 1)
nc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
          const Params p, const unsigned long long mbar_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* B = reinterpret_cast<Bars*>(smem + OFF_BAR);
  uint8_t* stile = smem + OFF_S;
  uint8_t* out = smem + OFF_OUT;
  const int t = threadIdx.x, warp = t / 32;
  const Split& sp = p.sp;
  const int N = sp.N, NC = sp.NC;
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
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_o);
  }
  for (int i = t; i < (int)(XT / 16); i += kThreads)  // rows 66..79 stay zero
    reinterpret_cast<uint4*>(stile)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    tmem_alloc(&B->tmem_slot, kCols);
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
    mbar_arrive_expect_tx(&B->full[j % 2], BLK);
    tma_load_3d_ef(smem + (j % 2) * BLK, &tm_q, 0, tok, h, &B->full[j % 2]);
    ++nload;
  };
  if (t == 0 && total > 0) load(0);

  uint32_t j = 0, nmma = 0;
  Piece pc;
  for (int i = 0; run.piece(sp, i, &pc); ++i) {
    // S_N of the piece's head: the sum of all its slots, in slot order
    const int h = pc.h;
    const Split& sr = p.sr;
    const int nb = sr.owner((long long)h * NC + NC - 1) - sr.owner((long long)h * NC) + 1;
    const bool last = pc.tok1 == N;  // this block holds the head's last chunk: it writes S_N, z_N
    const float4* Rh = reinterpret_cast<const float4*>(p.R + (size_t)h * sr.MPH * SZ);
    for (int f = t; f < SZ / 4; f += kThreads) {
      constexpr int U = 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k0 = 0; k0 < nb; k0 += U) {
        float4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          r[u] = k0 + u < nb ? __ldcg(Rh + (size_t)(k0 + u) * (SZ / 4) + f) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          acc.x += r[u].x; acc.y += r[u].y; acc.z += r[u].z; acc.w += r[u].w;
        }
      }
      const int row = f / 16, col = 4 * (f % 16);
      uint2 hi;
      hi.x = pack_bf16x2(acc.x, acc.y);
      hi.y = pack_bf16x2(acc.z, acc.w);
      if (row < D) {
        *reinterpret_cast<uint2*>(stile + sw128_offset(row, col / 8) + (col % 8) * 2) = hi;
      } else {  // z: hi in row 64, lo in row 65
        uint2 lo;
        lo.x = pack_bf16x2(acc.x - __uint_as_float(hi.x << 16), acc.y - __uint_as_float(hi.x & 0xFFFF0000u));
        lo.y = pack_bf16x2(acc.z - __uint_as_float(hi.y << 16), acc.w - __uint_as_float(hi.y & 0xFFFF0000u));
        *reinterpret_cast<uint2*>(stile + sw128_offset(64, col / 8) + (col % 8) * 2) = hi;
        *reinterpret_cast<uint2*>(stile + sw128_offset(65, col / 8) + (col % 8) * 2) = lo;
      }
      if (last && !aborted()) {
        if (row < D) {  // slot row j holds column j of S
          p.S_N[((size_t)h * D + col + 0) * D + row] = acc.x;
          p.S_N[((size_t)h * D + col + 1) * D + row] = acc.y;
          p.S_N[((size_t)h * D + col + 2) * D + row] = acc.z;
          p.S_N[((size_t)h * D + col + 3) * D + row] = acc.w;
        } else {
          reinterpret_cast<float4*>(p.z_N + (size_t)h * D)[col / 4] = acc;
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    for (int c = 0; c < pc.nch; ++c, ++j) {
      const int s = j % 2;
      uint8_t* qt = smem + s * BLK;
      const int tok = pc.tok0 + c * C;
      if (t == 0 && j + 1 < total && !aborted()) load(j + 1);
      waitb(x, &B->full[s], (j / 2) & 1);
      phi_row<8>(qt, t, 0, pc.tok1 - tok);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (t == 0) {
        if ((!p.force_wait || j > 0 || waitb(x, &B->never, 0)) && !aborted()) {
          tc_fence_after();
          const uint64_t a0 = sdesc_sw128(smem_u32(qt), 16, 1024);
          const uint64_t b0 = sdesc_sw128(smem_u32(stile), 16, 1024);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16_ss(tm, a0 + ks * (32 >> 4), b0 + ks * (32 >> 4), ID_N80, ks > 0 ? 1u : 0u);
        }
        mma_commit(&B->mma);
      }
      waitb(x, &B->mma, nmma & 1);
      ++nmma;
      tc_fence_after();
      uint32_t n0[32], n1[32], d2[2];
      tmem_ld32(tl, n0);
      tmem_ld32(tl + 32, n1);
      tmem_ld2(tl + D, d2);
      tmem_ld_wait();
      const float inv = 1.f / (__uint_as_float(d2[0]) + __uint_as_float(d2[1]) + p.eps);
      if (t == 0) bulk_wait_read_all();  // the previous chunk's store has read the staging
      tc_fence_before();
      __syncthreads();
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<float4*>(out + sw128_offset(t, cc)) =
            make_float4(__uint_as_float(n0[4 * cc]) * inv, __uint_as_float(n0[4 * cc + 1]) * inv,
                        __uint_as_float(n0[4 * cc + 2]) * inv, __uint_as_float(n0[4 * cc + 3]) * inv);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<float4*>(out + BLK + sw128_offset(t, cc)) =
            make_float4(__uint_as_float(n1[4 * cc]) * inv, __uint_as_float(n1[4 * cc + 1]) * inv,
                        __uint_as_float(n1[4 * cc + 2]) * inv, __uint_as_float(n1[4 * cc + 3]) * inv);
      fence_proxy_async_smem();
      __syncthreads();
      if (t == 0 && !aborted()) {  // rows past the sequence are not stored
        tma_store_3d_ef(&tm_o, out, 0, tok, h);
        tma_store_3d_ef(&tm_o, out + BLK, 32, tok, h);
        bulk_commit();
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
    tmem_dealloc(tm, kCols);
  }
}

}  // namespace

cudaError_t launch_prefill_nc64(const PrefillArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const Split sp = make_split(BH, a.N, sms);
  if (!a.workspace || prefill_prefix64_workspace_bytes(a.B, a.H, a.N) > a.ws_bytes)
    return cudaErrorInvalidValue;
  // the prefill's workspace layout: piece totals, prefix tiles, phi(K)
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  Prefix64Buffers b = {};
  b.R = reinterpret_cast<float*>(ws);
  b.P = reinterpret_cast<uint8_t*>(b.R + (size_t)BH * sp.MPH * SZ);
  b.phik = reinterpret_cast<__nv_bfloat16*>(b.P + (size_t)sp.TC() * 66 * 128);
  cudaError_t e = library_status_word(&b.status);
  if (e != cudaSuccess) return e;
  e = launch_prefix64_totals(a, b, stream);
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mo;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, C) ||
      !make_map(&mo, a.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, BH, 32, C))
    return cudaErrorInvalidValue;
  Params p = {};
  p.sp = make_split(BH, a.N, 2 * sms);  // 77 KB of shared memory: two blocks per SM
  p.sr = sp;
  p.eps = a.eps;
  p.R = b.R;
  p.S_N = a.S_N;
  p.z_N = a.z_N;
  p.status = b.status;
  p.force_wait = (int)env_ull("LA_TEST_FORCE_WAIT", 0);
  const unsigned long long mbar_ns = env_ull("LA_MBAR_TIMEOUT_NS", 2000000000ull);
  e = cudaFuncSetAttribute(nc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
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
  cfg.dynamicSmemBytes = SMEM;
  return cudaLaunchKernelEx(&cfg, nc_kernel, mq, mo, p, mbar_ns);
}

}  // namespace la
