// la_api.cu -- the C ABI of libla.so (declared in include/la.h): argument
// validation, path choice and launches on the caller's stream.  No entry point
// allocates memory; every tensor belongs to the caller.
#include "la.h"

#include "la_internal.h"

#include <algorithm>
#include <math.h>
#include <stdint.h>

namespace {

using la::PrefillArgs;

constexpr int kMaxDim = 128;
constexpr int kMaxDevices = 64;

// 0 = unknown, 1 = sm_103 device, 2 = other device.
int g_device_kind[kMaxDevices];

la_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LA_ERR_UNSUPPORTED;
  if (g_device_kind[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return LA_ERR_CUDA;
    g_device_kind[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return g_device_kind[dev] == 1 ? LA_OK : LA_ERR_UNSUPPORTED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
  uintptr_t lo, hi;  // [lo, hi)
};

Span span(const void* p, size_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {a, a + bytes};
}

bool overlap(Span a, Span b) {
  if (a.lo == a.hi || b.lo == b.hi || a.lo == 0 || b.lo == 0) return false;
  return a.lo < b.hi && b.lo < a.hi;
}

bool dims_ok(int B, int H, int N, int dk, int dv) {
  if (B < 1 || H < 1 || N < 0 || dk < 1 || dv < 1) return false;
  if (dk > kMaxDim || dv > kMaxDim) return false;
  const double elems = (double)B * H * (double)(N > 0 ? N : 1) * (dk > dv ? dk : dv);
  return elems < 1099511627776.0;  // 2^40
}

size_t elem_bytes(la_dtype t) { return t == LA_BF16 ? 2 : 4; }

bool dtype_ok(la_dtype t) { return t == LA_F32 || t == LA_BF16; }

la_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

// Copy (or zero) an initial state into a final state for N == 0.
cudaError_t copy_state(const float* src, float* dst, size_t bytes, cudaStream_t s) {
  if (src == dst) return cudaSuccess;
  if (src) return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
  return cudaMemsetAsync(dst, 0, bytes, s);
}

bool use_tensor_path(la_dtype t, int dk, int dv) {
  return t == LA_BF16 && dk == dv && (dk == 64 || dk == 128);
}

}  // namespace

extern "C" {

size_t la_state_bytes(int dk, int dv) {
  if (dk < 1 || dv < 1) return 0;
  return ((size_t)dk * dv + dk) * sizeof(float);
}

const char* la_status_string(la_status s) {
  switch (s) {
    case LA_OK: return "LA_OK";
    case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG: invalid argument";
    case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED: not supported on this device or build";
    case LA_ERR_CUDA: return "LA_ERR_CUDA: a CUDA call failed";
    case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT: a bounded inter-block wait gave up";
  }
  return "LA_ERR_UNKNOWN";
}

size_t la_prefill_workspace_bytes(int B, int H, int N, int dk, int dv,
                                  la_dtype in_dtype, int chunk) {
  if (!dims_ok(B, H, N, dk, dv) || !dtype_ok(in_dtype)) return 0;
  if (chunk != 0 && chunk != 128) return 0;
  size_t bytes = sizeof(la::WsHeader);
  if (use_tensor_path(in_dtype, dk, dv))
    bytes += la::prefill_tc_workspace_bytes(B, H, N, dk, chunk);
  else
    bytes += la::prefill_simt_workspace_bytes(B, H, N, dk, dv);
  return bytes;
}

la_status la_prefill(const void* q, const void* k, const void* v, la_dtype in_dtype,
                     int B, int H, int N, int dk, int dv, float eps,
                     const float* S0, const float* z0, float* o, float* S_N,
                     float* z_N, int chunk, void* workspace, size_t ws_bytes,
                     cudaStream_t stream) {
  return la::prefill_entry(q, k, v, in_dtype, B, H, N, dk, dv, eps, S0, z0, o, S_N, z_N, chunk,
                           workspace, ws_bytes, nullptr, stream);
}

}  // extern "C"

// la_prefill's validation and launch; `status` is where the tensor-core
// kernels record a bounded wait that gave up (NULL: the workspace header).
la_status la::prefill_entry(const void* q, const void* k, const void* v, la_dtype in_dtype,
                            int B, int H, int N, int dk, int dv, float eps, const float* S0,
                            const float* z0, float* o, float* S_N, float* z_N, int chunk,
                            void* workspace, size_t ws_bytes, unsigned* status,
                            cudaStream_t stream) {
  if (!dtype_ok(in_dtype) || !dims_ok(B, H, N, dk, dv)) return LA_ERR_INVALID_ARG;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  if (chunk != 0 && chunk != 128) return LA_ERR_INVALID_ARG;
  if (!S_N || !z_N || !workspace) return LA_ERR_INVALID_ARG;
  if (N > 0 && (!q || !k || !v || !o)) return LA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, S0, z0, o, S_N, z_N, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return LA_ERR_INVALID_ARG;
  const size_t need = la_prefill_workspace_bytes(B, H, N, dk, dv, in_dtype, chunk);
  if (need == 0 || ws_bytes < need) return LA_ERR_INVALID_ARG;

  const size_t heads = (size_t)B * H;
  const size_t eb = elem_bytes(in_dtype);
  const Span sq = span(q, heads * N * dk * eb), sk = span(k, heads * N * dk * eb);
  const Span sv = span(v, heads * N * dv * eb), so = span(o, heads * N * dv * 4);
  const Span sS0 = span(S0, heads * dk * dv * 4), sz0 = span(z0, heads * dk * 4);
  const Span sSN = span(S_N, heads * dk * dv * 4), szN = span(z_N, heads * dk * 4);
  const Span sws = span(workspace, ws_bytes);
  // outputs against every input and each other; S_N may equal S0 exactly
  const Span outs[] = {so, sSN, szN};
  const Span ins[] = {sq, sk, sv, sws};
  for (const Span& a : outs)
    for (const Span& b : ins)
      if (overlap(a, b)) return LA_ERR_INVALID_ARG;
  if (overlap(so, sSN) || overlap(so, szN) || overlap(sSN, szN)) return LA_ERR_INVALID_ARG;
  if (overlap(so, sS0) || overlap(so, sz0) || overlap(szN, sS0) || overlap(sSN, sz0))
    return LA_ERR_INVALID_ARG;
  if (overlap(sSN, sS0) && S_N != S0) return LA_ERR_INVALID_ARG;
  if (overlap(szN, sz0) && z_N != z0) return LA_ERR_INVALID_ARG;

  const la_status dev = check_device();
  if (dev != LA_OK) return dev;

  if (N == 0) {
    cudaError_t e = copy_state(S0, S_N, heads * dk * dv * 4, stream);
    if (e == cudaSuccess) e = copy_state(z0, z_N, heads * dk * 4, stream);
    return from_cuda(e);
  }

  PrefillArgs a = {};
  a.q = q; a.k = k; a.v = v;
  a.bf16 = in_dtype == LA_BF16;
  a.B = B; a.H = H; a.N = N; a.dk = dk; a.dv = dv;
  a.eps = eps;
  a.S0 = S0; a.z0 = z0;
  a.o = o; a.S_N = S_N; a.z_N = z_N;
  a.chunk = chunk == 0 ? 128 : chunk;
  a.workspace = workspace;
  a.ws_bytes = ws_bytes;
  a.status = status;
  if (use_tensor_path(in_dtype, dk, dv) && la::prefill_tc_supported(a))
    return from_cuda(la::launch_prefill_tc(a, stream));
  // the CUDA-core path's chunk slots follow the workspace header
  a.workspace = static_cast<uint8_t*>(workspace) + sizeof(la::WsHeader);
  a.ws_bytes = ws_bytes - sizeof(la::WsHeader);
  return from_cuda(la::launch_prefill_simt(a, stream));
}

extern "C" {

la_status la_decode_step(const void* q, const void* k, const void* v, la_dtype in_dtype,
                         int B, int H, int dk, int dv, float eps, float* S,
                         float* z, float* o, cudaStream_t stream) {
  if (!dtype_ok(in_dtype) || !dims_ok(B, H, 1, dk, dv)) return LA_ERR_INVALID_ARG;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  if (!q || !k || !v || !S || !z || !o) return LA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, S, z, o};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LA_ERR_INVALID_ARG;
  const size_t heads = (size_t)B * H;
  const size_t eb = elem_bytes(in_dtype);
  const Span sq = span(q, heads * dk * eb), sk = span(k, heads * dk * eb);
  const Span sv = span(v, heads * dv * eb), so = span(o, heads * dv * 4);
  const Span sS = span(S, heads * dk * dv * 4), sz = span(z, heads * dk * 4);
  const Span outs[] = {so, sS, sz};
  const Span ins[] = {sq, sk, sv};
  for (const Span& a : outs)
    for (const Span& b : ins)
      if (overlap(a, b)) return LA_ERR_INVALID_ARG;
  if (overlap(so, sS) || overlap(so, sz) || overlap(sS, sz)) return LA_ERR_INVALID_ARG;
  const la_status dev = check_device();
  if (dev != LA_OK) return dev;
  return from_cuda(la::launch_decode_step(q, k, v, in_dtype == LA_BF16, B, H, dk,
                                          dv, eps, S, z, o, stream));
}

size_t la_prefill_variant_workspace_bytes(int B, int H, int N, int dk, int dv, la_dtype in_dtype,
                                          la_mode mode, int decay) {
  if (!dtype_ok(in_dtype) || !dims_ok(B, H, N, dk, dv)) return 0;
  if (mode != LA_MODE_CAUSAL && mode != LA_MODE_READ_BEFORE_WRITE && mode != LA_MODE_NONCAUSAL)
    return 0;
  // with a decay (write then read, or read before write), bf16 at dk = dv = 64
  // or 128: the decayed tensor-core forms
  if (decay && in_dtype == LA_BF16 && dk == 64 && dv == 64 && N > 0)
    return la::prefill_decay64_workspace_bytes(B, H, N);
  if (decay && in_dtype == LA_BF16 && dk == 128 && dv == 128 && N > 0)
    return std::max(la::prefill_decay128_workspace_bytes(B, H, N),
                    la::prefill_simt_workspace_bytes(B, H, N, dk, dv));
  // no decay, another read order, bf16 at dk = dv = 64 or 128: the tensor-core
  // form, or the CUDA-core one if it cannot run
  if (!decay && mode != LA_MODE_CAUSAL && in_dtype == LA_BF16 && dk == dv && (dk == 64 || dk == 128) &&
      N > 0) {
    size_t tc = 0;
    if (dk == 64 && la::prefill_prefix64_chosen(B, H, N))
      tc = mode == LA_MODE_NONCAUSAL ? la::prefill_nc64_workspace_bytes(B, H, N)
                                     : la::prefill_prefix64_workspace_bytes(B, H, N);
    else if (mode == LA_MODE_READ_BEFORE_WRITE)
      tc = sizeof(la::WsHeader) + la::prefill_tc_workspace_bytes(B, H, N, dk, 128);
    else
      tc = la::prefill_nc_workspace_bytes(B, H, N, dk);
    return std::max(tc, la::prefill_simt_workspace_bytes(B, H, N, dk, dv));
  }
  return la::prefill_simt_workspace_bytes(B, H, N, dk, dv);
}

la_status la_prefill_variant(const void* q, const void* k, const void* v, la_dtype in_dtype,
                             int B, int H, int N, int dk, int dv, float eps,
                             const float* alpha, la_mode mode,
                             const float* S0, const float* z0, float* o, float* S_N,
                             float* z_N, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!dtype_ok(in_dtype) || !dims_ok(B, H, N, dk, dv)) return LA_ERR_INVALID_ARG;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  if (mode != LA_MODE_CAUSAL && mode != LA_MODE_READ_BEFORE_WRITE && mode != LA_MODE_NONCAUSAL)
    return LA_ERR_INVALID_ARG;
  if (mode == LA_MODE_NONCAUSAL && alpha) return LA_ERR_INVALID_ARG;
  if (!S_N || !z_N) return LA_ERR_INVALID_ARG;
  if (N > 0 && (!q || !k || !v || !o)) return LA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, alpha, S0, z0, o, S_N, z_N, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return LA_ERR_INVALID_ARG;
  if (workspace &&
      ws_bytes < la_prefill_variant_workspace_bytes(B, H, N, dk, dv, in_dtype, mode, alpha != nullptr))
    return LA_ERR_INVALID_ARG;

  const size_t heads = (size_t)B * H;
  const size_t eb = elem_bytes(in_dtype);
  const Span sq = span(q, heads * N * dk * eb), sk = span(k, heads * N * dk * eb);
  const Span sv = span(v, heads * N * dv * eb), so = span(o, heads * N * dv * 4);
  const Span sa = span(alpha, heads * N * 4);
  const Span sw = span(workspace, ws_bytes);
  const Span sS0 = span(S0, heads * dk * dv * 4), sz0 = span(z0, heads * dk * 4);
  const Span sSN = span(S_N, heads * dk * dv * 4), szN = span(z_N, heads * dk * 4);
  const Span outs[] = {so, sSN, szN};
  const Span ins[] = {sq, sk, sv, sa};
  for (const Span& x : outs)
    for (const Span& y : ins)
      if (overlap(x, y)) return LA_ERR_INVALID_ARG;
  const Span all[] = {sq, sk, sv, sa, so, sSN, szN, sS0, sz0};
  for (const Span& x : all)
    if (overlap(sw, x)) return LA_ERR_INVALID_ARG;
  if (overlap(so, sSN) || overlap(so, szN) || overlap(sSN, szN)) return LA_ERR_INVALID_ARG;
  if (overlap(so, sS0) || overlap(so, sz0) || overlap(szN, sS0) || overlap(sSN, sz0))
    return LA_ERR_INVALID_ARG;
  if (overlap(sSN, sS0) && S_N != S0) return LA_ERR_INVALID_ARG;
  if (overlap(szN, sz0) && z_N != z0) return LA_ERR_INVALID_ARG;

  const la_status dev = check_device();
  if (dev != LA_OK) return dev;
  if (N == 0) {
    cudaError_t e = copy_state(S0, S_N, heads * dk * dv * 4, stream);
    if (e == cudaSuccess) e = copy_state(z0, z_N, heads * dk * 4, stream);
    return from_cuda(e);
  }
  PrefillArgs a = {};
  a.q = q; a.k = k; a.v = v;
  a.bf16 = in_dtype == LA_BF16;
  a.B = B; a.H = H; a.N = N; a.dk = dk; a.dv = dv;
  a.eps = eps;
  a.S0 = S0; a.z0 = z0;
  a.o = o; a.S_N = S_N; a.z_N = z_N;
  a.chunk = 0;
  a.workspace = workspace;
  a.ws_bytes = workspace ? ws_bytes : 0;
  // bf16 at dk = dv = 64 with a decay: tensor cores (read before write in the
  // three-launch form with a strict mask, or one block per head)
  if (alpha && la::prefill_decay64_supported(a)) {
    PrefillArgs d = a;
    d.strict = mode == LA_MODE_READ_BEFORE_WRITE;
    return from_cuda(la::launch_prefill_decay64(d, alpha, stream));
  }
  // bf16 at dk = dv = 64 or 128, no decay, with a workspace: the tensor cores
  PrefillArgs tc = a;
  tc.chunk = 128;  // the tensor-core chunk
  // bf16 at dk = dv = 128, write then read with a decay, with a workspace: the
  // three-launch tensor-core form with decay weights
  if (alpha && dk == 128 && workspace && la::prefill_tc_supported(tc) &&
      ws_bytes >= la::prefill_decay128_workspace_bytes(B, H, N)) {
    tc.strict = mode == LA_MODE_READ_BEFORE_WRITE;
    return from_cuda(la::launch_prefill_decay128(tc, alpha, stream));
  }
  if (!alpha && mode != LA_MODE_CAUSAL && workspace && la::prefill_tc_supported(tc)) {
    // d = 64, at most 2048 chunks: the prefill's two launches, read before
    // write with a strict mask; non-causal from their piece totals
    if (dk == 64 && la::prefill_prefix64_chosen(B, H, N) && mode == LA_MODE_READ_BEFORE_WRITE &&
        ws_bytes >= la::prefill_prefix64_workspace_bytes(B, H, N))
      return from_cuda(la::launch_prefill_rbw64(a, stream));
    if (dk == 64 && la::prefill_prefix64_chosen(B, H, N) && mode == LA_MODE_NONCAUSAL &&
        ws_bytes >= la::prefill_nc64_workspace_bytes(B, H, N))
      return from_cuda(la::launch_prefill_nc64(a, stream));
    // otherwise the three-launch prefill of that width with a strict mask, or
    // its aggregate launch and the reads of the final state
    if (mode == LA_MODE_READ_BEFORE_WRITE &&
        ws_bytes >= sizeof(la::WsHeader) + la::prefill_tc_workspace_bytes(B, H, N, dk, 128) &&
        !(dk == 64 && la::prefill_prefix64_chosen(B, H, N))) {
      tc.strict = true;
      const cudaError_t e = la::library_status_word(&tc.status);
      if (e != cudaSuccess) return from_cuda(e);
      return from_cuda(dk == 64 ? la::launch_prefill_chunked64(tc, stream) : la::launch_prefill_chunked128(tc, stream));
    }
    if (mode == LA_MODE_NONCAUSAL && ws_bytes >= la::prefill_nc_workspace_bytes(B, H, N, dk))
      return from_cuda(la::launch_prefill_nc(tc, stream));
  }
  return from_cuda(la::launch_prefill_variant_simt(a, alpha, (int)mode, stream));
}

size_t la_prefill_backward_workspace_bytes(int B, int H, int N, int dk, int dv, la_dtype in_dtype) {
  if (!dtype_ok(in_dtype) || !dims_ok(B, H, N, dk, dv)) return 0;
  if (in_dtype == LA_BF16 && dk == 64 && dv == 64 && N > 0)
    return la::backward_tc64_workspace_bytes(B, H, N);
  return la::backward_simt_workspace_bytes(B, H, N, dk, dv);  // the CUDA cores' chunks (0: none)
}

la_status la_prefill_backward(const void* q, const void* k, const void* v, la_dtype in_dtype,
                              int B, int H, int N, int dk, int dv, float eps,
                              const float* S0, const float* z0, const float* dO,
                              const float* dS_N, const float* dz_N, float* dq, float* dk_out,
                              float* dv_out, float* dS0, float* dz0, void* workspace,
                              size_t ws_bytes, cudaStream_t stream) {
  if (!dtype_ok(in_dtype) || !dims_ok(B, H, N, dk, dv)) return LA_ERR_INVALID_ARG;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  if (N > 0 && (!q || !k || !v || !dO || !dq || !dk_out || !dv_out)) return LA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, S0, z0, dO, dS_N, dz_N, dq, dk_out, dv_out, dS0, dz0, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return LA_ERR_INVALID_ARG;
  if (workspace && ws_bytes < la_prefill_backward_workspace_bytes(B, H, N, dk, dv, in_dtype))
    return LA_ERR_INVALID_ARG;
  const size_t heads = (size_t)B * H;
  const size_t eb = elem_bytes(in_dtype);
  const Span ins[] = {span(q, heads * N * dk * eb), span(k, heads * N * dk * eb),
                      span(v, heads * N * dv * eb), span(S0, heads * dk * dv * 4),
                      span(z0, heads * dk * 4), span(dO, heads * N * dv * 4),
                      span(dS_N, heads * dk * dv * 4), span(dz_N, heads * dk * 4)};
  const Span outs[] = {span(dq, heads * N * dk * 4), span(dk_out, heads * N * dk * 4),
                       span(dv_out, heads * N * dv * 4), span(dS0, heads * dk * dv * 4),
                       span(dz0, heads * dk * 4)};
  for (const Span& x : outs) {
    for (const Span& y : ins)
      if (overlap(x, y)) return LA_ERR_INVALID_ARG;
    for (const Span& y : outs)
      if (&x != &y && overlap(x, y)) return LA_ERR_INVALID_ARG;
  }
  const Span sw = span(workspace, ws_bytes);
  for (const Span& x : ins)
    if (overlap(sw, x)) return LA_ERR_INVALID_ARG;
  for (const Span& x : outs)
    if (overlap(sw, x)) return LA_ERR_INVALID_ARG;
  const la_status dev = check_device();
  if (dev != LA_OK) return dev;
  if (N == 0) {
    cudaError_t e = cudaSuccess;
    if (dS0) e = copy_state(dS_N, dS0, heads * dk * dv * 4, stream);
    if (e == cudaSuccess && dz0) e = copy_state(dz_N, dz0, heads * dk * 4, stream);
    return from_cuda(e);
  }
  PrefillArgs a = {};
  a.q = q; a.k = k; a.v = v;
  a.bf16 = in_dtype == LA_BF16;
  a.B = B; a.H = H; a.N = N; a.dk = dk; a.dv = dv;
  a.eps = eps;
  a.S0 = S0; a.z0 = z0;
  a.o = nullptr; a.S_N = nullptr; a.z_N = nullptr;
  a.chunk = 0;
  a.workspace = workspace;
  a.ws_bytes = workspace ? ws_bytes : 0;
  if (la::backward_tc64_supported(a))
    return from_cuda(la::launch_backward_tc64(a, dO, dS_N, dz_N, dq, dk_out, dv_out, dS0, dz0, stream));
  return from_cuda(la::launch_prefill_backward(a, dO, dS_N, dz_N, dq, dk_out, dv_out, dS0, dz0,
                                               stream));
}

static la_status delta_common(const void* k, const void* v, la_dtype in_dtype,
                              const float* beta, const float* alpha, int B, int H, int N,
                              int dk, int dv, const float* S0, float* reads, float* S_N,
                              cudaStream_t stream) {
  if (!dtype_ok(in_dtype) || !dims_ok(B, H, N, dk, dv)) return LA_ERR_INVALID_ARG;
  if (!S_N) return LA_ERR_INVALID_ARG;
  if (N > 0 && (!k || !v || !beta || !reads)) return LA_ERR_INVALID_ARG;
  const void* ptrs[] = {k, v, beta, alpha, S0, reads, S_N};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return LA_ERR_INVALID_ARG;
  const size_t heads = (size_t)B * H;
  const size_t eb = elem_bytes(in_dtype);
  const Span sk = span(k, heads * N * dk * eb), sv = span(v, heads * N * dv * eb);
  const Span sb = span(beta, heads * N * 4), sa = span(alpha, heads * N * 4);
  const Span sr = span(reads, heads * N * dv * 4);
  const Span sS0 = span(S0, heads * dk * dv * 4), sSN = span(S_N, heads * dk * dv * 4);
  const Span outs[] = {sr, sSN};
  const Span ins[] = {sk, sv, sb, sa};
  for (const Span& x : outs)
    for (const Span& y : ins)
      if (overlap(x, y)) return LA_ERR_INVALID_ARG;
  if (overlap(sr, sSN) || overlap(sr, sS0)) return LA_ERR_INVALID_ARG;
  if (overlap(sSN, sS0) && S_N != S0) return LA_ERR_INVALID_ARG;
  const la_status dev = check_device();
  if (dev != LA_OK) return dev;
  if (N == 0) return from_cuda(copy_state(S0, S_N, heads * dk * dv * 4, stream));
  return from_cuda(la::launch_delta_prefill(k, v, in_dtype == LA_BF16, beta, alpha, B, H,
                                            N, dk, dv, S0, reads, S_N, stream));
}

la_status delta_prefill(const void* k, const void* v, la_dtype in_dtype, const float* beta,
                        int B, int H, int N, int dk, int dv, const float* S0,
                        float* reads, float* S_N, cudaStream_t stream) {
  return delta_common(k, v, in_dtype, beta, nullptr, B, H, N, dk, dv, S0, reads, S_N, stream);
}

la_status gated_delta_prefill(const void* k, const void* v, la_dtype in_dtype,
                              const float* beta, const float* alpha, int B, int H, int N,
                              int dk, int dv, const float* S0, float* reads, float* S_N,
                              cudaStream_t stream) {
  return delta_common(k, v, in_dtype, beta, alpha, B, H, N, dk, dv, S0, reads, S_N, stream);
}

la_status la_read_device_status(const void* workspace, cudaStream_t stream) {
  if (!workspace) return LA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return LA_ERR_CUDA;
  const la::WsHeader* h = reinterpret_cast<const la::WsHeader*>(workspace);
  unsigned status = 0;
  if (cudaMemcpy(&status, &h->status, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LA_ERR_CUDA;
  if (status != 0) {
    if (cudaMemset((void*)&h->status, 0, sizeof(status)) != cudaSuccess) return LA_ERR_CUDA;
  }
  return (status & la::kStatusTimeout) ? LA_ERR_TIMEOUT : LA_OK;
}

la_status delta_read_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return LA_ERR_CUDA;
  unsigned status = 0;
  if (la::delta_status_take(&status) != cudaSuccess) return LA_ERR_CUDA;
  if (status & la::kStatusLayout) return LA_ERR_UNSUPPORTED;
  return (status & la::kStatusTimeout) ? LA_ERR_TIMEOUT : LA_OK;
}

}  // extern "C"
