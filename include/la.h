/*
 * la.h -- C ABI of libla.so: normalized causal linear attention with the
 * ELU+1 feature map, and the delta-rule fast-weight memory, on one GB300
 * (sm_103a).
 *
 * Definitions (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03):
 *   phi(u) = u + 1 (u > 0), exp(u) (u <= 0), applied elementwise
 *   S_t = S_{t-1} + phi(k_t) v_t^T          (dk x dv, the "k v^T" layout)
 *   z_t = z_{t-1} + phi(k_t)                (dk)
 *   o_t^T = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps)      write, then read
 * Delta rule (same page, "从累加改成纠错"; page "sequence-models" practice
 * notes, "Delta-rule fast weight"):
 *   read_t = k_t^T S_{t-1};   S_t = S_{t-1} + beta_t k_t (v_t - read_t)^T
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layouts: row-major, contiguous, innermost dimension fastest.
 *   q, k        [B][H][N][dk]  (decode: [B][H][dk])   dtype in_dtype
 *   v           [B][H][N][dv]  (decode: [B][H][dv])   dtype in_dtype
 *   o, reads    [B][H][N][dv]  (decode: [B][H][dv])   float32
 *   S, S0, S_N  [B][H][dk][dv]                        float32, S[i][j] = sum phi(k)_i v_j
 *   z, z0, z_N  [B][H][dk]                            float32
 *   beta        [B][H][N]                             float32
 * Ownership: every tensor pointer is a DEVICE pointer owned by the caller.  The
 *   library allocates no device memory and keeps no per-call state; the only
 *   process-wide state is cached device attributes and kernel settings.
 * Alignment: every tensor pointer must be 16-byte aligned.
 * Sizes: B, H, dk, dv >= 1; dk, dv <= 128; N >= 0; B*H*N*max(dk,dv) < 2^40.
 *   N = 0 is valid: the final state is a copy of the initial state.
 * eps: finite and >= 0 (1e-6 in the pages' experiments).
 * Execution: every call is asynchronous on `stream` (NULL = legacy default
 *   stream).  The return value reports argument errors (LA_ERR_INVALID_ARG,
 *   LA_ERR_UNSUPPORTED, nothing launched) and launch errors (LA_ERR_CUDA).
 *   Errors a kernel detects while running (a bounded wait that gave up) are
 *   recorded in the workspace and read back with la_read_device_status.
 * Aliasing: outputs must not overlap inputs, except the state pairs named
 *   below (S_N may be S0, z_N may be z0).
 * Path choice: LA_BF16 inputs with dk = dv in {64, 128} run the tensor-core
 *   chunked kernel (tcgen05 MMA, TMEM accumulators, TMA loads); every other
 *   valid shape and LA_F32 inputs run the CUDA-core kernel.  Both run on the
 *   GPU; there is no CPU fallback.
 */
#ifndef LA_H
#define LA_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LA_OK = 0,
  LA_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment, aliasing or eps */
  LA_ERR_UNSUPPORTED = 2,  /* valid request the library cannot run here (e.g. no sm_103a device) */
  LA_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  LA_ERR_TIMEOUT = 4       /* a kernel's bounded inter-block wait gave up */
} la_status;

typedef enum { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

/* Read order of la_prefill_variant. */
typedef enum {
  LA_MODE_CAUSAL = 0,             /* write, then read (la_prefill's order) */
  LA_MODE_READ_BEFORE_WRITE = 1,  /* read, then write: strictly past */
  LA_MODE_NONCAUSAL = 2           /* the state over all N tokens, then every read */
} la_mode;

/*
 * la_prefill -- causal prefill of N tokens per (batch, head).
 * Computes o_t for t = 1..N from the recurrence above, starting from S0, z0
 * (NULL = zero state: the LinearMem page, section 05, resets the state per
 * request), and writes the final state S_N, z_N (the same page's appendix
 * script returns the outputs together with S and z).
 *   q, k, v     inputs, in_dtype (LA_F32 or LA_BF16)
 *   S0, z0      initial state or NULL; S_N may alias S0, z_N may alias z0
 *   o, S_N, z_N outputs, float32
 *   chunk       chunk length of the tensor-core path; 0 = automatic (128).
 *               The CUDA-core path (LA_F32, or dk, dv outside the
 *               tensor-core sizes) picks its own chunks: with the workspace
 *               la_prefill_workspace_bytes asks for, each head's sequence is
 *               cut into up to 64 chunks run in parallel (their increments,
 *               a scan of the states between them in chunk order, their
 *               outputs, all in fp32).
 *   workspace   device scratch of at least la_prefill_workspace_bytes(...)
 *               bytes.  Its first 256 bytes hold the device status word and
 *               must be zero before the workspace's first use (one
 *               cudaMemset after allocating it; la_read_device_status clears
 *               the word again); the rest need not be initialised, as every
 *               call writes what it reads.  Calls that share a workspace must
 *               be ordered on one stream.
 */
la_status la_prefill(const void* q, const void* k, const void* v, la_dtype in_dtype,
                     int B, int H, int N, int dk, int dv, float eps,
                     const float* S0, const float* z0,
                     float* o, float* S_N, float* z_N,
                     int chunk, void* workspace, size_t ws_bytes,
                     cudaStream_t stream);

/*
 * la_prefill_variant -- la_prefill's recurrence with a per-token decay of the
 * old state and a choice of read order:
 *   S_t = alpha_t S_{t-1} + phi(k_t) v_t^T,   z_t = alpha_t z_{t-1} + phi(k_t)
 * (the linear-attention recurrence with one scalar on the old state: page
 * "线性注意力与SSM", sections 3-4, Mamba-2; the normalizer decays with S), and
 *   LA_MODE_CAUSAL:            o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps)
 *   LA_MODE_READ_BEFORE_WRITE: o_t = phi(q_t)^T S_{t-1} / (phi(q_t)^T z_{t-1} + eps)
 *       (LinearMem sections 03 and 09: strictly past; from a zero state the
 *       first read is 0)
 *   LA_MODE_NONCAUSAL:         o_t = phi(q_t)^T S_N / (phi(q_t)^T z_N + eps), with
 *       S_N = S0 + sum_t phi(k_t) v_t^T (the linear-attention explainer,
 *       section 线性化核心; eps = 0 gives its form exactly).
 *   alpha   [B][H][N] float32, or NULL for no decay (then LA_MODE_CAUSAL is
 *           la_prefill exactly).  Must be NULL for LA_MODE_NONCAUSAL.
 *   workspace  device scratch of at least la_prefill_variant_workspace_bytes(...)
 *              bytes, or NULL; its contents need not be initialised.  Calls
 *              that share a workspace must be ordered on one stream.
 * Other arguments, layouts, aliasing and errors as la_prefill (a workspace
 * smaller than asked for, or overlapping another argument, is
 * LA_ERR_INVALID_ARG).  LA_BF16 at dk = dv = 64 with a decay in
 * LA_MODE_CAUSAL runs on the tensor cores with 128-token chunks and the decay
 * factors inside each chunk (the state enters the products as a bf16 copy of
 * the fp32 state; a zero alpha_t is taken as 1e-30): with a workspace, the
 * heads are split over every SM -- for calls of at most 2048 chunks of 128
 * tokens two launches (decayed prefix tiles, piece totals and decays, then
 * the outputs, each block folding its entry state from the earlier totals),
 * for larger ones three (decayed piece totals, the chained scan
 * E' = Gamma E + R, then the outputs); with NULL, one block per head.
 * LA_BF16 at dk = dv = 128 with a decay in LA_MODE_CAUSAL and a workspace
 * runs the same three launches on the tensor cores at that width.  With a
 * decay in LA_MODE_READ_BEFORE_WRITE, LA_BF16 at dk = dv = 64 (any
 * workspace, or none) and at 128 (with one) runs the three-launch forms (at
 * 64 without a workspace, one block per head) with a strict mask, each token
 * reading S_{t-1}.
 * LA_BF16 at dk = dv = 64 or 128 without a decay, with a workspace, also
 * runs on the tensor cores: LA_MODE_READ_BEFORE_WRITE as la_prefill's
 * launches with a strict mask inside each chunk; LA_MODE_NONCAUSAL as the
 * totals of the heads' pieces (la_prefill's first launch at dk = 64 for calls
 * of at most 2048 chunks of 128 tokens, else the aggregate launch of its
 * three-launch form), one fold per head into S_N, z_N and a bf16 copy of that
 * state (z as hi + lo), then every query reads it (one product per chunk).  A
 * bounded wait of those kernels that gives up is reported by
 * delta_read_device_status.  Everything else runs on the CUDA cores in fp32,
 * for LA_F32 and LA_BF16 inputs and any dk, dv <= 128: with a workspace of
 * la_prefill_variant_workspace_bytes, each head's sequence in up to 64
 * chunks run in parallel (as la_prefill's CUDA-core path; the chunks' decayed
 * increments and total decays chained as E' = gamma E + R); with NULL, one
 * block per head, token by token.
 */
la_status la_prefill_variant(const void* q, const void* k, const void* v, la_dtype in_dtype,
                             int B, int H, int N, int dk, int dv, float eps,
                             const float* alpha, la_mode mode,
                             const float* S0, const float* z0,
                             float* o, float* S_N, float* z_N,
                             void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Bytes of workspace la_prefill_variant uses for these arguments (decay:
 * nonzero when alpha is given); 0 when it uses none, or for invalid
 * arguments.  The figure of the tensor-core decayed form depends on the SM
 * count of the current device. */
size_t la_prefill_variant_workspace_bytes(int B, int H, int N, int dk, int dv,
                                          la_dtype in_dtype, la_mode mode, int decay);

/*
 * la_prefill_backward -- the gradient of la_prefill's map
 *   (q, k, v, S0, z0) -> (o, S_N, z_N)
 * given dO [B][H][N][dv] and dS_N [B][H][dk][dv], dz_N [B][H][dk] (NULL = zero).
 * The pages give no backward pass; the LinearMem page (section 03) notes only
 * that training must not keep every state and that recomputation handles it.
 * This recomputes the states: a forward sweep gives
 *   dnum_t = dO_t / den_t,  dden_t = -(dO_t . o_t) / den_t,  dq via
 *   dphi(q_t) = S_t dnum_t + dden_t z_t,
 * and a reverse sweep accumulates G_t = dS_N + sum_{tau >= t} phi(q_tau) dnum_tau^T
 * and g_t = dz_N + sum_{tau >= t} dden_tau phi(q_tau) for
 *   dphi(k_t) = G_t v_t + g_t,  dv_t = G_t^T phi(k_t),  dS0 = G_0,  dz0 = g_0,
 * with dq = dphi(q) phi'(q), dk = dphi(k) phi'(k), phi'(u) = 1 (u > 0), exp(u) (u <= 0).
 *   dq, dk_out [B][H][N][dk], dv_out [B][H][N][dv]: float32 outputs (the
 *               gradients with respect to q, k and v)
 *   dS0 [B][H][dk][dv], dz0 [B][H][dk]: float32 outputs, or NULL if not wanted
 *   workspace  device scratch of at least la_prefill_backward_workspace_bytes(...)
 *              bytes, or NULL; its contents need not be initialised.  Calls
 *              that share a workspace must be ordered on one stream.
 * Outputs must not overlap any input, each other or the workspace (a
 * workspace smaller than asked for is LA_ERR_INVALID_ARG).  LA_BF16 at
 * dk = dv = 64 runs on the tensor cores (bf16 operands, fp32 accumulation),
 * the heads cut into pieces over every SM when a workspace is given: calls of
 * at most 2048 chunks of 128 tokens (B * H * ceil(N / 128)) take every chunk
 * independently from per-chunk state tiles (four launches: the prefill's
 * prefix tiles and outputs, the gradient-state tiles, then dq, dk, dv), larger
 * ones a forward and a reverse sweep over each piece (the prefill's own
 * aggregate and scan give each piece its entry state, a reverse scan its
 * gradient state; dv_out holds bf16 intermediate rows between the sweeps).
 * With NULL, one block per head, both sweeps.  A bounded wait of those kernels
 * that gives up is reported by delta_read_device_status.  Everything else runs
 * on the CUDA cores in fp32, any dk, dv <= 128: with a workspace, each head
 * cut into chunks run in parallel (the state before every chunk from the
 * CUDA-core prefill's first two launches, a forward sweep per chunk, each
 * chunk's gradient-state increment, a reverse scan per head, a reverse sweep
 * per chunk); with NULL, one block per head, token by token.
 */
la_status la_prefill_backward(const void* q, const void* k, const void* v, la_dtype in_dtype,
                              int B, int H, int N, int dk, int dv, float eps,
                              const float* S0, const float* z0, const float* dO,
                              const float* dS_N, const float* dz_N,
                              float* dq, float* dk_out, float* dv_out, float* dS0, float* dz0,
                              void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Bytes of workspace la_prefill_backward uses for these arguments; 0 when it
 * uses none, or for invalid arguments.  The figure depends on the SM count of
 * the current device. */
size_t la_prefill_backward_workspace_bytes(int B, int H, int N, int dk, int dv, la_dtype in_dtype);

/* Bytes of workspace la_prefill needs for these arguments (always >= 256).
 * Returns 0 for arguments la_prefill would reject. */
size_t la_prefill_workspace_bytes(int B, int H, int N, int dk, int dv,
                                  la_dtype in_dtype, int chunk);

/*
 * la_decode_step -- one token per (batch, head) on a resident state, in place:
 *   S += phi(k) v^T;  z += phi(k);  o = phi(q)^T S / (phi(q)^T z + eps)
 * (update, then read: LinearMem page, section 03).  S and z are read once
 * and written once.
 *   q, k [B][H][dk], v [B][H][dv] in in_dtype;  o [B][H][dv] float32.
 */
la_status la_decode_step(const void* q, const void* k, const void* v, la_dtype in_dtype,
                         int B, int H, int dk, int dv, float eps,
                         float* S, float* z, float* o, cudaStream_t stream);

/*
 * delta_prefill -- the delta-rule memory over N tokens per (batch, head):
 *   reads[t] = k_t^T S_{t-1};  S_t = S_{t-1} + beta_t k_t (v_t - reads[t])^T
 * (prediction first, then the error write: "sequence-models" practice notes,
 * delta_memory).  No feature map, no normalizer, no eps.
 *   k [B][H][N][dk], v [B][H][N][dv] in in_dtype;  beta [B][H][N] float32
 *   S0 initial memory or NULL (zero); S_N may alias S0
 *   reads [B][H][N][dv], S_N [B][H][dk][dv] float32
 * bf16 inputs at dk = dv = 64, 96 or 128 run chunkwise on the tensor cores
 * (64-token chunks; the state enters the products as a bf16 copy of the fp32
 * state; widths below 128 run the width-128 kernel with the columns past dk
 * zero, so they take about as long); other inputs run token by token in fp32.  A bounded wait of the chunkwise
 * kernel that gives up is reported by delta_read_device_status.
 */
la_status delta_prefill(const void* k, const void* v, la_dtype in_dtype, const float* beta,
                        int B, int H, int N, int dk, int dv,
                        const float* S0, float* reads, float* S_N,
                        cudaStream_t stream);

/*
 * gated_delta_prefill -- the delta rule with forgetting (LinearMem section 03,
 * the forgetting factor alpha_t, and the appendix delta_step): per token the old
 * memory decays first, then the correction uses the decayed prediction:
 *   D = alpha_t S_{t-1};  reads[t] = k_t^T D;  S_t = D + beta_t k_t (v_t - reads[t])^T
 *   alpha [B][H][N] float32, or NULL (alpha_t = 1: exactly delta_prefill).
 * Other arguments as delta_prefill.  bf16 inputs at dk = dv = 64, 96 or 128
 * run chunkwise on the tensor cores (decay factors inside each 64-token chunk,
 * status through delta_read_device_status); everything else runs token by
 * token in fp32 on the CUDA cores.
 */
la_status gated_delta_prefill(const void* k, const void* v, la_dtype in_dtype,
                              const float* beta, const float* alpha,
                              int B, int H, int N, int dk, int dv,
                              const float* S0, float* reads, float* S_N,
                              cudaStream_t stream);

/* Bytes of one head's recurrent state, (dk*dv + dk) * 4: 16640 at 64 x 64
 * (LinearMem page, section 01).  0 for dk or dv < 1. */
size_t la_state_bytes(int dk, int dv);

/* Static, human-readable name of a status code. */
const char* la_status_string(la_status s);

/* Synchronizes `stream`, then returns and clears the status word that kernels
 * record in `workspace` (LA_ERR_TIMEOUT if a bounded wait gave up since the
 * last read, otherwise LA_OK).  LA_ERR_INVALID_ARG for a NULL workspace,
 * LA_ERR_CUDA if the synchronization or copy fails. */
la_status la_read_device_status(const void* workspace, cudaStream_t stream);

/* Synchronizes `stream`, then returns and clears the status word of the
 * tensor-core kernels whose calls take no workspace: delta_prefill and
 * gated_delta_prefill with bf16 inputs at dk = dv = 64, 96 or 128, the
 * tensor-core forms of la_prefill_variant and la_prefill_backward on bf16
 * inputs (also
 * when they are given a workspace), and la_prefill_noalloc.  LA_ERR_TIMEOUT if one of their
 * bounded waits gave up since the last read, otherwise LA_OK; LA_ERR_CUDA if
 * the synchronization or copy fails.  The word belongs to the current device
 * and is shared by every such call on it; the token-by-token kernels have no
 * waits and never set it.  LA_ERR_UNSUPPORTED if a launch found its
 * shared-memory window misaligned and did no work. */
la_status delta_read_device_status(cudaStream_t stream);

/*
 * la_prefill_noalloc -- la_prefill without a caller-provided workspace.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory -- code that runs while a CUDA graph is being
 * captured, plugins whose host framework only hands out input and output
 * buffers, or processes whose device memory belongs to another allocator.
 * It computes exactly what la_prefill computes, with the same arguments
 * minus the workspace, and allocates nothing: its scratch is one fixed 16 MiB
 * array inside this library's device image, which every GPU that loads the
 * library holds until the process exits.
 *   Limit: requests whose la_prefill_workspace_bytes(...) exceeds 16 MiB
 *   (16777216 bytes) are rejected with LA_ERR_INVALID_ARG, as are arguments
 *   la_prefill rejects.  At dk = dv = 64 the workspace is a bf16 copy of
 *   phi(K) (128 bytes per token), an 8.4 KB prefix tile per 128-token chunk
 *   and a 16.6 KB state slot per pair of head and block that meet: 8 heads of
 *   4096 tokens fit (10.3 MiB on a 152-SM GPU), 16 heads of 4096 just fit
 *   (15.2 MiB), 32 do not; past 2048 chunks (heads x chunks) the d = 64
 *   form keeps only two state slots per (head, block) pair, so 64 heads of
 *   65536 tokens take 8.1 MiB; at dk = dv = 128 the workspace is two arrays
 *   of 66 KB slots, one per (head, block) pair: 4 heads of 2048 tokens fit
 *   (8.6 MiB), 8 do not.  The CUDA-core path's chunk slots take
 *   (dk dv + dk + 1) * 4 bytes per chunk (1.2 MiB for 2 heads of 300 tokens
 *   at d = 64).  la_prefill_workspace_bytes gives the figure.
 *   Set-up: the first call on each device (with that device current) looks up
 *   the device addresses of the array and of the library's status word; it
 *   issues no device work, and concurrent first calls from several host
 *   threads are safe.  Make that first call before any stream capture.
 *   Contents: the array needs no initialisation; every call writes what it
 *   reads, and it keeps the last call's contents.
 *   Sharing: every call on a device uses the same array; calls whose
 *   executions overlap on the GPU (different streams, no ordering) race on it
 *   and must not be issued.
 *   Status: a bounded wait that gave up is recorded in the library status
 *   word, read back and cleared by delta_read_device_status.
 */
la_status la_prefill_noalloc(const void* q, const void* k, const void* v, la_dtype in_dtype,
                             int B, int H, int N, int dk, int dv, float eps,
                             const float* S0, const float* z0,
                             float* o, float* S_N, float* z_N,
                             int chunk, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LA_H */
