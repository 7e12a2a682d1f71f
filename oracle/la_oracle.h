/*
 * la_oracle.h -- fp64 CPU oracle for normalized causal linear attention
 * (ELU+1 feature map) and the delta-rule fast-weight memory.
 *
 * TEST INFRASTRUCTURE ONLY.  This header and la_oracle.c exist to check the
 * CUDA library against a plain, slow, obviously correct restatement of the
 * method.  Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark may load it.  The product library never links, includes or
 * calls anything in this directory, and this directory includes nothing from
 * the product library.
 *
 * Source of the definitions ("AIGC 基本功|线性、循环与记忆架构-LinearMem",
 * jefxiong.cn, abbreviated P1 below; "状态空间与线性注意力" (线性注意力与SSM),
 * ggaaooppeenngg.github.io, P3; "sequence-models" practice notes,
 * wineandchord.com, P5):
 *   phi(u) = u + 1 for u > 0, exp(u) for u <= 0             P1 section 03, "从检索权重开始"
 *   o_t = sum_{i<=t} (phi(q_t).phi(k_i)) v_i
 *         / (sum_{i<=t} phi(q_t).phi(k_i) + eps)            P1 section 03, "把历史和移到 query 外面"
 *   S_t = S_{t-1} + phi(k_t) v_t^T, z_t = z_{t-1} + phi(k_t),
 *   o_t^T = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps)         same section (write, then read)
 *   delta rule: read_t = k_t^T S_{t-1},
 *               S_t = S_{t-1} + beta_t k_t (v_t - read_t)^T P1 section 03, "从累加改成纠错";
 *                                                           P5, "Delta-rule fast weight"
 *
 * Layouts (all row-major, contiguous, double precision):
 *   q, k  [B][H][N][dk]     v, o, reads  [B][H][N][dv]
 *   S     [B][H][dk][dv]    (the "k v^T" convention: S[i][j] = sum phi(k)_i v_j)
 *   z     [B][H][dk]        beta [B][H][N]
 * S0 / z0 may be NULL, meaning a zero initial state.  nthreads <= 0 means
 * "one thread per available core"; work is split over the B*H heads only.
 * Every function returns 0 on success and -1 on an invalid argument.
 */
#ifndef LA_ORACLE_H
#define LA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* phi applied elementwise: out[i] = phi(u[i]). */
int orc_phi(const double* u, double* out, int64_t n);

/* Token-by-token recurrence, write before read (the primary oracle). */
int orc_la_recurrent(const double* q, const double* k, const double* v,
                     int B, int H, int N, int dk, int dv, double eps,
                     const double* S0, const double* z0,
                     double* o, double* S_N, double* z_N, int nthreads);

/* Quadratic masked form: explicit phi(Q) phi(K)^T weights with the causal
 * mask i <= t (diagonal included), plus the contribution of S0 / z0.
 * O(N^2) per head; meant for small N.  Does not produce a final state. */
int orc_la_quadratic(const double* q, const double* k, const double* v,
                     int B, int H, int N, int dk, int dv, double eps,
                     const double* S0, const double* z0,
                     double* o, int nthreads);

/* Chunkwise form with chunk length C >= 1 (C need not divide N): inside a
 * chunk the masked quadratic weights, across chunks only the state (S, z). */
int orc_la_chunked(const double* q, const double* k, const double* v,
                   int B, int H, int N, int dk, int dv, double eps,
                   const double* S0, const double* z0, int C,
                   double* o, double* S_N, double* z_N, int nthreads);

/* One decode step on every head: S += phi(k) v^T, z += phi(k), then
 * o = phi(q)^T S / (phi(q)^T z + eps).  q,k [B][H][dk], v,o [B][H][dv];
 * S and z are updated in place. */
int orc_la_decode_step(const double* q, const double* k, const double* v,
                       int B, int H, int dk, int dv, double eps,
                       double* S, double* z, double* o, int nthreads);

/* Delta-rule memory: reads[t] = k_t^T S_{t-1}, then
 * S_t = S_{t-1} + beta_t k_t (v_t - reads[t])^T.  No feature map, no
 * normalizer.  k [B][H][N][dk], v/reads [B][H][N][dv], beta [B][H][N]. */
int orc_delta(const double* k, const double* v, const double* beta,
              int B, int H, int N, int dk, int dv, const double* S0,
              double* reads, double* S_N, int nthreads);

/* Gated delta rule: D = alpha_t S_{t-1}; reads[t] = k_t^T D;
 * S_t = D + beta_t k_t (v_t - reads[t])^T.  alpha [B][H][N] or NULL (= 1). */
int orc_gated_delta(const double* k, const double* v, const double* beta,
                    const double* alpha, int B, int H, int N, int dk, int dv,
                    const double* S0, double* reads, double* S_N, int nthreads);

/* Variants of the recurrence: mode 0 write-then-read with a scalar decay of
 * the old (S, z) by alpha_t; mode 1 read-then-write (strictly past), same
 * decay; mode 2 non-causal (state over all tokens, then every query reads;
 * alpha must be NULL).  alpha [B][H][N] or NULL (= 1). */
int orc_la_variant(const double* q, const double* k, const double* v,
                   const double* alpha, int B, int H, int N, int dk, int dv,
                   double eps, int mode, const double* S0, const double* z0,
                   double* o, double* S_N, double* z_N, int nthreads);

/* The outputs of orc_la_variant from explicit (quadratic) weights. */
int orc_la_variant_quadratic(const double* q, const double* k, const double* v,
                             const double* alpha, int B, int H, int N, int dk,
                             int dv, double eps, int mode, const double* S0,
                             const double* z0, double* o, int nthreads);

/* Gradient of orc_la_recurrent with respect to q, k, v, S0, z0, given dO and
 * (optionally, NULL = 0) dS_N, dz_N; the states are recomputed.  dS0, dz0 may
 * be NULL. */
int orc_la_backward(const double* q, const double* k, const double* v, int B, int H,
                    int N, int dk, int dv, double eps, const double* S0,
                    const double* z0, const double* dO, const double* dS_N,
                    const double* dz_N, double* dq, double* dk_out, double* dv_out,
                    double* dS0, double* dz0, int nthreads);

/* Additive associative memory with the identity feature map (test-only
 * primitive): S = sum_m keys[m] values[m]^T, reads[p] = queries[p]^T S.
 * keys [M][dk], values [M][dv], queries [P][dk], reads [P][dv]. */
int orc_outer_read(const double* keys, const double* values, int M,
                   int dk, int dv, const double* queries, int P,
                   double* reads);

/* Number of worker threads that nthreads <= 0 resolves to. */
int orc_default_threads(void);

#ifdef __cplusplus
}
#endif

#endif /* LA_ORACLE_H */
