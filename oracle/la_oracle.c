/*
 * la_oracle.c -- plain fp64 restatement of normalized causal linear attention
 * (ELU+1 feature map) and of the delta-rule memory.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product library.  It shares no
 * code, header or constant with the CUDA path.  Every function is written to
 * be checked against the pages by eye: no blocking, fusion or reordering
 * beyond what the cited definition states.  Threads split the independent
 * (batch, head) pairs and nothing else.
 *
 * Citations (page title, section):
 *   P1 = "AIGC 基本功|线性、循环与记忆架构-LinearMem" (jefxiong.cn)
 *   P2 = linear-attention explainer (aiqz.cc), section 线性化核心 and its listing
 *   P3 = "线性注意力与SSM" (ggaaooppeenngg.github.io)
 *   P5 = "sequence-models" practice notes (wineandchord.com)
 */
#define _GNU_SOURCE
#include "la_oracle.h"

#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Feature map.  P1 section 03 "从检索权重开始": phi(u) = u + 1 when u > 0 and
 * exp(u) when u <= 0 (so phi(0) = 1, continuous, always positive). */
static double phi(double u) { return u > 0.0 ? u + 1.0 : exp(u); }

int orc_phi(const double* u, double* out, int64_t n) {
  if (n < 0 || (n > 0 && (!u || !out))) return -1;
  for (int64_t i = 0; i < n; ++i) out[i] = phi(u[i]);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Work split over heads.  Each job gets a contiguous range of head indices. */
typedef void (*head_fn)(void* ctx, int64_t head);

typedef struct {
  head_fn fn;
  void* ctx;
  int64_t begin, end;
} range_job;

static void* run_range(void* p) {
  range_job* j = (range_job*)p;
  for (int64_t h = j->begin; h < j->end; ++h) j->fn(j->ctx, h);
  return NULL;
}

int orc_default_threads(void) {
  cpu_set_t set;
  CPU_ZERO(&set);
  if (sched_getaffinity(0, sizeof(set), &set) == 0) {
    int c = CPU_COUNT(&set);
    if (c > 0) return c;
  }
  return 1;
}

static void for_each_head(int64_t nheads, int nthreads, head_fn fn, void* ctx) {
  if (nthreads <= 0) nthreads = orc_default_threads();
  if (nthreads > nheads) nthreads = (int)nheads;
  if (nthreads <= 1) {
    for (int64_t h = 0; h < nheads; ++h) fn(ctx, h);
    return;
  }
  pthread_t* tid = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
  range_job* jobs = (range_job*)malloc(sizeof(range_job) * nthreads);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].begin = nheads * t / nthreads;
    jobs[t].end = nheads * (t + 1) / nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tid[t], NULL, run_range, &jobs[t]) != 0) break;
    started = t;
  }
  run_range(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
  /* any range whose thread could not be created runs here */
  for (int t = started + 1; t < nthreads; ++t) run_range(&jobs[t]);
  free(jobs);
  free(tid);
}

/* Common argument bundle for the linear-attention forms. */
typedef struct {
  const double *q, *k, *v, *S0, *z0;
  int N, dk, dv, C;
  double eps;
  double *o, *S_N, *z_N;
} la_args;

static int la_check(const double* q, const double* k, const double* v, int B,
                    int H, int N, int dk, int dv, double eps, const double* o) {
  if (B < 1 || H < 1 || N < 0 || dk < 1 || dv < 1 || !(eps >= 0.0)) return -1;
  if (N > 0 && (!q || !k || !v || !o)) return -1;
  return 0;
}

/* ------------------------------------------------------------------------ */
/* (1) Recurrence, P1 section 03: S_0 = 0, z_0 = 0 (here: S0, z0), and for each
 * token first write  S_t = S_{t-1} + phi(k_t) v_t^T,  z_t = z_{t-1} + phi(k_t),
 * then read  o_t^T = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps).
 * Returns o, and the final S and z (P1 appendix: recurrent_linear returns
 * out, S, z). */
static void recurrent_head(void* p, int64_t h) {
  const la_args* a = (const la_args*)p;
  const int N = a->N, dk = a->dk, dv = a->dv;
  double* S = a->S_N + h * (int64_t)dk * dv;
  double* z = a->z_N + h * (int64_t)dk;
  if (a->S0) memcpy(S, a->S0 + h * (int64_t)dk * dv, sizeof(double) * dk * dv);
  else memset(S, 0, sizeof(double) * dk * dv);
  if (a->z0) memcpy(z, a->z0 + h * (int64_t)dk, sizeof(double) * dk);
  else memset(z, 0, sizeof(double) * dk);

  double* fk = (double*)malloc(sizeof(double) * dk);
  double* fq = (double*)malloc(sizeof(double) * dk);
  for (int t = 0; t < N; ++t) {
    const double* qt = a->q + (h * (int64_t)N + t) * dk;
    const double* kt = a->k + (h * (int64_t)N + t) * dk;
    const double* vt = a->v + (h * (int64_t)N + t) * dv;
    double* ot = a->o + (h * (int64_t)N + t) * dv;
    for (int i = 0; i < dk; ++i) fk[i] = phi(kt[i]);
    for (int i = 0; i < dk; ++i) fq[i] = phi(qt[i]);
    /* write */
    for (int i = 0; i < dk; ++i) {
      for (int j = 0; j < dv; ++j) S[i * dv + j] += fk[i] * vt[j];
      z[i] += fk[i];
    }
    /* read */
    double den = 0.0;
    for (int i = 0; i < dk; ++i) den += fq[i] * z[i];
    den += a->eps;
    for (int j = 0; j < dv; ++j) {
      double num = 0.0;
      for (int i = 0; i < dk; ++i) num += fq[i] * S[i * dv + j];
      ot[j] = num / den;
    }
  }
  free(fk);
  free(fq);
}

int orc_la_recurrent(const double* q, const double* k, const double* v, int B,
                     int H, int N, int dk, int dv, double eps, const double* S0,
                     const double* z0, double* o, double* S_N, double* z_N,
                     int nthreads) {
  if (la_check(q, k, v, B, H, N, dk, dv, eps, o) || !S_N || !z_N) return -1;
  la_args a = {q, k, v, S0, z0, N, dk, dv, 0, eps, o, S_N, z_N};
  for_each_head((int64_t)B * H, nthreads, recurrent_head, &a);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* (2) Quadratic masked form, P1 section 03 (the normalized sum over i <= t)
 * and P1 appendix explicit_linear: W = phi(Q) phi(K)^T with everything above
 * the diagonal removed, o = W V / (row sums of W + eps).  Extended with a
 * nonzero initial state: S0 / z0 add phi(q_t)^T S0 to the numerator and
 * phi(q_t)^T z0 to the denominator, which is what the recurrence gives when it
 * starts from S0, z0. */
static void quadratic_head(void* p, int64_t h) {
  const la_args* a = (const la_args*)p;
  const int N = a->N, dk = a->dk, dv = a->dv;
  const double* S0 = a->S0 ? a->S0 + h * (int64_t)dk * dv : NULL;
  const double* z0 = a->z0 ? a->z0 + h * (int64_t)dk : NULL;
  double* fq = (double*)malloc(sizeof(double) * dk);
  double* fk = (double*)malloc(sizeof(double) * dk);
  double* num = (double*)malloc(sizeof(double) * dv);
  for (int t = 0; t < N; ++t) {
    const double* qt = a->q + (h * (int64_t)N + t) * dk;
    for (int r = 0; r < dk; ++r) fq[r] = phi(qt[r]);
    double den = 0.0;
    for (int j = 0; j < dv; ++j) num[j] = 0.0;
    if (S0)
      for (int r = 0; r < dk; ++r)
        for (int j = 0; j < dv; ++j) num[j] += fq[r] * S0[r * dv + j];
    if (z0)
      for (int r = 0; r < dk; ++r) den += fq[r] * z0[r];
    for (int i = 0; i <= t; ++i) { /* causal mask: i <= t, diagonal kept */
      const double* ki = a->k + (h * (int64_t)N + i) * dk;
      const double* vi = a->v + (h * (int64_t)N + i) * dv;
      for (int r = 0; r < dk; ++r) fk[r] = phi(ki[r]);
      double w = 0.0;
      for (int r = 0; r < dk; ++r) w += fq[r] * fk[r];
      den += w;
      for (int j = 0; j < dv; ++j) num[j] += w * vi[j];
    }
    den += a->eps;
    double* ot = a->o + (h * (int64_t)N + t) * dv;
    for (int j = 0; j < dv; ++j) ot[j] = num[j] / den;
  }
  free(fq);
  free(fk);
  free(num);
}

int orc_la_quadratic(const double* q, const double* k, const double* v, int B,
                     int H, int N, int dk, int dv, double eps, const double* S0,
                     const double* z0, double* o, int nthreads) {
  if (la_check(q, k, v, B, H, N, dk, dv, eps, o)) return -1;
  la_args a = {q, k, v, S0, z0, N, dk, dv, 0, eps, o, NULL, NULL};
  for_each_head((int64_t)B * H, nthreads, quadratic_head, &a);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* (3) Chunkwise form.  P3 section 3 (Mamba-2 / SSD paragraph): inside a chunk
 * a small masked phi(Q)phi(K)^T attention, across chunks a recurrence; P5
 * "Chunked scan": chunks hand over only the final state.  For a chunk
 * [c0, c1) with incoming state (S_prev, z_prev):
 *   num_t = phi(q_t)^T S_prev + sum_{c0 <= i <= t} (phi(q_t).phi(k_i)) v_i
 *   den_t = phi(q_t)^T z_prev + sum_{c0 <= i <= t}  phi(q_t).phi(k_i) + eps
 *   o_t = num_t / den_t
 * and afterwards S_prev += sum_{i in chunk} phi(k_i) v_i^T,
 * z_prev += sum_{i in chunk} phi(k_i). */
static void chunked_head(void* p, int64_t h) {
  const la_args* a = (const la_args*)p;
  const int N = a->N, dk = a->dk, dv = a->dv, C = a->C;
  double* S = a->S_N + h * (int64_t)dk * dv;
  double* z = a->z_N + h * (int64_t)dk;
  if (a->S0) memcpy(S, a->S0 + h * (int64_t)dk * dv, sizeof(double) * dk * dv);
  else memset(S, 0, sizeof(double) * dk * dv);
  if (a->z0) memcpy(z, a->z0 + h * (int64_t)dk, sizeof(double) * dk);
  else memset(z, 0, sizeof(double) * dk);

  double* fq = (double*)malloc(sizeof(double) * (size_t)C * dk);
  double* fk = (double*)malloc(sizeof(double) * (size_t)C * dk);
  for (int c0 = 0; c0 < N; c0 += C) {
    const int c1 = (c0 + C < N) ? c0 + C : N;
    const int n = c1 - c0;
    for (int t = 0; t < n; ++t)
      for (int r = 0; r < dk; ++r) {
        fq[t * dk + r] = phi(a->q[(h * (int64_t)N + c0 + t) * dk + r]);
        fk[t * dk + r] = phi(a->k[(h * (int64_t)N + c0 + t) * dk + r]);
      }
    /* outputs of the chunk, read against the incoming state */
    for (int t = 0; t < n; ++t) {
      double* ot = a->o + (h * (int64_t)N + c0 + t) * dv;
      double den = 0.0;
      for (int r = 0; r < dk; ++r) den += fq[t * dk + r] * z[r];
      for (int j = 0; j < dv; ++j) {
        double s = 0.0;
        for (int r = 0; r < dk; ++r) s += fq[t * dk + r] * S[r * dv + j];
        ot[j] = s;
      }
      for (int i = 0; i <= t; ++i) {
        const double* vi = a->v + (h * (int64_t)N + c0 + i) * dv;
        double w = 0.0;
        for (int r = 0; r < dk; ++r) w += fq[t * dk + r] * fk[i * dk + r];
        den += w;
        for (int j = 0; j < dv; ++j) ot[j] += w * vi[j];
      }
      den += a->eps;
      for (int j = 0; j < dv; ++j) ot[j] /= den;
    }
    /* hand the chunk's contribution to the state */
    for (int i = 0; i < n; ++i) {
      const double* vi = a->v + (h * (int64_t)N + c0 + i) * dv;
      for (int r = 0; r < dk; ++r) {
        for (int j = 0; j < dv; ++j) S[r * dv + j] += fk[i * dk + r] * vi[j];
        z[r] += fk[i * dk + r];
      }
    }
  }
  free(fq);
  free(fk);
}

int orc_la_chunked(const double* q, const double* k, const double* v, int B,
                   int H, int N, int dk, int dv, double eps, const double* S0,
                   const double* z0, int C, double* o, double* S_N, double* z_N,
                   int nthreads) {
  if (la_check(q, k, v, B, H, N, dk, dv, eps, o) || C < 1 || !S_N || !z_N)
    return -1;
  la_args a = {q, k, v, S0, z0, N, dk, dv, C, eps, o, S_N, z_N};
  for_each_head((int64_t)B * H, nthreads, chunked_head, &a);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* (4) One decode step: one iteration of the recurrence (1) on a given state,
 * P1 section 03 (write the current token, then read it with the current
 * query). */
typedef struct {
  const double *q, *k, *v;
  int dk, dv;
  double eps;
  double *S, *z, *o;
} decode_args;

static void decode_head(void* p, int64_t h) {
  const decode_args* a = (const decode_args*)p;
  const int dk = a->dk, dv = a->dv;
  const double* qh = a->q + h * dk;
  const double* kh = a->k + h * dk;
  const double* vh = a->v + h * dv;
  double* Sh = a->S + h * (int64_t)dk * dv;
  double* zh = a->z + h * dk;
  double* oh = a->o + h * dv;
  /* write */
  for (int i = 0; i < dk; ++i) {
    const double fk = phi(kh[i]);
    for (int j = 0; j < dv; ++j) Sh[i * dv + j] += fk * vh[j];
    zh[i] += fk;
  }
  /* read */
  double den = 0.0;
  for (int i = 0; i < dk; ++i) den += phi(qh[i]) * zh[i];
  den += a->eps;
  for (int j = 0; j < dv; ++j) {
    double num = 0.0;
    for (int i = 0; i < dk; ++i) num += phi(qh[i]) * Sh[i * dv + j];
    oh[j] = num / den;
  }
}

int orc_la_decode_step(const double* q, const double* k, const double* v,
                       int B, int H, int dk, int dv, double eps, double* S,
                       double* z, double* o, int nthreads) {
  if (B < 1 || H < 1 || dk < 1 || dv < 1 || !(eps >= 0.0)) return -1;
  if (!q || !k || !v || !S || !z || !o) return -1;
  decode_args a = {q, k, v, dk, dv, eps, S, z, o};
  for_each_head((int64_t)B * H, nthreads, decode_head, &a);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* (5) Delta rule.  P1 section 03 "从累加改成纠错" (one gradient step on
 * 1/2 ||S^T k_t - v_t||^2 with step beta_t), P1 appendix delta_step with
 * alpha = 1, and P5 "Delta-rule fast weight" (read the prediction first, then
 * write the error):
 *   reads_t = k_t^T S_{t-1}
 *   S_t     = S_{t-1} + beta_t k_t (v_t - reads_t)^T
 * There is no feature map, normalizer or eps. */
typedef struct {
  const double *k, *v, *beta, *S0;
  int N, dk, dv;
  double *reads, *S_N;
} delta_args;

static void delta_head(void* p, int64_t h) {
  const delta_args* a = (const delta_args*)p;
  const int N = a->N, dk = a->dk, dv = a->dv;
  double* S = a->S_N + h * (int64_t)dk * dv;
  if (a->S0) memcpy(S, a->S0 + h * (int64_t)dk * dv, sizeof(double) * dk * dv);
  else memset(S, 0, sizeof(double) * dk * dv);
  double* err = (double*)malloc(sizeof(double) * dv);
  for (int t = 0; t < N; ++t) {
    const double* kt = a->k + (h * (int64_t)N + t) * dk;
    const double* vt = a->v + (h * (int64_t)N + t) * dv;
    const double bt = a->beta[h * (int64_t)N + t];
    double* rt = a->reads + (h * (int64_t)N + t) * dv;
    for (int j = 0; j < dv; ++j) {
      double r = 0.0;
      for (int i = 0; i < dk; ++i) r += kt[i] * S[i * dv + j];
      rt[j] = r;
      err[j] = vt[j] - r;
    }
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[i * dv + j] += bt * kt[i] * err[j];
  }
  free(err);
}

int orc_delta(const double* k, const double* v, const double* beta, int B,
              int H, int N, int dk, int dv, const double* S0, double* reads,
              double* S_N, int nthreads) {
  if (B < 1 || H < 1 || N < 0 || dk < 1 || dv < 1 || !S_N) return -1;
  if (N > 0 && (!k || !v || !beta || !reads)) return -1;
  delta_args a = {k, v, beta, S0, N, dk, dv, reads, S_N};
  for_each_head((int64_t)B * H, nthreads, delta_head, &a);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* (7) Gated delta rule, P1 section 03 (the forgetting factor alpha_t), the same
 * page's appendix delta_step(S, k, v, beta, alpha): first decay the old state,
 * then correct against the decayed prediction:
 *   D = alpha_t S_{t-1};  reads[t] = k_t^T D;  S_t = D + beta_t k_t (v_t - reads[t])^T.
 * alpha = NULL means alpha_t = 1 (the plain delta rule of (5)).  The reported
 * read is the prediction the correction uses, k_t^T D. */
typedef struct {
  const double *k, *v, *beta, *alpha, *S0;
  int N, dk, dv;
  double *reads, *S_N;
} gdelta_args;

static void gated_delta_head(void* p, int64_t h) {
  const gdelta_args* a = (const gdelta_args*)p;
  const int N = a->N, dk = a->dk, dv = a->dv;
  double* S = a->S_N + h * (int64_t)dk * dv;
  if (a->S0) memcpy(S, a->S0 + h * (int64_t)dk * dv, sizeof(double) * dk * dv);
  else memset(S, 0, sizeof(double) * dk * dv);
  double* corr = (double*)malloc(sizeof(double) * dv);
  for (int t = 0; t < N; ++t) {
    const double* key = a->k + (h * (int64_t)N + t) * dk;
    const double* val = a->v + (h * (int64_t)N + t) * dv;
    const double write_rate = a->beta[h * (int64_t)N + t];
    const double forget = a->alpha ? a->alpha[h * (int64_t)N + t] : 1.0;
    double* pred = a->reads + (h * (int64_t)N + t) * dv;
    /* decay: D = alpha_t S */
    for (int e = 0; e < dk * dv; ++e) S[e] *= forget;
    /* prediction from the decayed state, and the correction v - k^T D */
    for (int j = 0; j < dv; ++j) {
      double kd = 0.0;
      for (int i = 0; i < dk; ++i) kd += key[i] * S[i * dv + j];
      pred[j] = kd;
      corr[j] = val[j] - kd;
    }
    /* write: S = D + beta k corr^T */
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[i * dv + j] += write_rate * key[i] * corr[j];
  }
  free(corr);
}

int orc_gated_delta(const double* k, const double* v, const double* beta,
                    const double* alpha, int B, int H, int N, int dk, int dv,
                    const double* S0, double* reads, double* S_N, int nthreads) {
  if (B < 1 || H < 1 || N < 0 || dk < 1 || dv < 1 || !S_N) return -1;
  if (N > 0 && (!k || !v || !beta || !reads)) return -1;
  gdelta_args a = {k, v, beta, alpha, S0, N, dk, dv, reads, S_N};
  for_each_head((int64_t)B * H, nthreads, gated_delta_head, &a);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* (8) Variants of the recurrence of (1).
 *   mode 0 (write, then read; P1 section 03) with a scalar decay of the old
 *     state, P3 sections 3-4 (Mamba-2: S_t = alpha_t S_{t-1} + v_t k_t^T, the
 *     linear-attention recurrence with one scalar on the old state).  The
 *     normalizer is part of the state and decays with it:
 *       S_t = alpha_t S_{t-1} + phi(k_t) v_t^T,  z_t = alpha_t z_{t-1} + phi(k_t),
 *       o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps).
 *   mode 1 (read, then write: strictly past; P1 section 03 and section 09,
 *     first change): o_t = phi(q_t)^T S_{t-1} / (phi(q_t)^T z_{t-1} + eps),
 *     then the write of mode 0 (decay included).  From a zero state the first
 *     read is 0.
 *   mode 2 (non-causal; P2 section 线性化核心 and its linear_attention): the state is
 *     formed once over all N tokens, S = S0 + sum_t phi(k_t) v_t^T,
 *     z = z0 + sum_t phi(k_t), and every query reads it.  No decay (alpha must
 *     be NULL).
 * alpha = NULL means alpha_t = 1. */
typedef struct {
  const double *q, *k, *v, *alpha, *S0, *z0;
  int N, dk, dv, mode;
  double eps;
  double *o, *S_N, *z_N;
} var_args;

static void var_read(const double* fq, const double* S, const double* z, int dk,
                     int dv, double eps, double* ot) {
  double den = 0.0;
  for (int i = 0; i < dk; ++i) den += fq[i] * z[i];
  den += eps;
  for (int j = 0; j < dv; ++j) {
    double num = 0.0;
    for (int i = 0; i < dk; ++i) num += fq[i] * S[i * dv + j];
    ot[j] = num / den;
  }
}

static void var_write(const double* fk, const double* vt, double at, double* S,
                      double* z, int dk, int dv) {
  for (int i = 0; i < dk; ++i) {
    for (int j = 0; j < dv; ++j) S[i * dv + j] = at * S[i * dv + j] + fk[i] * vt[j];
    z[i] = at * z[i] + fk[i];
  }
}

static void variant_head(void* p, int64_t h) {
  const var_args* a = (const var_args*)p;
  const int N = a->N, dk = a->dk, dv = a->dv;
  double* S = a->S_N + h * (int64_t)dk * dv;
  double* z = a->z_N + h * (int64_t)dk;
  if (a->S0) memcpy(S, a->S0 + h * (int64_t)dk * dv, sizeof(double) * dk * dv);
  else memset(S, 0, sizeof(double) * dk * dv);
  if (a->z0) memcpy(z, a->z0 + h * (int64_t)dk, sizeof(double) * dk);
  else memset(z, 0, sizeof(double) * dk);
  double* fk = (double*)malloc(sizeof(double) * dk);
  double* fq = (double*)malloc(sizeof(double) * dk);
  if (a->mode == 2) {
    /* the state over all tokens first */
    for (int t = 0; t < N; ++t) {
      const double* kt = a->k + (h * (int64_t)N + t) * dk;
      const double* vt = a->v + (h * (int64_t)N + t) * dv;
      for (int i = 0; i < dk; ++i) fk[i] = phi(kt[i]);
      var_write(fk, vt, 1.0, S, z, dk, dv);
    }
    /* then every query reads it */
    for (int t = 0; t < N; ++t) {
      const double* qt = a->q + (h * (int64_t)N + t) * dk;
      for (int i = 0; i < dk; ++i) fq[i] = phi(qt[i]);
      var_read(fq, S, z, dk, dv, a->eps, a->o + (h * (int64_t)N + t) * dv);
    }
  } else {
    for (int t = 0; t < N; ++t) {
      const double* qt = a->q + (h * (int64_t)N + t) * dk;
      const double* kt = a->k + (h * (int64_t)N + t) * dk;
      const double* vt = a->v + (h * (int64_t)N + t) * dv;
      double* ot = a->o + (h * (int64_t)N + t) * dv;
      const double at = a->alpha ? a->alpha[h * (int64_t)N + t] : 1.0;
      for (int i = 0; i < dk; ++i) fk[i] = phi(kt[i]);
      for (int i = 0; i < dk; ++i) fq[i] = phi(qt[i]);
      if (a->mode == 1) var_read(fq, S, z, dk, dv, a->eps, ot);
      var_write(fk, vt, at, S, z, dk, dv);
      if (a->mode == 0) var_read(fq, S, z, dk, dv, a->eps, ot);
    }
  }
  free(fk);
  free(fq);
}

int orc_la_variant(const double* q, const double* k, const double* v,
                   const double* alpha, int B, int H, int N, int dk, int dv,
                   double eps, int mode, const double* S0, const double* z0,
                   double* o, double* S_N, double* z_N, int nthreads) {
  if (la_check(q, k, v, B, H, N, dk, dv, eps, o) || !S_N || !z_N) return -1;
  if (mode < 0 || mode > 2 || (mode == 2 && alpha)) return -1;
  var_args a = {q, k, v, alpha, S0, z0, N, dk, dv, mode, eps, o, S_N, z_N};
  for_each_head((int64_t)B * H, nthreads, variant_head, &a);
  return 0;
}

/* (9) The outputs of (8) from explicit weights, the pages' quadratic form
 * (P1 appendix explicit_linear) with the recurrence unrolled: the read at t
 * sees token s with weight phi(q_t).phi(k_s) times the decay applied to it
 * afterwards, and the initial state with the decay applied since the start:
 *   mode 0: tokens s <= t, decay prod_{s < r <= t} alpha_r; S0, z0 with
 *           prod_{r <= t} alpha_r
 *   mode 1: tokens s < t, decay prod_{s < r < t} alpha_r; S0, z0 with
 *           prod_{r < t} alpha_r
 *   mode 2: every token, no decay; S0, z0 as they are. */
static void variant_quadratic_head(void* p, int64_t h) {
  const var_args* a = (const var_args*)p;
  const int N = a->N, dk = a->dk, dv = a->dv, mode = a->mode;
  const double* S0 = a->S0 ? a->S0 + h * (int64_t)dk * dv : NULL;
  const double* z0 = a->z0 ? a->z0 + h * (int64_t)dk : NULL;
  const double* al = a->alpha ? a->alpha + h * (int64_t)N : NULL;
  double* fq = (double*)malloc(sizeof(double) * dk);
  double* fk = (double*)malloc(sizeof(double) * dk);
  double* num = (double*)malloc(sizeof(double) * dv);
  for (int t = 0; t < N; ++t) {
    const double* qt = a->q + (h * (int64_t)N + t) * dk;
    for (int r = 0; r < dk; ++r) fq[r] = phi(qt[r]);
    /* decay of the initial state up to the read */
    const int last = mode == 0 ? t : t - 1; /* alpha_r applied for r <= last */
    double g0 = 1.0;
    if (al && mode != 2)
      for (int r = 0; r <= last; ++r) g0 *= al[r];
    double den = 0.0;
    for (int j = 0; j < dv; ++j) num[j] = 0.0;
    if (S0)
      for (int r = 0; r < dk; ++r)
        for (int j = 0; j < dv; ++j) num[j] += g0 * fq[r] * S0[r * dv + j];
    if (z0)
      for (int r = 0; r < dk; ++r) den += g0 * fq[r] * z0[r];
    const int send = mode == 0 ? t : (mode == 1 ? t - 1 : N - 1);
    for (int s = 0; s <= send; ++s) {
      const double* ks = a->k + (h * (int64_t)N + s) * dk;
      const double* vs = a->v + (h * (int64_t)N + s) * dv;
      for (int r = 0; r < dk; ++r) fk[r] = phi(ks[r]);
      double g = 1.0;
      if (al && mode != 2)
        for (int r = s + 1; r <= last; ++r) g *= al[r];
      double w = 0.0;
      for (int r = 0; r < dk; ++r) w += fq[r] * fk[r];
      w *= g;
      den += w;
      for (int j = 0; j < dv; ++j) num[j] += w * vs[j];
    }
    den += a->eps;
    double* ot = a->o + (h * (int64_t)N + t) * dv;
    for (int j = 0; j < dv; ++j) ot[j] = num[j] / den;
  }
  free(fq);
  free(fk);
  free(num);
}

int orc_la_variant_quadratic(const double* q, const double* k, const double* v,
                             const double* alpha, int B, int H, int N, int dk,
                             int dv, double eps, int mode, const double* S0,
                             const double* z0, double* o, int nthreads) {
  if (la_check(q, k, v, B, H, N, dk, dv, eps, o)) return -1;
  if (mode < 0 || mode > 2 || (mode == 2 && alpha)) return -1;
  var_args a = {q, k, v, alpha, S0, z0, N, dk, dv, mode, eps, o, NULL, NULL};
  for_each_head((int64_t)B * H, nthreads, variant_quadratic_head, &a);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* (10) Gradient of (1).  The pages give no backward pass: P1 section 03 only
 * notes that training must not keep every state, and that prefix sums,
 * chunking and recomputation handle it.  This is the exact derivative of the
 * map (q, k, v, S0, z0) -> (o, S_N, z_N) of (1), with the states recomputed:
 * given dO (upstream gradient of o) and dS_N, dz_N (of the final state, NULL =
 * zero), with num_t = S_t^T phi(q_t), den_t = phi(q_t).z_t + eps, o_t = num_t / den_t:
 *   dnum_t = dO_t / den_t,   dden_t = -(dO_t . o_t) / den_t
 *   dphi(q_t) = S_t dnum_t + dden_t z_t                      (forward sweep)
 *   G_t = dS_N + sum_{tau >= t} phi(q_tau) dnum_tau^T,  g_t = dz_N + sum_{tau >= t} dden_tau phi(q_tau)
 *   dphi(k_t) = G_t v_t + g_t,   dv_t = G_t^T phi(k_t)      (reverse sweep)
 *   dS0 = G_0, dz0 = g_0;  dq = dphi(q) phi'(q), dk = dphi(k) phi'(k)
 * with phi'(u) = 1 for u > 0 and exp(u) for u <= 0. */
static double dphi(double u) { return u > 0.0 ? 1.0 : exp(u); }

typedef struct {
  const double *q, *k, *v, *S0, *z0, *dO, *dS_N, *dz_N;
  int N, dk, dv;
  double eps;
  double *dq, *dk_out, *dv_out, *dS0, *dz0;
} bwd_args;

static void backward_head(void* p, int64_t h) {
  const bwd_args* a = (const bwd_args*)p;
  const int N = a->N, dk = a->dk, dv = a->dv;
  double* S = (double*)malloc(sizeof(double) * dk * dv);
  double* z = (double*)malloc(sizeof(double) * dk);
  double* fq = (double*)malloc(sizeof(double) * dk);
  double* fk = (double*)malloc(sizeof(double) * dk);
  double* num = (double*)malloc(sizeof(double) * dv);
  double* dnum = (double*)malloc(sizeof(double) * (N > 0 ? N : 1) * dv);
  double* dden = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
  if (a->S0) memcpy(S, a->S0 + h * (int64_t)dk * dv, sizeof(double) * dk * dv);
  else memset(S, 0, sizeof(double) * dk * dv);
  if (a->z0) memcpy(z, a->z0 + h * (int64_t)dk, sizeof(double) * dk);
  else memset(z, 0, sizeof(double) * dk);
  /* forward sweep: the states again, the output's local gradients, dq */
  for (int t = 0; t < N; ++t) {
    const double* qt = a->q + (h * (int64_t)N + t) * dk;
    const double* kt = a->k + (h * (int64_t)N + t) * dk;
    const double* vt = a->v + (h * (int64_t)N + t) * dv;
    const double* gt = a->dO + (h * (int64_t)N + t) * dv;
    for (int i = 0; i < dk; ++i) fk[i] = phi(kt[i]);
    for (int i = 0; i < dk; ++i) fq[i] = phi(qt[i]);
    for (int i = 0; i < dk; ++i) {
      for (int j = 0; j < dv; ++j) S[i * dv + j] += fk[i] * vt[j];
      z[i] += fk[i];
    }
    double den = a->eps;
    for (int i = 0; i < dk; ++i) den += fq[i] * z[i];
    double go = 0.0;
    for (int j = 0; j < dv; ++j) {
      double nj = 0.0;
      for (int i = 0; i < dk; ++i) nj += fq[i] * S[i * dv + j];
      num[j] = nj;
      go += gt[j] * (nj / den);
    }
    for (int j = 0; j < dv; ++j) dnum[(int64_t)t * dv + j] = gt[j] / den;
    dden[t] = -go / den;
    double* dqt = a->dq + (h * (int64_t)N + t) * dk;
    for (int i = 0; i < dk; ++i) {
      double d = dden[t] * z[i];
      for (int j = 0; j < dv; ++j) d += S[i * dv + j] * dnum[(int64_t)t * dv + j];
      dqt[i] = d * dphi(qt[i]);
    }
  }
  /* reverse sweep: the gradient of every later state, dk, dv */
  double* G = S; /* reuse */
  double* g = z;
  if (a->dS_N) memcpy(G, a->dS_N + h * (int64_t)dk * dv, sizeof(double) * dk * dv);
  else memset(G, 0, sizeof(double) * dk * dv);
  if (a->dz_N) memcpy(g, a->dz_N + h * (int64_t)dk, sizeof(double) * dk);
  else memset(g, 0, sizeof(double) * dk);
  for (int t = N - 1; t >= 0; --t) {
    const double* qt = a->q + (h * (int64_t)N + t) * dk;
    const double* kt = a->k + (h * (int64_t)N + t) * dk;
    const double* vt = a->v + (h * (int64_t)N + t) * dv;
    for (int i = 0; i < dk; ++i) fq[i] = phi(qt[i]);
    for (int i = 0; i < dk; ++i) fk[i] = phi(kt[i]);
    for (int i = 0; i < dk; ++i) {
      for (int j = 0; j < dv; ++j) G[i * dv + j] += fq[i] * dnum[(int64_t)t * dv + j];
      g[i] += dden[t] * fq[i];
    }
    double* dkt = a->dk_out + (h * (int64_t)N + t) * dk;
    double* dvt = a->dv_out + (h * (int64_t)N + t) * dv;
    for (int i = 0; i < dk; ++i) {
      double d = g[i];
      for (int j = 0; j < dv; ++j) d += G[i * dv + j] * vt[j];
      dkt[i] = d * dphi(kt[i]);
    }
    for (int j = 0; j < dv; ++j) {
      double d = 0.0;
      for (int i = 0; i < dk; ++i) d += G[i * dv + j] * fk[i];
      dvt[j] = d;
    }
  }
  if (a->dS0) memcpy(a->dS0 + h * (int64_t)dk * dv, G, sizeof(double) * dk * dv);
  if (a->dz0) memcpy(a->dz0 + h * (int64_t)dk, g, sizeof(double) * dk);
  free(S); free(z); free(fq); free(fk); free(num); free(dnum); free(dden);
}

int orc_la_backward(const double* q, const double* k, const double* v, int B, int H,
                    int N, int dk, int dv, double eps, const double* S0,
                    const double* z0, const double* dO, const double* dS_N,
                    const double* dz_N, double* dq, double* dk_out, double* dv_out,
                    double* dS0, double* dz0, int nthreads) {
  if (la_check(q, k, v, B, H, N, dk, dv, eps, dO)) return -1;
  if (N > 0 && (!dq || !dk_out || !dv_out)) return -1;
  bwd_args a = {q, k, v, S0, z0, dO, dS_N, dz_N, N, dk, dv, eps, dq, dk_out, dv_out, dS0, dz0};
  for_each_head((int64_t)B * H, nthreads, backward_head, &a);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* (6) Additive outer-product memory with identity features, the write/read
 * primitive of P3 section 1.3 (memory collision) and of the two-entry example
 * on the associative-memory page: S = sum_m k_m v_m^T (k v^T convention), read
 * with a query from the left, q^T S = sum_m (q . k_m) v_m^T. */
int orc_outer_read(const double* keys, const double* values, int M, int dk,
                   int dv, const double* queries, int P, double* reads) {
  if (M < 0 || P < 0 || dk < 1 || dv < 1) return -1;
  if ((M > 0 && (!keys || !values)) || (P > 0 && (!queries || !reads))) return -1;
  double* S = (double*)calloc((size_t)dk * dv, sizeof(double));
  for (int m = 0; m < M; ++m)
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[i * dv + j] += keys[m * dk + i] * values[m * dv + j];
  for (int p = 0; p < P; ++p)
    for (int j = 0; j < dv; ++j) {
      double r = 0.0;
      for (int i = 0; i < dk; ++i) r += queries[p * dk + i] * S[i * dv + j];
      reads[p * dv + j] = r;
    }
  free(S);
  return 0;
}
