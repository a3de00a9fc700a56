/*
 * CPU oracle for mha_prefill -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library.  The product path (the CUDA library and its Python
 * binding) never calls it and shares no code with it.
 *
 * What it computes (TokenSpeed-kernel README, "Public API": the `mha_prefill`
 * call; the attention it serves is GPT-OSS attention with attention sinks and
 * a mix of sliding-window and full layers, page "TokenSpeed-kernel:
 * multi-silicon ...", section "Числа: Gluon на AMD MI355X", and the ai-radar.it
 * article, section "AMD MI355X: la prova sul campo").  The pages do not write
 * the formula out; the reading taken here is the plain one:
 *
 *   for sequence s with tokens [start, start+L), token t, query head h,
 *   KV head g = h / (Hq/Hkv):
 *     J      = { j : max(start, t-W+1) <= j <= t }       (W <= 0: j >= start)
 *     s_j    = scale * sum_d q[t,h,d] * k[j,g,d]
 *     M      = max(max_j s_j, sink_h)                   (no sinks: sink term absent)
 *     Z      = sum_j exp(s_j - M) + exp(sink_h - M)
 *     out    = sum_j exp(s_j - M) * v[j,g,:] / Z
 *     lse    = M + log(Z)                                (natural log, sink included)
 *
 * The sink is a raw logit: it is not multiplied by `scale`.  Inputs q, k, v
 * are bf16 bit patterns widened exactly to double; every sum is in double.
 * Each row is evaluated in the two-pass form (max, then exponentials).
 *
 * Prefill over a key/value cache (the README's `mha_prefill_with_kvcache`
 * call, section "Public API"; the pages give no formula): sequence s has Lq
 * new query tokens (rows cu_q[s].. of q) and Lk >= Lq keys (rows cu_k[s].. of
 * k and v: the cached prefix followed by the new tokens' keys).  New token i
 * sits at key position P = Lk - Lq + i and attends to key positions
 * max(0, P-W+1) .. P (causal aligned to the end of the keys).  With Lk == Lq
 * this is the prefill above.
 *
 * Plain C99 + pthreads; portable (no architecture-specific code).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
  const uint16_t *q, *k, *v;
  const double *sinks;
  const int32_t *cu;   /* query sequence offsets */
  int num_seqs, Hq, Hkv, D, window;
  double scale;
  const int32_t *cu_k; /* key sequence offsets (== cu for plain prefill) */
} problem_t;

static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* One output row: query row tq (absolute), query head h; the query sits at
 * absolute key row t of a key sequence starting at start_k.  `work` holds at
 * least t-start_k+1 doubles. */
static void one_row(const problem_t *p, int64_t tq, int64_t start_k, int64_t t, int h,
                    double *out_row, double *lse_out, double *work, double *qrow) {
  /* tq: absolute query row; t: absolute key row of the query's own position */
  const int D = p->D, G = p->Hq / p->Hkv, g = h / G;
  int64_t lo = start_k;
  if (p->window > 0 && t - p->window + 1 > lo) lo = t - p->window + 1;
  const int64_t n = t - lo + 1;

  for (int d = 0; d < D; ++d) qrow[d] = bf16_to_double(p->q[(tq * p->Hq + h) * (int64_t)D + d]);

  /* pass 1: scores and their maximum (sink included) */
  double M = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    const uint16_t *kr = p->k + ((lo + j) * p->Hkv + g) * (int64_t)D;
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qrow[d] * bf16_to_double(kr[d]);
    work[j] = p->scale * acc;
    if (work[j] > M) M = work[j];
  }
  const int has_sink = p->sinks != 0;
  const double sink = has_sink ? p->sinks[h] : -INFINITY;
  if (has_sink && sink > M) M = sink;

  /* pass 2: exponentials, normaliser, weighted sum of values */
  double Z = 0.0;
  for (int d = 0; d < D; ++d) out_row[d] = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    const double e = exp(work[j] - M);
    Z += e;
    const uint16_t *vr = p->v + ((lo + j) * p->Hkv + g) * (int64_t)D;
    for (int d = 0; d < D; ++d) out_row[d] += e * bf16_to_double(vr[d]);
  }
  if (has_sink) Z += exp(sink - M);
  for (int d = 0; d < D; ++d) out_row[d] /= Z;
  if (lse_out) *lse_out = M + log(Z);
}

static int64_t seq_of_token(const problem_t *p, int64_t t) {
  int lo = 0, hi = p->num_seqs - 1; /* last s with cu[s] <= t, skipping empty ones */
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (p->cu[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  while (lo + 1 <= p->num_seqs - 1 && p->cu[lo + 1] <= t) ++lo;
  return lo;
}

typedef struct {
  const problem_t *p;
  /* full mode */
  double *out, *lse;
  /* row mode */
  const int64_t *row_t;
  const int32_t *row_h;
  int64_t nrows;
  int mode; /* 0 full, 1 rows */
  int64_t max_len;
  int64_t next; /* shared counter, protected by mu */
  pthread_mutex_t *mu;
  int err;
} shared_t;

static int64_t grab(shared_t *sh, int64_t chunk) {
  pthread_mutex_lock(sh->mu);
  int64_t r = sh->next;
  sh->next += chunk;
  pthread_mutex_unlock(sh->mu);
  return r;
}

static void *worker(void *arg) {
  shared_t *sh = (shared_t *)arg;
  const problem_t *p = sh->p;
  double *work = (double *)malloc(sizeof(double) * (size_t)(sh->max_len + 1));
  double *qrow = (double *)malloc(sizeof(double) * (size_t)p->D);
  if (!work || !qrow) {
    free(work);
    free(qrow);
    pthread_mutex_lock(sh->mu);
    sh->err = 1;
    pthread_mutex_unlock(sh->mu);
    return 0;
  }
  const int64_t total = sh->mode == 0 ? (int64_t)p->cu[p->num_seqs] * p->Hq : sh->nrows;
  const int64_t chunk = 16;
  for (;;) {
    int64_t b = grab(sh, chunk);
    if (b >= total) break;
    int64_t e = b + chunk < total ? b + chunk : total;
    for (int64_t i = b; i < e; ++i) {
      int64_t t;
      int h;
      double *orow, *lrow;
      if (sh->mode == 0) {
        t = i / p->Hq;
        h = (int)(i % p->Hq);
        orow = sh->out + i * p->D;
        lrow = sh->lse ? sh->lse + i : 0;
      } else {
        t = sh->row_t[i];
        h = sh->row_h[i];
        orow = sh->out + i * p->D;
        lrow = sh->lse ? sh->lse + i : 0;
      }
      int64_t s = seq_of_token(p, t);
      const int64_t lq = (int64_t)p->cu[s + 1] - p->cu[s];
      const int64_t lk = (int64_t)p->cu_k[s + 1] - p->cu_k[s];
      const int64_t pos = p->cu_k[s] + (lk - lq) + (t - p->cu[s]);
      one_row(p, t, p->cu_k[s], pos, h, orow, lrow, work, qrow);
    }
  }
  free(work);
  free(qrow);
  return 0;
}

static int check_problem(const problem_t *p) {
  if (!p->q || !p->k || !p->v || !p->cu || !p->cu_k) return -1;
  if (p->num_seqs < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0) return -1;
  if (p->Hq % p->Hkv) return -1;
  if (p->cu[0] != 0 || p->cu_k[0] != 0) return -1;
  for (int s = 0; s < p->num_seqs; ++s) {
    if (p->cu[s + 1] < p->cu[s] || p->cu_k[s + 1] < p->cu_k[s]) return -1;
    if (p->cu_k[s + 1] - p->cu_k[s] < p->cu[s + 1] - p->cu[s]) return -1; /* Lk >= Lq */
  }
  return 0;
}

static int run(shared_t *sh, int nthreads) {
  const problem_t *p = sh->p;
  int64_t max_len = 1;
  for (int s = 0; s < p->num_seqs; ++s) {
    int64_t L = (int64_t)p->cu_k[s + 1] - p->cu_k[s];
    if (L > max_len) max_len = L;
  }
  sh->max_len = max_len;
  if (nthreads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = n > 0 ? (int)n : 1;
  }
  if (nthreads > 512) nthreads = 512;
  pthread_t th[512];
  int started = 0;
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&th[i], 0, worker, sh) != 0) break;
    started = i;
  }
  worker(sh);
  for (int i = 1; i <= started; ++i) pthread_join(th[i], 0);
  return sh->err ? -2 : started + 1;
}

static int run_full(const problem_t *p, double *out, double *lse, int nthreads) {
  if (check_problem(p) || !out) return -1;
  pthread_mutex_t mu = PTHREAD_MUTEX_INITIALIZER;
  shared_t sh;
  memset(&sh, 0, sizeof sh);
  sh.p = p;
  sh.out = out;
  sh.lse = lse;
  sh.mode = 0;
  sh.mu = &mu;
  return run(&sh, nthreads);
}

static int run_rows(const problem_t *p, const int64_t *row_t, const int32_t *row_h,
                    int64_t nrows, double *out, double *lse, int nthreads) {
  if (check_problem(p) || !out || (nrows > 0 && (!row_t || !row_h))) return -1;
  const int64_t T = p->cu[p->num_seqs];
  for (int64_t i = 0; i < nrows; ++i)
    if (row_t[i] < 0 || row_t[i] >= T || row_h[i] < 0 || row_h[i] >= p->Hq) return -1;
  pthread_mutex_t mu = PTHREAD_MUTEX_INITIALIZER;
  shared_t sh;
  memset(&sh, 0, sizeof sh);
  sh.p = p;
  sh.out = out;
  sh.lse = lse;
  sh.row_t = row_t;
  sh.row_h = row_h;
  sh.nrows = nrows;
  sh.mode = 1;
  sh.mu = &mu;
  return run(&sh, nthreads);
}

/*
 * Full evaluation.  q: [T,Hq,D], k/v: [T,Hkv,D] bf16 bits; sinks: [Hq] or NULL;
 * cu_seqlens: [num_seqs+1]; out: [T,Hq,D] double; lse: [T,Hq] double or NULL.
 * Returns the number of threads used (> 0) or a negative error.
 */
int oracle_mha_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const double *sinks, const int32_t *cu_seqlens, int num_seqs, int Hq,
                       int Hkv, int D, int window, double scale, double *out, double *lse,
                       int nthreads) {
  problem_t p = {q, k, v, sinks, cu_seqlens, num_seqs, Hq, Hkv, D, window, scale, cu_seqlens};
  return run_full(&p, out, lse, nthreads);
}

/*
 * Selected rows only: row i is (token row_t[i], head row_h[i]).
 * out: [nrows, D] double; lse: [nrows] double or NULL.
 */
int oracle_mha_prefill_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const double *sinks, const int32_t *cu_seqlens, int num_seqs,
                            int Hq, int Hkv, int D, int window, double scale,
                            const int64_t *row_t, const int32_t *row_h, int64_t nrows,
                            double *out, double *lse, int nthreads) {
  problem_t p = {q, k, v, sinks, cu_seqlens, num_seqs, Hq, Hkv, D, window, scale, cu_seqlens};
  return run_rows(&p, row_t, row_h, nrows, out, lse, nthreads);
}

/*
 * Prefill over a key/value cache.  q: [Tq,Hq,D] with cu_q; k/v: [Tk,Hkv,D] with
 * cu_k (per sequence Lk >= Lq); out: [Tq,Hq,D]; lse: [Tq,Hq] or NULL.
 */
int oracle_mha_prefill_kvcache(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const double *sinks, const int32_t *cu_q, const int32_t *cu_k,
                               int num_seqs, int Hq, int Hkv, int D, int window, double scale,
                               double *out, double *lse, int nthreads) {
  problem_t p = {q, k, v, sinks, cu_q, num_seqs, Hq, Hkv, D, window, scale, cu_k};
  return run_full(&p, out, lse, nthreads);
}

int oracle_mha_prefill_kvcache_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                    const double *sinks, const int32_t *cu_q,
                                    const int32_t *cu_k, int num_seqs, int Hq, int Hkv, int D,
                                    int window, double scale, const int64_t *row_t,
                                    const int32_t *row_h, int64_t nrows, double *out,
                                    double *lse, int nthreads) {
  problem_t p = {q, k, v, sinks, cu_q, num_seqs, Hq, Hkv, D, window, scale, cu_k};
  return run_rows(&p, row_t, row_h, nrows, out, lse, nthreads);
}
