/*
 * Exact softmax-attention forward: the fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline / reference arm may load or call this code.  The
 * product path never does, and this file shares no code with the CUDA path.
 *
 * What it computes is the plain definition of attention, with no tiling and no
 * online recurrence ("FlashAttention V2", section 3: the method reaches this
 * same result exactly up to rounding; "FlashAttention-2 in an attention layer",
 * Triton FA2 kernel: scores = scale * q.k, causal keeps key <= query, softmax
 * over keys, weighted sum of V rows).  For one query row i of head (b, h):
 *
 *   s_j   = scale * sum_d q_id k_jd          for every allowed key j
 *           (allowed: j < S; with the causal mask also j <= i)
 *   m     = max_j s_j
 *   l     = sum_j exp(s_j - m)
 *   O_id  = (sum_j exp(s_j - m) v_jd) / l
 *   LSE_i = m + ln(l)                         (natural log, scaled scores)
 *
 * Each row's full score vector is materialised (length S, fp64).  Rows are
 * independent, so a pool of POSIX threads takes contiguous ranges of rows.
 *
 * Inputs are fp64 [B, H, S, D] row-major; the 16-bit values are widened
 * exactly before they get here.  Outputs are fp64.  A subset of rows may be
 * requested (``rows`` holds global row indices bh * S + i); the outputs are
 * then packed in the order of that list.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

enum {
  ORACLE_OK = 0,
  ORACLE_EINVAL = -1,
  ORACLE_ENOMEM = -2,
  ORACLE_ENORM = -3, /* a row's normaliser came out below 1: cannot happen */
};

typedef struct {
  const double *q, *k, *v;
  long long S, D, BH;
  int causal;
  double scale;
  const long long *rows; /* NULL: every row, in order */
  double *o, *lse, *p;   /* p optional: [nrows, S] softmax probabilities */
  long long r0, r1;      /* this worker's output-row range */
  int status;
} oracle_job;

/* One query row.  ``g`` is its global index bh * S + i, ``out`` the output
 * slot, ``w`` a scratch vector of length S. */
static int oracle_row(const oracle_job *J, long long out, long long g,
                      double *w) {
  const long long S = J->S, D = J->D;
  const long long bh = g / S, i = g % S;
  const double *qi = J->q + g * D;
  const double *kh = J->k + bh * S * D;
  const double *vh = J->v + bh * S * D;
  const long long n = J->causal ? i + 1 : S; /* keys 0 .. n-1 are allowed */

  /* scores, materialised */
  for (long long j = 0; j < n; ++j) {
    const double *kj = kh + j * D;
    double acc = 0.0;
    for (long long d = 0; d < D; ++d) acc += qi[d] * kj[d];
    w[j] = J->scale * acc;
  }
  /* row maximum */
  double m = w[0];
  for (long long j = 1; j < n; ++j)
    if (w[j] > m) m = w[j];
  /* unnormalised weights and their sum */
  double l = 0.0;
  for (long long j = 0; j < n; ++j) {
    w[j] = exp(w[j] - m);
    l += w[j];
  }
  if (!(l >= 1.0)) return ORACLE_ENORM; /* the maximum contributes exp(0)=1 */
  /* weighted sum of V rows, one division at the end */
  double *oi = J->o + out * D;
  for (long long d = 0; d < D; ++d) oi[d] = 0.0;
  for (long long j = 0; j < n; ++j) {
    const double *vj = vh + j * D;
    const double wj = w[j];
    for (long long d = 0; d < D; ++d) oi[d] += wj * vj[d];
  }
  for (long long d = 0; d < D; ++d) oi[d] /= l;
  J->lse[out] = m + log(l);
  if (J->p) {
    double *pi = J->p + out * S;
    for (long long j = 0; j < S; ++j) pi[j] = j < n ? w[j] / l : 0.0;
  }
  return ORACLE_OK;
}

static void *oracle_worker(void *arg) {
  oracle_job *J = (oracle_job *)arg;
  double *w = (double *)malloc(sizeof(double) * (size_t)(J->S > 0 ? J->S : 1));
  if (!w) {
    J->status = ORACLE_ENOMEM;
    return NULL;
  }
  for (long long r = J->r0; r < J->r1 && J->status == ORACLE_OK; ++r) {
    const long long g = J->rows ? J->rows[r] : r;
    J->status = oracle_row(J, r, g, w);
  }
  free(w);
  return NULL;
}

/* Returns ORACLE_OK or a negative code.  ``nthreads`` <= 0 means one. */
int oracle_attn_fwd(const double *q, const double *k, const double *v,
                    long long B, long long H, long long S, long long D,
                    int causal, double scale, const long long *rows,
                    long long nrows, double *o, double *lse, double *p,
                    int nthreads) {
  if (!q || !k || !v || !o || !lse || B < 1 || H < 1 || S < 1 || D < 1)
    return ORACLE_EINVAL;
  if (!(scale > 0.0) || !isfinite(scale)) return ORACLE_EINVAL;
  const long long BH = B * H;
  const long long total = rows ? nrows : BH * S;
  if (rows) {
    for (long long r = 0; r < nrows; ++r)
      if (rows[r] < 0 || rows[r] >= BH * S) return ORACLE_EINVAL;
  }
  if (total <= 0) return ORACLE_OK;
  if (nthreads < 1) nthreads = 1;
  if ((long long)nthreads > total) nthreads = (int)total;

  oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
  pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  char *made = (char *)calloc((size_t)nthreads, 1);
  if (!jobs || !tid || !made) {
    free(jobs);
    free(tid);
    free(made);
    return ORACLE_ENOMEM;
  }
  int status = ORACLE_OK;
  for (int t = 0; t < nthreads; ++t) {
    oracle_job *J = &jobs[t];
    J->q = q; J->k = k; J->v = v;
    J->S = S; J->D = D; J->BH = BH;
    J->causal = causal;
    J->scale = scale;
    J->rows = rows;
    J->o = o; J->lse = lse; J->p = p;
    J->r0 = total * t / nthreads;
    J->r1 = total * (t + 1) / nthreads;
    J->status = ORACLE_OK;
    if (nthreads > 1 && pthread_create(&tid[t], NULL, oracle_worker, J) == 0)
      made[t] = 1;
    else
      oracle_worker(J); /* one thread, or no thread could be made */
  }
  for (int t = 0; t < nthreads; ++t)
    if (made[t]) pthread_join(tid[t], NULL);
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].status != ORACLE_OK) status = jobs[t].status;
  free(jobs);
  free(tid);
  free(made);
  return status;
}

/*
 * Attention of a few new query rows against a key/value cache
 * ("FlashAttention V2", section 6, the table of when V2 is used: inference
 * with a KV cache is served by its decoding variant).
 *
 * Head (b, h) holds len_b cached positions 0 .. len_b - 1 in rows of a
 * [B, H, Sk, D] cache (Sk >= len_b is the cache's capacity; rows at or past
 * len_b are ignored whatever they hold).  The Sq new queries are the last Sq
 * positions of that sequence, so query i sits at position len_b - Sq + i.
 * Allowed keys for query i: every j < len_b; with the causal mask only
 * j <= len_b - Sq + i (the same "key <= query" rule as the self-attention
 * case, positions counted from the start of the sequence).  Then, as above,
 *
 *   s_j = scale * q_i . k_j,  m = max s_j,  l = sum exp(s_j - m),
 *   O_i = sum_j exp(s_j - m) v_j / l,  LSE_i = m + ln l.
 *
 * A query with no allowed key (len_b = 0, or causal with len_b - Sq + i < 0)
 * gets O_i = 0 and LSE_i = -inf, the logarithm of an empty sum.
 *
 * q, o: [B, H, Sq, D]; k, v: [B, H, Sk, D]; lse: [B, H, Sq]; lens: [B] or
 * NULL for len_b = Sk.  Every len_b must lie in [0, Sk].
 */
typedef struct {
  const double *q, *k, *v;
  const long long *lens;
  long long H, Sq, Sk, D;
  int causal;
  double scale;
  double *o, *lse;
  long long r0, r1;
  int status;
} oracle_kv_job;

static int oracle_kv_row(const oracle_kv_job *J, long long g, double *w) {
  const long long Sq = J->Sq, Sk = J->Sk, D = J->D;
  const long long bh = g / Sq, i = g % Sq, b = bh / J->H;
  const long long len = J->lens ? J->lens[b] : Sk;
  const double *qi = J->q + g * D;
  const double *kh = J->k + bh * Sk * D;
  const double *vh = J->v + bh * Sk * D;
  double *oi = J->o + g * D;
  long long n = len; /* keys 0 .. n-1 are allowed */
  if (J->causal && len - Sq + i + 1 < n) n = len - Sq + i + 1;
  for (long long d = 0; d < D; ++d) oi[d] = 0.0;
  if (n <= 0) {
    J->lse[g] = -INFINITY;
    return ORACLE_OK;
  }
  for (long long j = 0; j < n; ++j) {
    const double *kj = kh + j * D;
    double acc = 0.0;
    for (long long d = 0; d < D; ++d) acc += qi[d] * kj[d];
    w[j] = J->scale * acc;
  }
  double m = w[0];
  for (long long j = 1; j < n; ++j)
    if (w[j] > m) m = w[j];
  double l = 0.0;
  for (long long j = 0; j < n; ++j) {
    w[j] = exp(w[j] - m);
    l += w[j];
  }
  if (!(l >= 1.0)) return ORACLE_ENORM;
  for (long long j = 0; j < n; ++j) {
    const double *vj = vh + j * D;
    for (long long d = 0; d < D; ++d) oi[d] += w[j] * vj[d];
  }
  for (long long d = 0; d < D; ++d) oi[d] /= l;
  J->lse[g] = m + log(l);
  return ORACLE_OK;
}

static void *oracle_kv_worker(void *arg) {
  oracle_kv_job *J = (oracle_kv_job *)arg;
  double *w = (double *)malloc(sizeof(double) * (size_t)(J->Sk > 0 ? J->Sk : 1));
  if (!w) {
    J->status = ORACLE_ENOMEM;
    return NULL;
  }
  for (long long r = J->r0; r < J->r1 && J->status == ORACLE_OK; ++r)
    J->status = oracle_kv_row(J, r, w);
  free(w);
  return NULL;
}

int oracle_attn_kvcache(const double *q, const double *k, const double *v,
                        long long B, long long H, long long Sq, long long Sk,
                        long long D, const long long *lens, int causal,
                        double scale, double *o, double *lse, int nthreads) {
  if (!q || !k || !v || !o || !lse || B < 1 || H < 1 || Sq < 1 || Sk < 1 ||
      D < 1)
    return ORACLE_EINVAL;
  if (!(scale > 0.0) || !isfinite(scale)) return ORACLE_EINVAL;
  if (lens)
    for (long long b = 0; b < B; ++b)
      if (lens[b] < 0 || lens[b] > Sk) return ORACLE_EINVAL;
  const long long total = B * H * Sq;
  if (nthreads < 1) nthreads = 1;
  if ((long long)nthreads > total) nthreads = (int)total;
  oracle_kv_job *jobs =
      (oracle_kv_job *)calloc((size_t)nthreads, sizeof(oracle_kv_job));
  pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  char *made = (char *)calloc((size_t)nthreads, 1);
  if (!jobs || !tid || !made) {
    free(jobs);
    free(tid);
    free(made);
    return ORACLE_ENOMEM;
  }
  int status = ORACLE_OK;
  for (int t = 0; t < nthreads; ++t) {
    oracle_kv_job *J = &jobs[t];
    J->q = q; J->k = k; J->v = v;
    J->lens = lens;
    J->H = H; J->Sq = Sq; J->Sk = Sk; J->D = D;
    J->causal = causal;
    J->scale = scale;
    J->o = o; J->lse = lse;
    J->r0 = total * t / nthreads;
    J->r1 = total * (t + 1) / nthreads;
    J->status = ORACLE_OK;
    if (nthreads > 1 && pthread_create(&tid[t], NULL, oracle_kv_worker, J) == 0)
      made[t] = 1;
    else
      oracle_kv_worker(J);
  }
  for (int t = 0; t < nthreads; ++t)
    if (made[t]) pthread_join(tid[t], NULL);
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].status != ORACLE_OK) status = jobs[t].status;
  free(jobs);
  free(tid);
  free(made);
  return status;
}
