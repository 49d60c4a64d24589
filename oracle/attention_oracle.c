/*
 * Attention oracle: plain, slow, fp64 CPU restatement of exact scaled-dot-product
 * attention and its gradients.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the benchmark's CPU-baseline leg may call it; the product path never
 * does.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (one attention head at a time, row-major [N, d] operands):
 *
 *   S_ij   = scale * sum_c q_ic k_jc              for visible (i, j)
 *   m_i    = max_j S_ij,   l_i = sum_j exp(S_ij - m_i)
 *   P_ij   = exp(S_ij - m_i) / l_i                ("softmax(x_i) = exp(x_i)/sum exp(x_j)")
 *   O_i    = sum_j P_ij v_j
 *   LSE_i  = m_i + ln l_i
 *
 * Sources: "FlashAttention: how a memory trick unlocked..." (khetwal.com),
 * section "The Quadratic Memory Bottleneck" (S = Q K^T, scaled; P = softmax(S);
 * O = P V), section "The Trick: Online Softmax" (the softmax definition), and the
 * "Standard Attention" listing of its worked example.  The scale factor follows
 * the first of those sections, where the score step is written with a scale
 * before the softmax.  The log-sum-exp output is the per-row softmax statistic
 * the galileo blog ("How FlashAttention Eliminates Transformer Memory
 * Bottlenecks", Innovation #3) says is the only thing kept for the backward pass;
 * the pages do not define it, so it is read as the natural log of the softmax
 * denominator including the row max.
 *
 * Backward pass: the pages give no formulas, so this is the chain rule applied
 * directly to the scalar L = sum_ic O_ic * dO_ic, written out term by term:
 *
 *   dP_ij = sum_c dO_ic v_jc
 *   D_i   = sum_j P_ij dP_ij                      (from P and dP, not from O)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_i dS_ij q_i
 *   dV_j  = sum_i P_ij dO_i
 *
 * Visibility of key j to query i (readings where the pages are silent):
 *   - key padding: j < kv_len;
 *   - causal: j <= i (queries and keys aligned at index 0);
 *   - block mask: block_mask[(i / tile) * n_tiles + (j / tile)] != 0, the
 *     tile-level mask of Innovation #5 ("skip tiles that correspond to zeroed-out
 *     blocks"), no element-level mask inside a kept tile.
 * A row that sees no key has O = 0, LSE = -inf and dQ = 0.
 *
 * Inputs are double precision (the bf16 or fp32 values the device path is given,
 * converted exactly); all arithmetic is in double precision.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
  const double *q, *k, *v, *dout;
  int N, d;
  double scale;
  int causal;
  int kv_len;
  const uint8_t *block_mask;
  int tile, n_tiles;
} head_t;

static int visible(const head_t *h, int i, int j) {
  if (j >= h->kv_len) return 0;
  if (h->causal && j > i) return 0;
  if (h->block_mask && !h->block_mask[(long)(i / h->tile) * h->n_tiles + (j / h->tile)]) return 0;
  return 1;
}

static double dot_rows(const double *a, const double *b, int d) {
  double acc = 0.0;
  for (int c = 0; c < d; ++c) acc += a[c] * b[c];
  return acc;
}

/* ---------------------------------------------------------------- thread pool */

typedef struct {
  void (*fn)(void *ctx, long item, double *scratch);
  void *ctx;
  long n_items;
  long next;
  long scratch_len;
  int failed;
} job_t;

static void *worker(void *arg) {
  job_t *job = (job_t *)arg;
  double *scratch = (double *)malloc(sizeof(double) * (size_t)(job->scratch_len > 0 ? job->scratch_len : 1));
  if (!scratch) {
    __atomic_store_n(&job->failed, 1, __ATOMIC_SEQ_CST);
    return NULL;
  }
  for (;;) {
    long item = __atomic_fetch_add(&job->next, 1, __ATOMIC_SEQ_CST);
    if (item >= job->n_items) break;
    job->fn(job->ctx, item, scratch);
  }
  free(scratch);
  return NULL;
}

static int run_parallel(job_t *job, int nthreads) {
  if (nthreads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = n > 0 ? (int)n : 1;
  }
  if (nthreads > 256) nthreads = 256;
  if ((long)nthreads > job->n_items) nthreads = (int)(job->n_items > 0 ? job->n_items : 1);
  job->next = 0;
  job->failed = 0;
  pthread_t tids[256];
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[started], NULL, worker, job) != 0) break;
    ++started;
  }
  worker(job);
  for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
  return job->failed ? -1 : 0;
}

/* ------------------------------------------------------------------ row pass */

typedef struct {
  head_t h;
  const int32_t *rows;
  double *o, *lse, *m, *l, *Dsum, *dq;
} rows_ctx;

static void row_item(void *vctx, long item, double *s) {
  rows_ctx *ctx = (rows_ctx *)vctx;
  const head_t *h = &ctx->h;
  const int N = h->N, d = h->d;
  const int i = ctx->rows[item];
  double *o = ctx->o + item * (long)d;
  double *dq = ctx->dq ? ctx->dq + item * (long)d : NULL;
  double *dp = s + N; /* second half of scratch: dP_ij */
  const double *qi = h->q + (long)i * d;

  /* scores and the row max over visible keys */
  double m = -INFINITY;
  int n_visible = 0;
  for (int j = 0; j < N; ++j) {
    if (!visible(h, i, j)) continue;
    s[j] = h->scale * dot_rows(qi, h->k + (long)j * d, d);
    if (s[j] > m) m = s[j];
    ++n_visible;
  }
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  if (dq)
    for (int c = 0; c < d; ++c) dq[c] = 0.0;
  if (n_visible == 0) {
    ctx->lse[item] = -INFINITY;
    if (ctx->m) ctx->m[item] = -INFINITY;
    if (ctx->l) ctx->l[item] = 0.0;
    if (ctx->Dsum) ctx->Dsum[item] = 0.0;
    return;
  }
  /* softmax denominator */
  double l = 0.0;
  for (int j = 0; j < N; ++j)
    if (visible(h, i, j)) l += exp(s[j] - m);
  /* O_i = sum_j P_ij v_j */
  for (int j = 0; j < N; ++j) {
    if (!visible(h, i, j)) continue;
    const double p = exp(s[j] - m) / l;
    const double *vj = h->v + (long)j * d;
    for (int c = 0; c < d; ++c) o[c] += p * vj[c];
  }
  ctx->lse[item] = m + log(l);
  if (ctx->m) ctx->m[item] = m;
  if (ctx->l) ctx->l[item] = l;
  if (!h->dout) return;

  /* backward quantities of this row */
  const double *doi = h->dout + (long)i * d;
  double D = 0.0;
  for (int j = 0; j < N; ++j) {
    if (!visible(h, i, j)) continue;
    const double p = exp(s[j] - m) / l;
    dp[j] = dot_rows(doi, h->v + (long)j * d, d);
    D += p * dp[j];
  }
  if (ctx->Dsum) ctx->Dsum[item] = D;
  if (!dq) return;
  for (int j = 0; j < N; ++j) {
    if (!visible(h, i, j)) continue;
    const double p = exp(s[j] - m) / l;
    const double ds = p * (dp[j] - D);
    const double *kj = h->k + (long)j * d;
    for (int c = 0; c < d; ++c) dq[c] += h->scale * ds * kj[c];
  }
}

/* --------------------------------------------------------------- column pass */

typedef struct {
  head_t h;
  const int32_t *cols;
  const double *m, *l, *Dsum; /* per-row statistics, indexed by query row (length N) */
  double *dk, *dv;
} cols_ctx;

static void col_item(void *vctx, long item, double *unused) {
  (void)unused;
  cols_ctx *ctx = (cols_ctx *)vctx;
  const head_t *h = &ctx->h;
  const int N = h->N, d = h->d;
  const int j = ctx->cols[item];
  double *dk = ctx->dk + item * (long)d;
  double *dv = ctx->dv + item * (long)d;
  for (int c = 0; c < d; ++c) dk[c] = dv[c] = 0.0;
  const double *kj = h->k + (long)j * d;
  const double *vj = h->v + (long)j * d;
  for (int i = 0; i < N; ++i) {
    if (!visible(h, i, j)) continue;
    if (!(ctx->l[i] > 0.0)) continue;
    const double *qi = h->q + (long)i * d;
    const double *doi = h->dout + (long)i * d;
    const double sij = h->scale * dot_rows(qi, kj, d);
    const double p = exp(sij - ctx->m[i]) / ctx->l[i];
    const double dpij = dot_rows(doi, vj, d);
    const double ds = p * (dpij - ctx->Dsum[i]);
    for (int c = 0; c < d; ++c) {
      dv[c] += p * doi[c];
      dk[c] += h->scale * ds * qi[c];
    }
  }
}

/* ------------------------------------------------------------------- C ABI */

static int fill_head(head_t *h, const double *q, const double *k, const double *v, const double *dout,
                     int N, int d, double scale, int causal, int kv_len,
                     const uint8_t *block_mask, int tile) {
  if (N <= 0 || d <= 0 || !q || !k || !v) return -1;
  if (block_mask && tile <= 0) return -1;
  h->q = q; h->k = k; h->v = v; h->dout = dout;
  h->N = N; h->d = d; h->scale = scale; h->causal = causal;
  h->kv_len = (kv_len < 0 || kv_len > N) ? N : kv_len;
  h->block_mask = block_mask;
  h->tile = tile > 0 ? tile : 1;
  h->n_tiles = (N + h->tile - 1) / h->tile;
  return 0;
}

/* Per-row pass for the query rows rows[0..nrows) of one head.
 * Outputs are indexed by position in `rows`: o[nrows*d], lse, m, l, Dsum [nrows],
 * dq[nrows*d].  dout, m, l, Dsum and dq may be NULL (forward only).
 * kv_len < 0 means "no key padding"; kv_len = 0 means no key is visible.
 * Returns 0 on success. */
int oracle_rows(const double *q, const double *k, const double *v, const double *dout,
                int N, int d, double scale, int causal, int kv_len,
                const uint8_t *block_mask, int tile,
                const int32_t *rows, int nrows,
                double *o, double *lse, double *m, double *l, double *Dsum, double *dq,
                int nthreads) {
  rows_ctx ctx;
  memset(&ctx, 0, sizeof(ctx));
  if (fill_head(&ctx.h, q, k, v, dout, N, d, scale, causal, kv_len, block_mask, tile)) return -1;
  if (!rows || nrows < 0 || !o || !lse) return -1;
  for (int r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return -1;
  ctx.rows = rows;
  ctx.o = o; ctx.lse = lse; ctx.m = m; ctx.l = l; ctx.Dsum = Dsum; ctx.dq = dout ? dq : NULL;
  job_t job = {row_item, &ctx, nrows, 0, 2L * N, 0};
  return run_parallel(&job, nthreads);
}

/* Per-column pass for the keys cols[0..ncols) of one head.  m, l and Dsum are
 * the row statistics of every query row that sees one of those keys (arrays of
 * length N indexed by query row, as written by oracle_rows over those rows).
 * Outputs dk[ncols*d], dv[ncols*d] are indexed by position in `cols`. */
int oracle_cols(const double *q, const double *k, const double *v, const double *dout,
                int N, int d, double scale, int causal, int kv_len,
                const uint8_t *block_mask, int tile,
                const double *m, const double *l, const double *Dsum,
                const int32_t *cols, int ncols, double *dk, double *dv, int nthreads) {
  cols_ctx ctx;
  memset(&ctx, 0, sizeof(ctx));
  if (fill_head(&ctx.h, q, k, v, dout, N, d, scale, causal, kv_len, block_mask, tile)) return -1;
  if (!dout || !m || !l || !Dsum || !cols || ncols < 0 || !dk || !dv) return -1;
  for (int c = 0; c < ncols; ++c)
    if (cols[c] < 0 || cols[c] >= N) return -1;
  ctx.cols = cols; ctx.m = m; ctx.l = l; ctx.Dsum = Dsum; ctx.dk = dk; ctx.dv = dv;
  job_t job = {col_item, &ctx, ncols, 0, 1, 0};
  return run_parallel(&job, nthreads);
}

/* Number of worker threads a call with nthreads <= 0 uses. */
int oracle_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)(n > 256 ? 256 : n) : 1;
}
