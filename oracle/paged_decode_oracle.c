/*
 * Paged decode attention: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg may load this file's library.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * What it computes, for every sequence s, query token i in [0, M) and query
 * head hq (definitions from the decode semantics of the pages):
 *
 *   h    = hq / G, G = Hq / Hkv        contiguous GQA groups: the rows of a
 *                                      kv head are gqa * M query rows
 *                                      (rocm_rdna_hip, KernelVariant.rows_padded)
 *   n_i  = L_s - M + i + 1             keys row i sees: seq_len includes the
 *                                      M query tokens, and query i of a
 *                                      request sees K length
 *                                      seq_len - q_len + i + 1
 *                                      (rocm_octave_attn, _fill_query_maps)
 *   keys k in [lo, n_i), lo = window ? max(0, n_i - window) : 0
 *                                      window counted in keys, 0 = full
 *                                      causal (rocm_rdna_hip, KernelVariant
 *                                      "window"); the first key of query
 *                                      `first` is context + first - window + 1
 *                                      (rocm_rdna_hip, plan_prefill)
 *   K_k  = K[block_table[s][k / P]][k % P][h][:]   (paged gather)
 *   x_k  = scale * sum_d q[d] K_k[d]
 *   o    = sum_k softmax(x)_k V_k     (max subtracted, all in fp64)
 *   o    = 0 when no key is visible   (padding queries get K length 0,
 *                                      rocm_octave_attn, _fill_query_maps)
 *
 * With variable query lengths (rocm_octave_attn, _fill_query_maps) the rows
 * are the tokens t of a batch described by query_start[0..S]: the request of
 * t is the number of entries query_start[1..S] that are <= t (a right-sided
 * search), its q_len is query_start[r+1] - query_start[r], and t sees
 * K length L_r - q_len + (t - query_start[r]) + 1; a token at or past
 * query_start[S] belongs to no request and gets K length 0.
 *
 * Inputs are the raw 16-bit fp16/bf16 words; they are widened to double
 * exactly (IEEE binary16 / bfloat16 definitions below), so the oracle sees
 * exactly the values the GPU reads.  The cache is addressed through four
 * strides (page, token, kv head, d), so NHD, HND and the packed K|V cache
 * are all the same code: only the strides differ.
 *
 * Parity of this oracle against the pages themselves is pinned by closed
 * forms, invariants and a library routine (see tests), not by printed
 * values: the pages print none for this kernel.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(f | 0x400), e - 25); /* (1 + f/2^10) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

typedef struct {
  const uint16_t *q;
  int64_t q_s0, q_s1, q_s2; /* q[t][hq][d] */
  const uint16_t *k, *v;
  int64_t kv_sp, kv_st, kv_sh, kv_sd; /* K[page][token][kv head][d] */
  const int32_t *block_table;
  int64_t bt_stride, bt_width;
  const int32_t *seq_lens;
  int num_seqs, is_bf16, Hq, Hkv, D, P, M, window;
  double scale;
  const int32_t *qsl; /* query_start [S + 1], or NULL: token t = s * M + i */
} pdo_args;

static double widen(const pdo_args *a, uint16_t w) {
  return a->is_bf16 ? bf16_to_double(w) : half_to_double(w);
}

/* The request s of query row t and the keys [lo, hi) it sees; 0 when t
 * belongs to no request (then it sees no key). */
static int visible_range(const pdo_args *a, int64_t t, int *s_out, int64_t *lo, int64_t *hi) {
  int64_t n;
  int s;
  *lo = 0;
  *hi = 0;
  if (a->qsl) {
    /* right-sided search of t in query_start[1..S] */
    int lo_i = 0, hi_i = a->num_seqs;
    while (lo_i < hi_i) {
      int mid = (lo_i + hi_i) / 2;
      if (a->qsl[mid + 1] <= t)
        lo_i = mid + 1;
      else
        hi_i = mid;
    }
    s = lo_i;
    if (s >= a->num_seqs) return 0;
    int64_t q_len = (int64_t)a->qsl[s + 1] - a->qsl[s];
    n = (int64_t)a->seq_lens[s] - q_len + (t - a->qsl[s]) + 1;
  } else {
    s = (int)(t / a->M);
    n = (int64_t)a->seq_lens[s] - a->M + (t % a->M) + 1;
  }
  *s_out = s;
  if (n < 0) n = 0;
  *hi = n;
  if (a->window > 0 && n - a->window > 0) *lo = n - a->window;
  return 1;
}

static const uint16_t *key_row(const pdo_args *a, const uint16_t *base, int s, int64_t k, int h) {
  int64_t page = k / a->P;
  int64_t tok = k % a->P;
  int64_t phys = a->block_table[(int64_t)s * a->bt_stride + page];
  return base + phys * a->kv_sp + tok * a->kv_st + (int64_t)h * a->kv_sh;
}

/*
 * Unnormalised partial over keys [klo, khi) intersected with the row's
 * visible range: m = max logit, l = sum exp(x - m), acc = sum exp(x - m) V.
 * An empty range gives m = -inf, l = 0, acc = 0.
 */
static void row_partial(const pdo_args *a, int64_t t, int hq, int64_t klo, int64_t khi,
                        double *x /* scratch, >= khi-klo */, double *acc, double *m_out,
                        double *l_out) {
  int G = a->Hq / a->Hkv;
  int h = hq / G;
  int s = 0;
  int64_t lo, hi;
  visible_range(a, t, &s, &lo, &hi);
  if (klo > lo) lo = klo;
  if (khi < hi) hi = khi;
  for (int d = 0; d < a->D; ++d) acc[d] = 0.0;
  *m_out = -INFINITY;
  *l_out = 0.0;
  if (hi <= lo) return;
  const uint16_t *qrow = a->q + t * a->q_s0 + (int64_t)hq * a->q_s1;
  double m = -INFINITY;
  for (int64_t k = lo; k < hi; ++k) {
    const uint16_t *kr = key_row(a, a->k, s, k, h);
    double dot = 0.0;
    for (int d = 0; d < a->D; ++d)
      dot += widen(a, qrow[d * a->q_s2]) * widen(a, kr[d * a->kv_sd]);
    x[k - lo] = a->scale * dot;
    if (x[k - lo] > m) m = x[k - lo];
  }
  double l = 0.0;
  for (int64_t k = lo; k < hi; ++k) {
    double p = exp(x[k - lo] - m);
    l += p;
    const uint16_t *vr = key_row(a, a->v, s, k, h);
    for (int d = 0; d < a->D; ++d) acc[d] += p * widen(a, vr[d * a->kv_sd]);
  }
  *m_out = m;
  *l_out = l;
}

typedef struct {
  const pdo_args *a;
  const int64_t *sel; /* output rows as t * Hq + hq, or NULL for all */
  int64_t nrows, begin, end;
  int64_t klo, khi;   /* key restriction (partial mode) */
  int partial;
  double *out, *m, *l;
  int status;
} pdo_job;

static void *pdo_worker(void *p) {
  pdo_job *j = (pdo_job *)p;
  const pdo_args *a = j->a;
  int64_t maxkeys = 1;
  for (int s = 0; s < a->num_seqs; ++s)
    if (a->seq_lens[s] > maxkeys) maxkeys = a->seq_lens[s];
  double *x = (double *)malloc(sizeof(double) * (size_t)maxkeys);
  double *acc = (double *)malloc(sizeof(double) * (size_t)a->D);
  if (!x || !acc) {
    free(x);
    free(acc);
    j->status = -1;
    return NULL;
  }
  for (int64_t r = j->begin; r < j->end; ++r) {
    int64_t id = j->sel ? j->sel[r] : r;
    int64_t t = id / a->Hq;
    int hq = (int)(id % a->Hq);
    double m, l;
    row_partial(a, t, hq, j->klo, j->khi, x, acc, &m, &l);
    double *o = j->out + r * a->D;
    if (j->partial) {
      for (int d = 0; d < a->D; ++d) o[d] = acc[d];
      j->m[r] = m;
      j->l[r] = l;
    } else {
      for (int d = 0; d < a->D; ++d) o[d] = (l > 0.0) ? acc[d] / l : 0.0;
    }
  }
  free(x);
  free(acc);
  j->status = 0;
  return NULL;
}

static int run(const pdo_args *a, const int64_t *sel, int64_t nrows, int64_t klo, int64_t khi,
               int partial, double *out, double *m, double *l, int nthreads) {
  if (a->Hkv <= 0 || a->Hq % a->Hkv != 0 || a->D <= 0 || a->P <= 0 || a->M <= 0) return -1;
  for (int s = 0; s < a->num_seqs; ++s) {
    int64_t L = a->seq_lens[s];
    if (L > a->bt_width * (int64_t)a->P) return -2; /* would index past the block table */
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nrows) nthreads = (int)(nrows > 0 ? nrows : 1);
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  pdo_job *jobs = (pdo_job *)calloc((size_t)nthreads, sizeof(pdo_job));
  if (!th || !jobs) {
    free(th);
    free(jobs);
    return -3;
  }
  int rc = 0;
  for (int w = 0; w < nthreads; ++w) {
    pdo_job *j = &jobs[w];
    j->a = a;
    j->sel = sel;
    j->nrows = nrows;
    j->begin = nrows * w / nthreads;
    j->end = nrows * (w + 1) / nthreads;
    j->klo = klo;
    j->khi = khi;
    j->partial = partial;
    j->out = out;
    j->m = m;
    j->l = l;
    if (w > 0 && pthread_create(&th[w], NULL, pdo_worker, j) != 0) {
      pdo_worker(j); /* no thread available: do it here */
      th[w] = 0;
    }
  }
  pdo_worker(&jobs[0]);
  for (int w = 1; w < nthreads; ++w)
    if (th[w]) pthread_join(th[w], NULL);
  for (int w = 0; w < nthreads; ++w)
    if (jobs[w].status != 0) rc = -3;
  free(th);
  free(jobs);
  return rc;
}

#define PDO_ARGS_FROM_PARAMS                                                              \
  pdo_args a;                                                                             \
  a.q = q; a.q_s0 = q_s0; a.q_s1 = q_s1; a.q_s2 = q_s2;                                   \
  a.k = k; a.v = v; a.kv_sp = kv_sp; a.kv_st = kv_st; a.kv_sh = kv_sh; a.kv_sd = kv_sd;   \
  a.block_table = block_table; a.bt_stride = bt_stride; a.bt_width = bt_width;            \
  a.seq_lens = seq_lens; a.num_seqs = num_seqs; a.is_bf16 = is_bf16;                      \
  a.Hq = num_q_heads; a.Hkv = num_kv_heads; a.D = head_size; a.P = page_size;            \
  a.M = max_query_len; a.window = window; a.scale = scale; a.qsl = NULL;

/* Full outputs: out[r][d] for the selected rows (or all S*M*Hq rows). */
int pdo_attention(const uint16_t *q, int64_t q_s0, int64_t q_s1, int64_t q_s2,
                  const uint16_t *k, const uint16_t *v, int64_t kv_sp, int64_t kv_st,
                  int64_t kv_sh, int64_t kv_sd, const int32_t *block_table, int64_t bt_stride,
                  int64_t bt_width, const int32_t *seq_lens, int num_seqs, int is_bf16,
                  int num_q_heads, int num_kv_heads, int head_size, int page_size,
                  int max_query_len, int window, double scale, const int64_t *sel, int64_t nsel,
                  double *out, int nthreads) {
  PDO_ARGS_FROM_PARAMS
  int64_t nrows = sel ? nsel : (int64_t)num_seqs * max_query_len * num_q_heads;
  return run(&a, sel, nrows, 0, INT64_MAX, 0, out, NULL, NULL, nthreads);
}

/* Full outputs of a batch with variable query lengths: rows t in
 * [0, num_tokens) described by query_start[0..num_seqs] (non-decreasing). */
int pdo_attention_varlen(const uint16_t *q, int64_t q_s0, int64_t q_s1, int64_t q_s2,
                         const uint16_t *k, const uint16_t *v, int64_t kv_sp, int64_t kv_st,
                         int64_t kv_sh, int64_t kv_sd, const int32_t *block_table,
                         int64_t bt_stride, int64_t bt_width, const int32_t *seq_lens,
                         int num_seqs, int is_bf16, int num_q_heads, int num_kv_heads,
                         int head_size, int page_size, int max_query_len, int window,
                         double scale, const int32_t *query_start, int64_t num_tokens,
                         const int64_t *sel, int64_t nsel, double *out, int nthreads) {
  PDO_ARGS_FROM_PARAMS
  a.qsl = query_start;
  for (int s = 0; s < num_seqs; ++s)
    if (query_start[s + 1] < query_start[s] || query_start[s] < 0) return -4;
  int64_t nrows = sel ? nsel : num_tokens * num_q_heads;
  return run(&a, sel, nrows, 0, INT64_MAX, 0, out, NULL, NULL, nthreads);
}

/* Unnormalised partials (acc, m, l) over keys [key_lo, key_hi). */
int pdo_partial(const uint16_t *q, int64_t q_s0, int64_t q_s1, int64_t q_s2, const uint16_t *k,
                const uint16_t *v, int64_t kv_sp, int64_t kv_st, int64_t kv_sh, int64_t kv_sd,
                const int32_t *block_table, int64_t bt_stride, int64_t bt_width,
                const int32_t *seq_lens, int num_seqs, int is_bf16, int num_q_heads,
                int num_kv_heads, int head_size, int page_size, int max_query_len, int window,
                double scale, int64_t key_lo, int64_t key_hi, double *acc, double *m, double *l,
                int nthreads) {
  PDO_ARGS_FROM_PARAMS
  int64_t nrows = (int64_t)num_seqs * max_query_len * num_q_heads;
  return run(&a, NULL, nrows, key_lo, key_hi, 1, acc, m, l, nthreads);
}

/* The exact widening used above, exposed so tests can pin it. */
double pdo_widen(uint16_t w, int is_bf16) {
  return is_bf16 ? bf16_to_double(w) : half_to_double(w);
}
