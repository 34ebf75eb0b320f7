/*
 * ssd_oracle.c -- plain, slow, float64 CPU oracle for sparse self-speculative decoding attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the benchmark's CPU
 * baseline may load or run this code; the product path never does.  It shares no code, header,
 * table or helper with the CUDA library: it reads the same input bytes and recomputes every
 * result from the plain definitions below, one (request, KV head) unit at a time.
 *
 * Sources (page title, section):
 *  [SS]  "Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with Sparse
 *        Attention" (SparseSpec / PillarAttn).  §4.1: verification runs full attention for the
 *        candidates, its attention scores are dumped, reduced over the query heads of a GQA group
 *        and the verify positions, and Top-K of them is the sparse pattern the next k drafts use.
 *        §4.2: sparse and full attention share one PagedAttention pipeline (page size 1 = a token
 *        list).  §2.3: a verify step checks k drafted tokens plus one bonus position.
 *  [SA]  "SpecAttn: Co-Designing Sparse Attention with Self-Speculative Decoding", abstract: the
 *        criticality of each KV entry is a byproduct of verification.
 *  [SSA] "SpecSA" forum post, "overlap-aware grouped query execution": candidates that share KV
 *        blocks execute together over the shared blocks.
 *  [SD]  "SparDA: Sparse Decoupled Attention ...", §2 training strategy: fine scores are max-pooled
 *        to the coarser selection grid.
 *  [SSR] "SpecSA" forum post, "refresh/reuse NSA kernel fusion" and "branch handling": the KV of
 *        accepted tokens is kept for later queries and the KV of rejected tokens is dropped.
 *
 * Readings of points the pages leave open (each one is listed in the design notes as well):
 *  R1  Request b holds L_b tokens including its n_c = k+1 candidates at positions L_b-n_c .. L_b-1.
 *      Candidate i (0-based) sees tokens t <= L_b - n_c + i (causal among the candidates).
 *  R2  Logits are scale * q.k with natural-base softmax; no soft-cap.
 *  R3  Criticality is the softmax probability SUMMED (not averaged) over the G query heads of the
 *      group and all n_c verify positions.  A constant factor, so the Top-K ranking is unchanged.
 *  R4  Top-K keeps the K largest scores; equal scores are broken toward the lower index; the kept
 *      indices are returned in ascending order.
 *  R5  The draft attends exactly the given index list (softmax over it, no causal mask).
 *  R6  Block mode: per-candidate criticality (summed over the G heads only) max-pooled over
 *      block_size tokens; each candidate keeps its own top blocks; the union of a group's candidate
 *      block sets is loaded once, and candidate i attends only its own blocks (causal as R1).
 *  R7  An empty token set gives output 0 and lse = -inf.
 *  R9  Phase assignment ([SS] §4.2, workload-aware scheduling): there is one bucket per phase offset
 *      (n_buckets = k+1: k draft steps and the verify); an arriving request joins the bucket with the
 *      fewest live requests, ties to the lowest offset.  At step s a request with offset o is in
 *      phase (s + o) mod n_buckets; the last phase (n_buckets - 1) is its verify, the others drafts.
 *  R10 Top-p (variable K): a row keeps the smallest number K of its largest entries (ties toward
 *      the lower index) whose sum reaches p times the row's total, both sums in double precision,
 *      the prefix taken in that descending order; K = 0 when p times the total is not positive;
 *      K is capped at k_max.  The kept set is then exactly the Top-K set of R4 with that K.
 *  R8  KV append writes token j of request b (its K and V rows for every KV head) at position
 *      seq_lens[b] + j through the page table; a position at or past max_seq_len, or a page id
 *      outside the pool, skips the request (nothing of it is written).  Advancing adds delta[b] to
 *      seq_lens[b]; a result outside [0, max_seq_len] leaves it unchanged.  Accepting a of the n_c
 *      candidates of a verify is an advance by -(n_c - a): the rejected candidates' KV stays in the
 *      pages but lies past the request's length.
 *
 * Element types: 0 = float32, 1 = bfloat16 (converted exactly to double).
 * KV pool layout [num_pages][2][h_kv][page_size][d]; index 0 = K, 1 = V.
 * All functions return 0 on success and a negative code on invalid input.
 */
#define _POSIX_C_SOURCE 200809L
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_OK = 0, ORC_EARG = -1, ORC_EPAGE = -2, ORC_EIDX = -3, ORC_ENOMEM = -4, ORC_EKMAX = -5 };

static double orc_elem(const void *base, int64_t i, int dtype) {
  if (dtype == ORC_F32) return (double)((const float *)base)[i];
  uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

typedef struct {
  const void *pool;
  int dtype;
  int64_t num_pages;
  int page_size;
  int h_kv;
  int d;
  const int32_t *page_table;
  int max_pages;
  const int32_t *seq_lens;
  int batch;
} orc_kv;

/* [SS] §4.2 PagedAttention: token t of request b is slot t % page_size of page
 * page_table[b][t / page_size].  Writes the element offset of row (K or V, head g, token t). */
static int orc_row(const orc_kv *kv, int b, int which, int g, int t, int64_t *off) {
  int j = t / kv->page_size;
  if (t < 0 || j >= kv->max_pages) return ORC_EPAGE;
  int32_t p = kv->page_table[(int64_t)b * kv->max_pages + j];
  if (p < 0 || (int64_t)p >= kv->num_pages) return ORC_EPAGE;
  *off = ((((int64_t)p * 2 + which) * kv->h_kv + g) * kv->page_size + (t % kv->page_size)) * kv->d;
  return ORC_OK;
}

/* Plain dot product of a query row (element offset qoff in q) with the K row of token t. */
static int orc_logit(const orc_kv *kv, const void *q, int qdtype, int64_t qoff, int b, int g, int t,
                     double scale, double *s) {
  int64_t off;
  int rc = orc_row(kv, b, 0, g, t, &off);
  if (rc) return rc;
  double acc = 0.0;
  for (int k = 0; k < kv->d; ++k) acc += orc_elem(q, qoff + k, qdtype) * orc_elem(kv->pool, off + k, kv->dtype);
  *s = scale * acc;
  return ORC_OK;
}

/* Softmax attention of one query row over an explicit token list (tokens[0..n)).  Writes out[d]
 * (= sum_j p_j V_{t_j}), *lse, and, when p_out != NULL, the probabilities p_out[j].  [SS] §4.2:
 * full and sparse attention are the same computation over different token lists. */
static int orc_attend(const orc_kv *kv, const void *q, int qdtype, int64_t qoff, int b, int g,
                      const int32_t *tokens, int n, double scale, double *s_buf, double *out,
                      double *lse, double *p_out) {
  for (int k = 0; k < kv->d; ++k) out[k] = 0.0;
  if (n == 0) {
    *lse = -INFINITY; /* R7 */
    return ORC_OK;
  }
  double m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    int rc = orc_logit(kv, q, qdtype, qoff, b, g, tokens[j], scale, &s_buf[j]);
    if (rc) return rc;
    if (s_buf[j] > m) m = s_buf[j];
  }
  double z = 0.0;
  for (int j = 0; j < n; ++j) z += exp(s_buf[j] - m);
  for (int j = 0; j < n; ++j) {
    double p = exp(s_buf[j] - m) / z;
    if (p_out) p_out[j] = p;
    int64_t off;
    int rc = orc_row(kv, b, 1, g, tokens[j], &off);
    if (rc) return rc;
    for (int k = 0; k < kv->d; ++k) out[k] += p * orc_elem(kv->pool, off + k, kv->dtype);
  }
  *lse = m + log(z);
  return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* A tiny thread pool: units 0..n_units-1 are handed out round-robin to nthreads workers.     */
/* ------------------------------------------------------------------------------------------ */
typedef int (*orc_unit_fn)(void *ctx, int unit, void *scratch);
typedef struct {
  orc_unit_fn fn;
  void *ctx;
  int n_units, stride, first;
  size_t scratch_bytes;
  int rc;
} orc_job;

static void *orc_worker(void *arg) {
  orc_job *job = (orc_job *)arg;
  void *scratch = job->scratch_bytes ? malloc(job->scratch_bytes) : NULL;
  if (job->scratch_bytes && !scratch) {
    job->rc = ORC_ENOMEM;
    return NULL;
  }
  for (int u = job->first; u < job->n_units; u += job->stride) {
    int rc = job->fn(job->ctx, u, scratch);
    if (rc) {
      job->rc = rc;
      break;
    }
  }
  free(scratch);
  return NULL;
}

static int orc_run(orc_unit_fn fn, void *ctx, int n_units, int nthreads, size_t scratch_bytes) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > n_units) nthreads = n_units > 0 ? n_units : 1;
  orc_job *jobs = (orc_job *)calloc((size_t)nthreads, sizeof(orc_job));
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return ORC_ENOMEM;
  }
  for (int i = 0; i < nthreads; ++i) {
    jobs[i] = (orc_job){fn, ctx, n_units, nthreads, i, scratch_bytes, 0};
    if (i > 0) pthread_create(&th[i], NULL, orc_worker, &jobs[i]);
  }
  orc_worker(&jobs[0]);
  int rc = jobs[0].rc;
  for (int i = 1; i < nthreads; ++i) {
    pthread_join(th[i], NULL);
    if (jobs[i].rc && !rc) rc = jobs[i].rc;
  }
  free(jobs);
  free(th);
  return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* Verify: full attention of the n_c candidates + criticality.                                 */
/* ------------------------------------------------------------------------------------------ */
typedef struct {
  orc_kv kv;
  const void *q;
  int qdtype, h_q, n_c;
  double scale;
  double *out, *lse, *crit, *crit_cand;
  int64_t crit_stride;
} orc_verify_ctx;

/* One (request b, KV head g) unit.  [SS] §4.1 with R1-R3: for every candidate i and query head h of
 * group g, softmax over tokens 0..L-n_c+i; the probabilities summed over (h, i) are crit[b,g,t],
 * summed over h alone they are crit_cand[b,g,i,t]. */
static int orc_verify_unit(void *vctx, int unit, void *scratch) {
  orc_verify_ctx *c = (orc_verify_ctx *)vctx;
  const orc_kv *kv = &c->kv;
  int b = unit / kv->h_kv, g = unit % kv->h_kv;
  int G = c->h_q / kv->h_kv, L = kv->seq_lens[b], d = kv->d;
  if (L < c->n_c || (int64_t)L > c->crit_stride) return ORC_EARG;
  double *s_buf = (double *)scratch;
  double *p = s_buf + L;
  int32_t *tokens = (int32_t *)(p + L);
  double *crit = c->crit ? c->crit + ((int64_t)b * kv->h_kv + g) * c->crit_stride : NULL;
  if (crit)
    for (int t = 0; t < L; ++t) crit[t] = 0.0;
  for (int t = 0; t < L; ++t) tokens[t] = t;
  for (int i = 0; i < c->n_c; ++i) {
    int last = L - c->n_c + i; /* R1 */
    double *cc = c->crit_cand
                     ? c->crit_cand + (((int64_t)b * kv->h_kv + g) * c->n_c + i) * c->crit_stride
                     : NULL;
    if (cc)
      for (int t = 0; t < L; ++t) cc[t] = 0.0;
    for (int hl = 0; hl < G; ++hl) {
      int h = g * G + hl; /* query head h reads KV head h / G */
      int64_t row = ((int64_t)b * c->n_c + i) * c->h_q + h;
      int rc = orc_attend(kv, c->q, c->qdtype, row * d, b, g, tokens, last + 1, c->scale, s_buf,
                          c->out + row * d, &c->lse[row], p);
      if (rc) return rc;
      for (int t = 0; t <= last; ++t) {
        if (crit) crit[t] += p[t];
        if (cc) cc[t] += p[t];
      }
    }
  }
  return ORC_OK;
}

int oracle_verify(const void *pool, int dtype, int64_t num_pages, int page_size, int h_kv, int d,
                  const int32_t *page_table, int max_pages, const int32_t *seq_lens, int batch,
                  const void *q, int qdtype, int h_q, int n_c, double scale, double *out,
                  double *lse, double *crit, double *crit_cand, int64_t crit_stride, int nthreads) {
  if (!pool || !page_table || !seq_lens || !q || !out || !lse || h_kv <= 0 || h_q % h_kv || n_c < 1 ||
      batch < 0 || d <= 0 || page_size <= 0)
    return ORC_EARG;
  int Lmax = 0;
  for (int b = 0; b < batch; ++b) Lmax = seq_lens[b] > Lmax ? seq_lens[b] : Lmax;
  orc_verify_ctx c = {{pool, dtype, num_pages, page_size, h_kv, d, page_table, max_pages, seq_lens, batch},
                      q, qdtype, h_q, n_c, scale, out, lse, crit, crit_cand, crit_stride};
  size_t scratch = (size_t)Lmax * (sizeof(int32_t) + 2 * sizeof(double)) + 64;
  return orc_run(orc_verify_unit, &c, batch * h_kv, nthreads, scratch);
}

/* ------------------------------------------------------------------------------------------ */
/* Draft: single-query sparse attention over the selected tokens.                               */
/* ------------------------------------------------------------------------------------------ */
typedef struct {
  orc_kv kv;
  const void *q;
  int qdtype, h_q;
  const int32_t *idx, *cnt;
  int k_max;
  double scale;
  double *out, *lse;
} orc_draft_ctx;

/* [SS] §4.1: the k drafts after a verify attend only the selected tokens; R5. */
static int orc_draft_unit(void *vctx, int unit, void *scratch) {
  orc_draft_ctx *c = (orc_draft_ctx *)vctx;
  const orc_kv *kv = &c->kv;
  int b = unit / kv->h_kv, g = unit % kv->h_kv, G = c->h_q / kv->h_kv, L = kv->seq_lens[b];
  int n = c->cnt[(int64_t)b * kv->h_kv + g];
  if (n < 0 || n > c->k_max) return ORC_EARG;
  const int32_t *tok = c->idx + ((int64_t)b * kv->h_kv + g) * c->k_max;
  for (int j = 0; j < n; ++j)
    if (tok[j] < 0 || tok[j] >= L) return ORC_EIDX;
  for (int hl = 0; hl < G; ++hl) {
    int64_t row = (int64_t)b * c->h_q + g * G + hl;
    int rc = orc_attend(kv, c->q, c->qdtype, row * kv->d, b, g, tok, n, c->scale, (double *)scratch,
                        c->out + row * kv->d, &c->lse[row], NULL);
    if (rc) return rc;
  }
  return ORC_OK;
}

int oracle_draft(const void *pool, int dtype, int64_t num_pages, int page_size, int h_kv, int d,
                 const int32_t *page_table, int max_pages, const int32_t *seq_lens, int batch,
                 const void *q, int qdtype, int h_q, const int32_t *idx, int k_max, const int32_t *cnt,
                 double scale, double *out, double *lse, int nthreads) {
  if (!pool || !page_table || !seq_lens || !q || !idx || !cnt || !out || !lse || h_kv <= 0 ||
      h_q % h_kv || k_max < 0)
    return ORC_EARG;
  orc_draft_ctx c = {{pool, dtype, num_pages, page_size, h_kv, d, page_table, max_pages, seq_lens, batch},
                     q, qdtype, h_q, idx, cnt, k_max, scale, out, lse};
  return orc_run(orc_draft_unit, &c, batch * h_kv, nthreads, (size_t)(k_max + 1) * sizeof(double));
}

/* ------------------------------------------------------------------------------------------ */
/* Top-K selection.                                                                            */
/* ------------------------------------------------------------------------------------------ */
typedef struct {
  float v;
  int32_t i;
} orc_pair;

/* Larger score first; equal scores: lower index first (R4). */
static int orc_cmp_desc(const void *a, const void *b) {
  const orc_pair *x = (const orc_pair *)a, *y = (const orc_pair *)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i > y->i) - (x->i < y->i);
}

static int orc_cmp_int(const void *a, const void *b) {
  int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return (x > y) - (x < y);
}

/* [SS] §4.1 "apply Top-K on the dumped scores".  Row r has length ceil(lens[r/rows_per_group] /
 * len_div) and keeps min(ks[r/rows_per_group], length) entries, chosen by a full sort of
 * (score desc, index asc) and returned in ascending index order, -1 padded to k_max. */
int oracle_topk(const float *scores, int64_t stride, const int32_t *lens, const int32_t *ks,
                int n_groups, int rows_per_group, int len_div, int32_t *idx, int k_max, int32_t *cnt) {
  if (!scores || !lens || !ks || !idx || !cnt || rows_per_group <= 0 || len_div <= 0 || k_max < 0)
    return ORC_EARG;
  int64_t n_rows = (int64_t)n_groups * rows_per_group;
  for (int64_t r = 0; r < n_rows; ++r) {
    int grp = (int)(r / rows_per_group);
    int n = (lens[grp] + len_div - 1) / len_div;
    int k = ks[grp] < n ? ks[grp] : n;
    if (n < 0 || k < 0 || (int64_t)n > stride) return ORC_EARG;
    if (k > k_max) return ORC_EKMAX;
    orc_pair *pairs = (orc_pair *)malloc((size_t)(n > 0 ? n : 1) * sizeof(orc_pair));
    if (!pairs) return ORC_ENOMEM;
    for (int t = 0; t < n; ++t) {
      float v = scores[r * stride + t];
      if (v != v) {
        free(pairs);
        return ORC_EARG; /* NaN scores are not ordered */
      }
      pairs[t].v = v;
      pairs[t].i = t;
    }
    qsort(pairs, (size_t)n, sizeof(orc_pair), orc_cmp_desc);
    int32_t *out = idx + r * k_max;
    for (int j = 0; j < k; ++j) out[j] = pairs[j].i;
    qsort(out, (size_t)k, sizeof(int32_t), orc_cmp_int);
    for (int j = k; j < k_max; ++j) out[j] = -1;
    cnt[r] = k;
    free(pairs);
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Block granularity.                                                                          */
/* ------------------------------------------------------------------------------------------ */

/* [SD] §2 / R6: bscore[b,g,i,j] = max over tokens t of block j (t < L_b) of crit_cand[b,g,i,t]. */
int oracle_block_maxpool(const double *crit_cand, int64_t stride, const int32_t *seq_lens, int batch,
                         int h_kv, int n_c, int block, double *bscore, int64_t bstride) {
  if (!crit_cand || !seq_lens || !bscore || block <= 0) return ORC_EARG;
  for (int b = 0; b < batch; ++b) {
    int L = seq_lens[b], nb = (L + block - 1) / block;
    if ((int64_t)nb > bstride) return ORC_EARG;
    for (int g = 0; g < h_kv; ++g)
      for (int i = 0; i < n_c; ++i) {
        const double *src = crit_cand + (((int64_t)b * h_kv + g) * n_c + i) * stride;
        double *dst = bscore + (((int64_t)b * h_kv + g) * n_c + i) * bstride;
        for (int j = 0; j < nb; ++j) {
          double m = -INFINITY;
          for (int t = j * block; t < (j + 1) * block && t < L; ++t) m = src[t] > m ? src[t] : m;
          dst[j] = m;
        }
      }
  }
  return ORC_OK;
}

typedef struct {
  int32_t blk;
  int32_t cand;
} orc_bc;

static int orc_cmp_bc(const void *a, const void *b) {
  const orc_bc *x = (const orc_bc *)a, *y = (const orc_bc *)b;
  if (x->blk != y->blk) return (x->blk > y->blk) - (x->blk < y->blk);
  return (x->cand > y->cand) - (x->cand < y->cand);
}

/* [SSA] overlap-aware grouping: per unit, the union of the candidates' block sets in ascending order,
 * each with a bit mask of the candidates (bit i) that selected it.  blocks is [units][n_c][kb] with
 * bcnt[units][n_c] valid entries each. */
int oracle_block_union(const int32_t *blocks, const int32_t *bcnt, int n_units, int n_c, int kb,
                       int32_t *uidx, uint32_t *umask, int32_t *ucnt, int umax) {
  if (!blocks || !bcnt || !uidx || !umask || !ucnt || n_c < 1 || n_c > 32 || kb < 0) return ORC_EARG;
  orc_bc *all = (orc_bc *)malloc((size_t)(n_c * kb + 1) * sizeof(orc_bc));
  if (!all) return ORC_ENOMEM;
  for (int u = 0; u < n_units; ++u) {
    int n = 0;
    for (int i = 0; i < n_c; ++i) {
      int c = bcnt[(int64_t)u * n_c + i];
      if (c < 0 || c > kb) {
        free(all);
        return ORC_EARG;
      }
      for (int j = 0; j < c; ++j) all[n++] = (orc_bc){blocks[((int64_t)u * n_c + i) * kb + j], i};
    }
    qsort(all, (size_t)n, sizeof(orc_bc), orc_cmp_bc);
    int m = 0;
    for (int j = 0; j < n; ++j) {
      if (m > 0 && uidx[(int64_t)u * umax + m - 1] == all[j].blk) {
        umask[(int64_t)u * umax + m - 1] |= 1u << all[j].cand;
        continue;
      }
      if (m >= umax) {
        free(all);
        return ORC_EKMAX;
      }
      uidx[(int64_t)u * umax + m] = all[j].blk;
      umask[(int64_t)u * umax + m] = 1u << all[j].cand;
      ++m;
    }
    for (int j = m; j < umax; ++j) {
      uidx[(int64_t)u * umax + j] = -1;
      umask[(int64_t)u * umax + j] = 0;
    }
    ucnt[u] = m;
  }
  free(all);
  return ORC_OK;
}

typedef struct {
  orc_kv kv;
  const void *q;
  int qdtype, h_q, n_c;
  const int32_t *blocks, *bcnt;
  int kb, block;
  double scale;
  double *out, *lse;
} orc_battn_ctx;

/* [SSA] / R6: candidate i of request b attends to the tokens of its own selected blocks that are
 * visible to it (t < L, t <= L - n_c + i).  A block listed twice counts once (a set). */
static int orc_battn_unit(void *vctx, int unit, void *scratch) {
  orc_battn_ctx *c = (orc_battn_ctx *)vctx;
  const orc_kv *kv = &c->kv;
  int b = unit / kv->h_kv, g = unit % kv->h_kv, G = c->h_q / kv->h_kv, L = kv->seq_lens[b];
  int nb = (L + c->block - 1) / c->block;
  int32_t *tokens = (int32_t *)scratch;
  unsigned char *take = (unsigned char *)(tokens + L + 1);
  double *s_buf = (double *)(((uintptr_t)(take + nb + 16)) & ~(uintptr_t)7);
  for (int i = 0; i < c->n_c; ++i) {
    memset(take, 0, (size_t)nb);
    int nsel = c->bcnt[((int64_t)b * kv->h_kv + g) * c->n_c + i];
    if (nsel < 0 || nsel > c->kb) return ORC_EARG;
    const int32_t *bl = c->blocks + (((int64_t)b * kv->h_kv + g) * c->n_c + i) * c->kb;
    for (int j = 0; j < nsel; ++j) {
      if (bl[j] < 0 || bl[j] >= nb) return ORC_EIDX;
      take[bl[j]] = 1;
    }
    int last = L - c->n_c + i, n = 0;
    for (int t = 0; t <= last; ++t)
      if (take[t / c->block]) tokens[n++] = t;
    for (int hl = 0; hl < G; ++hl) {
      int64_t row = ((int64_t)b * c->n_c + i) * c->h_q + g * G + hl;
      int rc = orc_attend(kv, c->q, c->qdtype, row * kv->d, b, g, tokens, n, c->scale, s_buf,
                          c->out + row * kv->d, &c->lse[row], NULL);
      if (rc) return rc;
    }
  }
  return ORC_OK;
}

int oracle_block_attn(const void *pool, int dtype, int64_t num_pages, int page_size, int h_kv, int d,
                      const int32_t *page_table, int max_pages, const int32_t *seq_lens, int batch,
                      const void *q, int qdtype, int h_q, int n_c, const int32_t *blocks,
                      const int32_t *bcnt, int kb, int block, double scale, double *out, double *lse,
                      int nthreads) {
  if (!pool || !page_table || !seq_lens || !q || !blocks || !bcnt || !out || !lse || h_kv <= 0 ||
      h_q % h_kv || block <= 0 || n_c < 1)
    return ORC_EARG;
  int Lmax = 0;
  for (int b = 0; b < batch; ++b) Lmax = seq_lens[b] > Lmax ? seq_lens[b] : Lmax;
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] < n_c) return ORC_EARG;
  orc_battn_ctx c = {{pool, dtype, num_pages, page_size, h_kv, d, page_table, max_pages, seq_lens, batch},
                     q, qdtype, h_q, n_c, blocks, bcnt, kb, block, scale, out, lse};
  size_t scratch = (size_t)(Lmax + 1) * sizeof(int32_t) + (size_t)Lmax / block + 64 +
                   (size_t)(Lmax + 1) * sizeof(double);
  return orc_run(orc_battn_unit, &c, batch * h_kv, nthreads, scratch);
}

/* ---------------------------------------------------------------------------------------------
 * KV append and length advance (R8, [SSR]).  Plain element copies, no arithmetic.
 *   pool       [num_pages][2][h_kv][page_size][d], element size esize bytes, modified in place
 *   k_new/v_new [batch][n_new][h_kv][d]
 *   ok[b]      set to 1 when request b was written, 0 when it was skipped
 */
int oracle_kv_append(void *pool, int esize, int64_t num_pages, int page_size, int h_kv, int d,
                     const int32_t *page_table, int max_pages, const int32_t *seq_lens, int batch,
                     int max_seq_len, const void *k_new, const void *v_new, int n_new, int32_t *ok) {
  if (!pool || (esize != 2 && esize != 4) || page_size <= 0 || h_kv <= 0 || d <= 0 || n_new < 0 || batch < 0)
    return -1;
  const int64_t row_bytes = (int64_t)d * esize;
  for (int b = 0; b < batch; ++b) {
    ok[b] = 0;
    const int L = seq_lens[b];
    int good = L >= 0 && (int64_t)L + n_new <= max_seq_len;
    for (int j = 0; good && j < n_new; ++j) {
      const int t = L + j, pj = t / page_size;
      if (pj >= max_pages) { good = 0; break; }
      const int32_t p = page_table[(int64_t)b * max_pages + pj];
      if (p < 0 || (int64_t)p >= num_pages) good = 0;
    }
    if (!good) continue;
    for (int j = 0; j < n_new; ++j) {
      const int t = L + j;
      const int32_t p = page_table[(int64_t)b * max_pages + t / page_size];
      for (int g = 0; g < h_kv; ++g) {
        for (int which = 0; which < 2; ++which) {
          const int64_t dst = ((((int64_t)p * 2 + which) * h_kv + g) * page_size + t % page_size) * row_bytes;
          const int64_t src = ((((int64_t)b * n_new + j) * h_kv) + g) * row_bytes;
          memcpy((char *)pool + dst, (const char *)(which ? v_new : k_new) + src, (size_t)row_bytes);
        }
      }
    }
    ok[b] = 1;
  }
  return 0;
}

int oracle_kv_advance(int32_t *seq_lens, const int32_t *delta, int batch, int max_seq_len) {
  if (!seq_lens || !delta || batch < 0) return -1;
  for (int b = 0; b < batch; ++b) {
    const int64_t v = (int64_t)seq_lens[b] + delta[b];
    if (v >= 0 && v <= max_seq_len) seq_lens[b] = (int32_t)v;
  }
  return 0;
}

/* ---------------------------------------------------------------------------------------------
 * Phase assignment and per-step phase flags (R9).
 *   counts     [n_buckets] live requests per offset, updated in place
 *   offset_out [n_new] the offset given to each arriving request, in arrival order
 *   verify_out [batch] 1 when request b verifies at `step`, else 0
 */
int oracle_phase_assign(int32_t *counts, int n_buckets, int n_new, int32_t *offset_out) {
  if (!counts || n_buckets <= 0 || n_new < 0 || (n_new > 0 && !offset_out)) return -1;
  for (int r = 0; r < n_new; ++r) {
    int best = 0;
    for (int o = 1; o < n_buckets; ++o)
      if (counts[o] < counts[best]) best = o;
    counts[best] += 1;
    offset_out[r] = best;
  }
  return 0;
}

int oracle_phase_flags(const int32_t *offsets, int batch, int n_buckets, int64_t step, uint8_t *verify_out) {
  if (!offsets || !verify_out || batch < 0 || n_buckets <= 0 || step < 0) return -1;
  for (int b = 0; b < batch; ++b) {
    if (offsets[b] < 0 || offsets[b] >= n_buckets) return -1;
    verify_out[b] = (uint8_t)(((step + offsets[b]) % n_buckets) == n_buckets - 1);
  }
  return 0;
}

/* ---------------------------------------------------------------------------------------------
 * Top-p entry counts (R10).  kout[r] = min(K_p(r), k_max) for every row r (rows grouped as in
 * oracle_topk: row r uses lens[r / rows_per_group] and has ceil(len / len_div) entries).
 */
int oracle_topp_k(const float *scores, int64_t stride, const int32_t *lens, double p, int n_groups,
                  int rows_per_group, int len_div, int k_max, int32_t *kout) {
  if (!scores || !lens || !kout || rows_per_group <= 0 || len_div <= 0 || k_max < 0 || !(p >= 0.0)) return ORC_EARG;
  const int64_t n_rows = (int64_t)n_groups * rows_per_group;
  for (int64_t r = 0; r < n_rows; ++r) {
    const int n = (lens[r / rows_per_group] + len_div - 1) / len_div;
    if (n < 0 || (int64_t)n > stride) return ORC_EARG;
    orc_pair *pairs = (orc_pair *)malloc((size_t)(n > 0 ? n : 1) * sizeof(orc_pair));
    if (!pairs) return ORC_ENOMEM;
    double total = 0.0;
    for (int t = 0; t < n; ++t) {
      const float v = scores[r * stride + t];
      if (v != v || v < 0.f) {
        free(pairs);
        return ORC_EARG; /* scores are non-negative probabilities, never NaN */
      }
      pairs[t].v = v;
      pairs[t].i = t;
    }
    qsort(pairs, (size_t)n, sizeof(orc_pair), orc_cmp_desc);
    for (int t = 0; t < n; ++t) total += (double)pairs[t].v;
    const double target = p * total;
    int k = 0;
    double acc = 0.0;
    while (k < n && acc < target) acc += (double)pairs[k++].v;
    kout[r] = k < k_max ? k : k_max;
    free(pairs);
  }
  return 0;
}

/* ---------------------------------------------------------------------------------------------
 * Split-KV combine ([SS] §4.1: the verify caches each part's log-sum-exp, so partial attention
 * results over disjoint parts of the token set merge into the result over their union).
 * For each row: o_parts [n_rows][n_splits][d] holds every split's normalised output and lse_parts
 * [n_rows][n_splits] its natural-log log-sum-exp (-inf for an empty split).  The merged result is
 *   lse = log sum_j exp(lse_j),   out = sum_j exp(lse_j - lse) o_j,
 * evaluated with the largest lse_j factored out of the sum (the same value, without overflow).  A
 * row whose splits are all empty (or that has none) gives out = 0 and lse = -inf (R7).
 */
int oracle_combine(const float *o_parts, const float *lse_parts, int n_rows, int n_splits, int d, double *out,
                   double *lse) {
  if (n_rows < 0 || n_splits < 0 || d <= 0 || !out || !lse) return ORC_EARG;
  if (n_rows > 0 && n_splits > 0 && (!o_parts || !lse_parts)) return ORC_EARG;
  for (int r = 0; r < n_rows; ++r) {
    const float *lp = lse_parts ? lse_parts + (int64_t)r * n_splits : NULL;
    double m = -INFINITY;
    for (int j = 0; j < n_splits; ++j)
      if ((double)lp[j] > m) m = (double)lp[j];
    double *o = out + (int64_t)r * d;
    for (int k = 0; k < d; ++k) o[k] = 0.0;
    if (m == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double z = 0.0;
    for (int j = 0; j < n_splits; ++j) z += exp((double)lp[j] - m);
    const double total = m + log(z);
    for (int j = 0; j < n_splits; ++j) {
      const double w = exp((double)lp[j] - total);
      const float *oj = o_parts + ((int64_t)r * n_splits + j) * d;
      for (int k = 0; k < d; ++k) o[k] += w * (double)oj[k];
    }
    lse[r] = total;
  }
  return ORC_OK;
}
