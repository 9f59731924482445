/*
 * pisa_oracle.c -- plain, slow fp64 CPU oracle for the PISA pyramid Top-K
 * block selector.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the tests, the package smoke check and the CPU-baseline leg of the
 * benchmark load it.  It shares no code, header or constant with the CUDA
 * library; both sides only read the same seeded inputs.
 *
 * Sources (web pages about arXiv 2609.31093, "Block Sparse Attention with
 * Log-Linear Complexity"):
 *  [AGI]  agihunt.info paper summary -- pyramid paragraph ("Keys are stacked
 *         into a pyramid"), LSE/forced-blocks paragraph, kernel paragraph
 *         (GQA groups share selected blocks).
 *  [RCAP] rcap.io post -- "Think of the keys as leaves of a tree" (mean-pooled
 *         pyramid, g = 2), "Selection walks the tree top-down" (bounded
 *         candidate set, children of kept blocks), "The scoring rule matters"
 *         (LogSumExp over child summaries), and the pisa_select sketch that
 *         follows it.
 *  [AIKDE] aikde.pages.dev news piece, "Architecture and How It Works" item 1.
 *
 * Everything is computed in fp64 from the exact fp64 images of the inputs.
 * Readings of points the pages leave open:
 *  - a node summary is the plain mean of the raw keys inside its span, which
 *    for full spans equals the mean of its children's means [AGI pyramid
 *    paragraph: "mean-pool adjacent blocks"];
 *  - the walk starts at the root and keeps everything while a level has at
 *    most K candidates [RCAP pisa_select sketch, "start at coarsest level"];
 *  - a node is eligible when its leaf range meets E = [1, qb-2]; summaries
 *    themselves are not masked (prefill summaries include later keys), unless
 *    the prefix-consistent reading is asked for (po_params.prefix): then every
 *    summary a query at position t reads is the mean of its span's keys at
 *    positions <= t, the pyramid of the sequence's first t + 1 keys, which is
 *    what a decode step at length t + 1 sees [AGI pyramid paragraph, decode
 *    routing; RCAP pisa_select sketch];
 *  - "LSE" is the literal log-sum-exp, summed over the query heads of a GQA
 *    group; the scale is 1/sqrt(d) unless another is given; the PISA-1 and
 *    PISA-2 scorers replace it by its first- and second-order cumulant
 *    truncations over the same summands (po_reduce);
 *  - forced blocks F = {0, qb-1, qb} are added to the Top-K of the rest;
 *  - ties in Top-K go to the lower node index;
 *  - attention over the selection (po_sparse_attention) reads the keys of the
 *    union of the selected blocks at positions <= t, with the selection's
 *    score scale, and plain softmax-weighted values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PO_MAX_LEVELS 48

typedef struct {
  int64_t B;      /* batch */
  int64_t N;      /* sequence length (key capacity for decode layouts) */
  int32_t Hq;     /* query heads */
  int32_t Hkv;    /* key heads; Hq % Hkv == 0, group size G = Hq / Hkv */
  int32_t d;      /* head dimension */
  int32_t C;      /* leaf block size */
  int32_t K;      /* Top-K per level */
  double scale;   /* score scale inside exp(); <= 0 means 1/sqrt(d) */
  int32_t scorer; /* 0: log-sum-exp; 1: PISA-1; 2: PISA-2 (po_reduce) */
  int32_t prefix; /* 0: node summaries over all keys of the span (default);
                     1: over the span's keys at positions <= t (prefix-
                     consistent prefill, po_summary) */
} po_params;

/* ---------------------------------------------------------------- tree shape
 * Level 1 holds the nb = ceil(n/C) leaf blocks; each coarser level pools two
 * adjacent nodes (g = 2), n_l = ceil(n_{l-1} / 2), until one node is left.
 * [AGI pyramid paragraph; RCAP "Think of the keys as leaves of a tree"]   */
static int64_t po_ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Number of levels and the node count of each level (sizes[0] = level 1). */
static int po_level_sizes(int64_t nb, int64_t* sizes) {
  int L = 0;
  int64_t n = nb;
  if (nb <= 0) return 0;
  for (;;) {
    sizes[L++] = n;
    if (n == 1) break;
    n = po_ceil_div(n, 2);
  }
  return L;
}

int po_num_levels(int64_t N, int32_t C) {
  int64_t sizes[PO_MAX_LEVELS];
  return po_level_sizes(po_ceil_div(N, C), sizes);
}

/* Total number of pyramid nodes per (batch, key head) for capacity N. */
int64_t po_num_nodes(int64_t N, int32_t C) {
  int64_t sizes[PO_MAX_LEVELS];
  int L = po_level_sizes(po_ceil_div(N, C), sizes);
  int64_t P = 0;
  for (int l = 0; l < L; ++l) P += sizes[l];
  return P;
}

/* Row offset of level `level` (1-based) inside one (batch, head) slab. */
static int64_t po_level_offset(const int64_t* sizes, int level) {
  int64_t off = 0;
  for (int l = 1; l < level; ++l) off += sizes[l - 1];
  return off;
}

static double po_scale(const po_params* p) {
  return p->scale > 0.0 ? p->scale : 1.0 / sqrt((double)p->d);
}

/* ------------------------------------------------------------- key pyramid
 * pyr[b][h][node][d]: the mean of the raw keys k[b][h][j] over the node's
 * span, j in [lo*C, min(hi*C, len)), where [lo, hi) is the node's leaf range
 * and len = seq_lens[b] (or N).  Empty spans hold zeros.  The layout is the
 * one of capacity N; a shorter len only changes which keys are present.   */
int po_build_pyramid(const po_params* p, const double* k,
                     const int32_t* seq_lens, double* pyr) {
  int64_t sizes[PO_MAX_LEVELS];
  const int64_t nb_cap = po_ceil_div(p->N, p->C);
  const int L = po_level_sizes(nb_cap, sizes);
  const int64_t P = po_num_nodes(p->N, p->C);
  const int d = p->d;
  for (int64_t b = 0; b < p->B; ++b) {
    const int64_t len = seq_lens ? seq_lens[b] : p->N;
    if (len < 0 || len > p->N) return -1;
    for (int32_t h = 0; h < p->Hkv; ++h) {
      const double* kh = k + ((b * p->Hkv + h) * p->N) * d;
      double* ph = pyr + ((b * p->Hkv + h) * P) * d;
      for (int level = 1; level <= L; ++level) {
        const int64_t off = po_level_offset(sizes, level);
        const int64_t span = (int64_t)1 << (level - 1); /* leaves per node */
        for (int64_t j = 0; j < sizes[level - 1]; ++j) {
          double* out = ph + (off + j) * d;
          int64_t lo = j * span * p->C;
          int64_t hi = (j + 1) * span * p->C;
          if (hi > len) hi = len;
          for (int c = 0; c < d; ++c) out[c] = 0.0;
          if (hi <= lo) continue;
          for (int64_t t = lo; t < hi; ++t)
            for (int c = 0; c < d; ++c) out[c] += kh[t * d + c];
          for (int c = 0; c < d; ++c) out[c] /= (double)(hi - lo);
        }
      }
    }
  }
  return 0;
}

/* ---------------------------------------------------------------- scoring */
static double po_dot(const double* a, const double* b, int d) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += a[c] * b[c];
  return s;
}

/* log(sum_i exp(x_i)) with the maximum taken out first. */
static double po_lse(const double* x, int64_t n) {
  double m = -INFINITY, s = 0.0;
  if (n <= 0) return -INFINITY;
  for (int64_t i = 0; i < n; ++i) if (x[i] > m) m = x[i];
  for (int64_t i = 0; i < n; ++i) s += exp(x[i] - m);
  return m + log(s);
}

/* The block score over n summands x_i (scaled dots with child summaries or
 * raw keys) [AGI LSE paragraph: "PISA-1 keeps only the mean; PISA-2 adds the
 * variance term from the LSE Taylor expansion"; RCAP "The scoring rule
 * matters": truncations at first and second order].  Writing
 * LSE(x) = log n + log((1/n) sum_i exp(x_i)) and expanding the second term
 * in cumulants of the x_i around their mean:
 *   scorer 0: LSE(x) itself;
 *   scorer 1: log n + mean(x);
 *   scorer 2: log n + mean(x) + var(x) / 2, var the population variance. */
static double po_reduce(const double* x, int64_t n, int scorer) {
  double mean = 0.0, var = 0.0;
  if (scorer == 0 || n <= 0) return po_lse(x, n);
  for (int64_t i = 0; i < n; ++i) mean += x[i];
  mean /= (double)n;
  if (scorer == 1) return log((double)n) + mean;
  for (int64_t i = 0; i < n; ++i) var += (x[i] - mean) * (x[i] - mean);
  var /= (double)n;
  return log((double)n) + mean + 0.5 * var;
}

/* Context of one query: batch b, key head h, position t, sequence length
 * len (prefill: N; decode: the sequence's current length). */
typedef struct {
  const po_params* p;
  const double* q;     /* [B, Hq, N, d] (prefill) -- or row pointers below */
  const double* k;     /* [B, Hkv, N, d] */
  const double* pyr;   /* [B, Hkv, P, d] */
  const double* qrow[64]; /* the G query-head rows of this query */
  int64_t b, t, len, qb, nb;
  int32_t h, G;
  int64_t sizes[PO_MAX_LEVELS];
  int L_cap, L_len;
  int64_t P;
  double s;
} po_query;

/* E = [1, qb-2]: leaf blocks that are complete, strictly in the past and not
 * forced.  A level-`level` node is eligible when its leaf range meets E. */
static int po_eligible(const po_query* Q, int level, int64_t j) {
  const int64_t span = (int64_t)1 << (level - 1);
  const int64_t lo = j * span, hi = (j + 1) * span - 1; /* inclusive */
  const int64_t e_lo = 1, e_hi = Q->qb - 2;
  if (e_hi < e_lo) return 0;
  return lo <= e_hi && hi >= e_lo;
}

static const double* po_node(const po_query* Q, int level, int64_t j) {
  const int64_t off = po_level_offset(Q->sizes, level);
  return Q->pyr + (((Q->b * Q->p->Hkv + Q->h) * Q->P) + off + j) * Q->p->d;
}

/* Summary of node (level, j) as query Q reads it.  Default: its pyramid row
 * (the mean of the keys of its span present in the sequence).  With
 * p->prefix, a span that reaches past position t is summarised by the mean of
 * its keys at positions <= t, computed here from the raw keys into buf (d
 * doubles); a span with no such key reads as zeros. */
static const double* po_summary(const po_query* Q, int level, int64_t j, double* buf) {
  if (Q->p->prefix) {
    const int64_t span = (int64_t)Q->p->C << (level - 1);
    const int64_t lo = j * span;
    int64_t hi = lo + span;
    if (hi > Q->len) hi = Q->len;
    if (hi > Q->t + 1) {
      const int d = Q->p->d;
      const double* kh = Q->k + ((Q->b * Q->p->Hkv + Q->h) * Q->p->N) * d;
      const int64_t end = Q->t + 1;
      for (int c = 0; c < d; ++c) buf[c] = 0.0;
      if (end <= lo) return buf;
      for (int64_t i = lo; i < end; ++i)
        for (int c = 0; c < d; ++c) buf[c] += kh[i * d + c];
      for (int c = 0; c < d; ++c) buf[c] /= (double)(end - lo);
      return buf;
    }
  }
  return po_node(Q, level, j);
}

/* Score of candidate j at `level`, summed over the G query heads of the group
 * [AGI kernel paragraph: heads of one GQA group share the selection].
 *  level >= 2: log-sum-exp over the eligible children's summaries
 *              [RCAP "The scoring rule matters"];
 *  level == 1: log-sum-exp over the C raw keys of the leaf block
 *              [AGI kernel paragraph: "leaf LSE scoring"].
 * counters (nullable): [1] child dots, [2] leaf keys. */
static double po_score(const po_query* Q, int level, int64_t j,
                       int64_t* counters) {
  const int d = Q->p->d;
  double total = 0.0;
  if (level >= 2) {
    const double* kids[2];
    double* bufs = (double*)malloc(sizeof(double) * 2 * (size_t)d);
    int nk = 0;
    for (int64_t c = 2 * j; c <= 2 * j + 1; ++c) {
      if (c >= Q->sizes[level - 2]) continue;
      if (!po_eligible(Q, level - 1, c)) continue;
      kids[nk] = po_summary(Q, level - 1, c, bufs + (size_t)nk * d);
      ++nk;
    }
    if (counters) counters[1] += nk;
    for (int g = 0; g < Q->G; ++g) {
      double x[2];
      for (int i = 0; i < nk; ++i) x[i] = Q->s * po_dot(Q->qrow[g], kids[i], d);
      total += po_reduce(x, nk, Q->p->scorer);
    }
    free(bufs);
    return total;
  }
  /* leaf: keys [j*C, min((j+1)*C, len)) of key head h */
  {
    const int64_t lo = j * Q->p->C;
    int64_t hi = (j + 1) * Q->p->C;
    if (hi > Q->len) hi = Q->len;
    const int64_t n = hi - lo;
    double* x = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    const double* kh = Q->k + ((Q->b * Q->p->Hkv + Q->h) * Q->p->N) * d;
    if (counters) counters[2] += n;
    for (int g = 0; g < Q->G; ++g) {
      for (int64_t i = 0; i < n; ++i)
        x[i] = Q->s * po_dot(Q->qrow[g], kh + (lo + i) * d, d);
      total += po_reduce(x, n, Q->p->scorer);
    }
    free(x);
    return total;
  }
}

/* Higher score first; equal scores go to the lower index. */
typedef struct { double score; int64_t idx; } po_cand;
static int po_cmp_desc(const void* a, const void* b) {
  const po_cand* x = (const po_cand*)a;
  const po_cand* y = (const po_cand*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}
static int po_cmp_idx(const void* a, const void* b) {
  const int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
  return (x > y) - (x < y);
}

/* q_mode 0: q is [B, Hq, N, d]; 1: q is [B, Hq, d] (one decode query per
 * sequence); 2: q points at this query's own [G, d] head rows. */
static int po_setup(po_query* Q, const po_params* p, const double* q,
                    const double* k, const double* pyr, int64_t b, int32_t h,
                    int64_t t, int64_t len, int q_mode) {
  Q->p = p; Q->q = q; Q->k = k; Q->pyr = pyr;
  Q->b = b; Q->h = h; Q->t = t; Q->len = len;
  Q->G = p->Hq / p->Hkv;
  if (Q->G > 64 || Q->G < 1) return -1;
  Q->qb = t / p->C;
  Q->nb = po_ceil_div(len, p->C);
  Q->L_cap = po_level_sizes(po_ceil_div(p->N, p->C), Q->sizes);
  {
    int64_t tmp[PO_MAX_LEVELS];
    Q->L_len = po_level_sizes(Q->nb, tmp);
  }
  Q->P = po_num_nodes(p->N, p->C);
  Q->s = po_scale(p);
  for (int g = 0; g < Q->G; ++g) {
    const int64_t hq = (int64_t)h * Q->G + g;
    if (q_mode == 1)
      Q->qrow[g] = q + (b * p->Hq + hq) * p->d;
    else if (q_mode == 2)
      Q->qrow[g] = q + (int64_t)g * p->d;
    else
      Q->qrow[g] = q + ((b * p->Hq + hq) * p->N + t) * p->d;
  }
  return 0;
}

/* One query's selection.  Writes K+3 indices (ascending, -1 padded) and
 * their scores (group-summed leaf LSE; +inf for forced blocks; -inf for
 * padding).  *margin gets the smallest gap between the K-th and (K+1)-th
 * scores over the levels that had more than K candidates (+inf if none).
 * trace (nullable) gets, per level l = 1..L_cap, the kept set (K slots, -1
 * padded, ascending); levels above the query's root stay -1. */
static int po_select_one(po_query* Q, int32_t* out_idx, double* out_score,
                         double* margin, int32_t* trace, int64_t* counters) {
  const int K = Q->p->K;
  const int W = K + 3;
  int64_t forced[3];
  int nf = 0;
  *margin = INFINITY;
  for (int i = 0; i < W; ++i) { out_idx[i] = -1; out_score[i] = -INFINITY; }
  if (trace)
    for (int i = 0; i < Q->L_cap * K; ++i) trace[i] = -1;

  /* Forced blocks F = {0, qb-1, qb} n [0, qb] [AGI LSE/forced paragraph]. */
  forced[nf++] = 0;
  if (Q->qb - 1 > 0) forced[nf++] = Q->qb - 1;
  if (Q->qb > 0) forced[nf++] = Q->qb;

  po_cand* kept = (po_cand*)malloc(sizeof(po_cand) * (size_t)(2 * K + 2));
  po_cand* cand = (po_cand*)malloc(sizeof(po_cand) * (size_t)(2 * K + 2));
  int nkept = 0;
  const int64_t n_elig = Q->qb - 2 >= 1 ? Q->qb - 2 : 0; /* |E| */

  if (n_elig > 0) {
    /* Walk from the root (level L_len, node 0) down to the leaves
     * [RCAP pisa_select sketch]. */
    int ncand = 1;
    cand[0].idx = 0;
    for (int level = Q->L_len; level >= 1; --level) {
      if (ncand > K) {
        for (int i = 0; i < ncand; ++i)
          cand[i].score = po_score(Q, level, cand[i].idx, counters);
        if (counters) { counters[0] += 1; counters[3] += ncand; }
        qsort(cand, (size_t)ncand, sizeof(po_cand), po_cmp_desc);
        {
          const double gap = cand[K - 1].score - cand[K].score;
          if (gap < *margin) *margin = gap;
        }
        nkept = K;
      } else {
        /* At most K candidates: all are kept.  Scores are still needed at the
         * leaves, where they are reported. */
        if (level == 1)
          for (int i = 0; i < ncand; ++i)
            cand[i].score = po_score(Q, level, cand[i].idx, counters);
        nkept = ncand;
      }
      for (int i = 0; i < nkept; ++i) kept[i] = cand[i];
      if (trace) {
        int64_t* tmp = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nkept > 0 ? nkept : 1));
        for (int i = 0; i < nkept; ++i) tmp[i] = kept[i].idx;
        qsort(tmp, (size_t)nkept, sizeof(int64_t), po_cmp_idx);
        for (int i = 0; i < nkept; ++i) trace[(level - 1) * K + i] = (int32_t)tmp[i];
        free(tmp);
      }
      if (level == 1) break;
      /* Children of the kept nodes become the next candidates; ineligible
       * children are dropped [RCAP "Selection walks the tree top-down"]. */
      ncand = 0;
      for (int i = 0; i < nkept; ++i)
        for (int64_t c = 2 * kept[i].idx; c <= 2 * kept[i].idx + 1; ++c) {
          if (c >= Q->sizes[level - 2]) continue;
          if (!po_eligible(Q, level - 1, c)) continue;
          cand[ncand].idx = c;
          cand[ncand].score = 0.0;
          ++ncand;
        }
    }
  }

  /* Output: Top-K of E together with F, ascending, -1 padded. */
  {
    po_cand* all = (po_cand*)malloc(sizeof(po_cand) * (size_t)(K + 3));
    int n = 0;
    for (int i = 0; i < nkept; ++i) all[n++] = kept[i];
    for (int i = 0; i < nf; ++i) { all[n].idx = forced[i]; all[n].score = INFINITY; ++n; }
    /* ascending index order */
    for (int i = 1; i < n; ++i) {
      po_cand v = all[i];
      int j = i - 1;
      while (j >= 0 && all[j].idx > v.idx) { all[j + 1] = all[j]; --j; }
      all[j + 1] = v;
    }
    for (int i = 0; i < n; ++i) { out_idx[i] = (int32_t)all[i].idx; out_score[i] = all[i].score; }
    free(all);
  }
  free(kept);
  free(cand);
  return 0;
}

/* Selection for a list of queries.  sel holds nsel triples (b, h, t); a NULL
 * sel means every (b, h, t) of a prefill, t in [0, N).
 * mode 0 (prefill): q is [B, Hq, N, d], all keys [0, N) are present.
 * mode 1 (decode):  q is [B, Hq, d]; sequence b holds keys [0, seq_lens[b]),
 *                   and its query sits at position seq_lens[b]-1 (sel is
 *                   ignored; one query per (b, h) in (b, h) order).
 * mode 2 (rows):    like prefill with a sel list, but q holds only the
 *                   selected queries' head rows, [nsel, G, d].
 * Outputs per query: out_idx[K+3] (int32), out_score[K+3], margin;
 * trace (nullable) [nq, L_cap, K]; counters (nullable) int64[4] =
 * {levels scored, child dots, leaf keys, candidates scored}. */
int po_select(const po_params* p, const double* q, const double* k,
              const double* pyr, const int32_t* seq_lens, int mode,
              int64_t nsel, const int64_t* sel, int32_t* out_idx,
              double* out_score, double* out_margin, int32_t* trace,
              int64_t* counters) {
  const int W = p->K + 3;
  const int L_cap = po_num_levels(p->N, p->C);
  int64_t nq;
  if (p->Hkv <= 0 || p->Hq % p->Hkv != 0 || p->K < 1 || p->C < 1 || p->d < 1)
    return -1;
  if (mode == 1) nq = p->B * p->Hkv;
  else nq = sel ? nsel : p->B * p->Hkv * p->N;
  if (mode == 2 && !sel) return -1;
  int64_t c0 = 0, c1 = 0, c2 = 0, c3 = 0;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : c0, c1, c2, c3)
  for (int64_t i = 0; i < nq; ++i) {
    int64_t b, t, len;
    int32_t h;
    if (mode == 1) {
      b = i / p->Hkv; h = (int32_t)(i % p->Hkv);
      len = seq_lens ? seq_lens[b] : p->N;
      t = len - 1;
    } else if (sel) {
      b = sel[3 * i]; h = (int32_t)sel[3 * i + 1]; t = sel[3 * i + 2];
      len = p->N;
    } else {
      b = i / (p->Hkv * p->N);
      h = (int32_t)((i / p->N) % p->Hkv);
      t = i % p->N;
      len = p->N;
    }
    if (t < 0 || t >= len || len > p->N) { err = 1; continue; }
    po_query Q;
    int64_t cnt[4] = {0, 0, 0, 0};
    const double* qbase = mode == 2 ? q + i * (int64_t)(p->Hq / p->Hkv) * p->d : q;
    if (po_setup(&Q, p, qbase, k, pyr, b, h, t, len, mode) != 0) { err = 1; continue; }
    po_select_one(&Q, out_idx + i * W, out_score + i * W, out_margin + i,
                  trace ? trace + i * (int64_t)L_cap * p->K : NULL, cnt);
    c0 += cnt[0]; c1 += cnt[1]; c2 += cnt[2]; c3 += cnt[3];
  }
  if (counters) { counters[0] = c0; counters[1] = c1; counters[2] = c2; counters[3] = c3; }
  return err ? -1 : 0;
}

/* Scores of arbitrary nodes at one level for one query (the same po_score
 * used by the walk).  Used by tests that re-check a Top-K level by level. */
int po_score_nodes(const po_params* p, const double* q, const double* k,
                   const double* pyr, int64_t len, int mode, int64_t b,
                   int32_t h, int64_t t, int level, int64_t n,
                   const int64_t* nodes, double* out) {
  po_query Q;
  if (t < 0 || t >= len || len > p->N) return -1;
  if (po_setup(&Q, p, q, k, pyr, b, h, t, len, mode) != 0) return -1;
  if (level < 1 || level > Q.L_cap) return -1;
  for (int64_t i = 0; i < n; ++i) {
    if (nodes[i] < 0 || nodes[i] >= Q.sizes[level - 1]) return -1;
    out[i] = po_score(&Q, level, nodes[i], NULL);
  }
  return 0;
}

/* Eligibility of a node for one query (exported for tests). */
int po_node_eligible(const po_params* p, int64_t t, int level, int64_t j) {
  po_query Q;
  memset(&Q, 0, sizeof(Q));
  Q.p = p;
  Q.qb = t / p->C;
  return po_eligible(&Q, level, j);
}

/* ------------------------------------------------------ flat comparator
 * BSA-style flat selector [AGI model paragraph: "NSA's selected branch with
 * mean summaries"; RCAP "The direct comparison point is BSA"].  Each query
 * head h' scores every complete past block i in [0, qb-1] by
 * p_h'(i) = softmax_i(s q_h' . mu(1, i)); block score = sum over the group's
 * heads; Top-K over E, plus F, same output format as po_select.         */
int po_select_flat(const po_params* p, const double* q, const double* pyr,
                   int64_t nsel, const int64_t* sel, int32_t* out_idx,
                   double* out_score, double* out_margin) {
  const int K = p->K, W = K + 3;
  const int64_t nq = sel ? nsel : p->B * p->Hkv * p->N;
  const int64_t P = po_num_nodes(p->N, p->C);
  const double s = po_scale(p);
  const int32_t G = p->Hq / p->Hkv;
  int err = 0;
  if (p->Hkv <= 0 || p->Hq % p->Hkv != 0 || K < 1) return -1;
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t i = 0; i < nq; ++i) {
    int64_t b, t; int32_t h;
    if (sel) { b = sel[3 * i]; h = (int32_t)sel[3 * i + 1]; t = sel[3 * i + 2]; }
    else {
      b = i / (p->Hkv * p->N); h = (int32_t)((i / p->N) % p->Hkv); t = i % p->N;
    }
    if (t < 0 || t >= p->N) { err = 1; continue; }
    const int64_t qb = t / p->C;
    const int64_t nprev = qb; /* complete past blocks 0 .. qb-1 */
    int32_t* oi = out_idx + i * W;
    double* os = out_score + i * W;
    for (int j = 0; j < W; ++j) { oi[j] = -1; os[j] = -INFINITY; }
    out_margin[i] = INFINITY;
    double* score = (double*)calloc((size_t)(nprev > 0 ? nprev : 1), sizeof(double));
    double* z = (double*)malloc(sizeof(double) * (size_t)(nprev > 0 ? nprev : 1));
    const double* mu = pyr + ((b * p->Hkv + h) * P) * p->d; /* level 1 at offset 0 */
    for (int32_t g = 0; g < G; ++g) {
      const double* qr = q + ((b * p->Hq + (int64_t)h * G + g) * p->N + t) * p->d;
      for (int64_t j = 0; j < nprev; ++j) z[j] = s * po_dot(qr, mu + j * p->d, p->d);
      const double lse = po_lse(z, nprev);
      for (int64_t j = 0; j < nprev; ++j) score[j] += exp(z[j] - lse);
    }
    /* Top-K over E = [1, qb-2] */
    int64_t ne = qb - 2 >= 1 ? qb - 2 : 0;
    po_cand* c = (po_cand*)malloc(sizeof(po_cand) * (size_t)(ne > 0 ? ne : 1));
    for (int64_t j = 0; j < ne; ++j) { c[j].idx = 1 + j; c[j].score = score[1 + j]; }
    qsort(c, (size_t)ne, sizeof(po_cand), po_cmp_desc);
    int nk = ne < K ? (int)ne : K;
    if (ne > K) out_margin[i] = c[K - 1].score - c[K].score;
    po_cand* all = (po_cand*)malloc(sizeof(po_cand) * (size_t)(K + 3));
    int n = 0;
    for (int j = 0; j < nk; ++j) all[n++] = c[j];
    all[n].idx = 0; all[n++].score = INFINITY;
    if (qb - 1 > 0) { all[n].idx = qb - 1; all[n++].score = INFINITY; }
    if (qb > 0) { all[n].idx = qb; all[n++].score = INFINITY; }
    for (int a = 1; a < n; ++a) {
      po_cand v = all[a];
      int j = a - 1;
      while (j >= 0 && all[j].idx > v.idx) { all[j + 1] = all[j]; --j; }
      all[j + 1] = v;
    }
    for (int j = 0; j < n; ++j) { oi[j] = (int32_t)all[j].idx; os[j] = all[j].score; }
    free(all); free(c); free(z); free(score);
  }
  return err ? -1 : 0;
}

/* ------------------------------------------- attention over the selection
 * Block-sparse attention that reads only the selected blocks [AGI opening
 * paragraph: each query reads only its Top-K tiles, so the attention pass is
 * linear in N; RCAP "Selection walks the tree top-down": the leaf indices are
 * then used for sparse attention over the original keys].  For the query
 * (b, key head h, position t) and each query head g of its group:
 *   A(t) = union over the selected blocks j >= 0 of idx[b, h, t, :] of the
 *          key positions i in [j C, (j+1) C) with i <= t   (causal);
 *   o_g  = sum_{i in A} exp(s q_g . k_i) v_i / sum_{i in A} exp(s q_g . k_i),
 * with s the score scale of the selection (1/sqrt(d) unless given).  A block
 * listed twice counts once.  q [B, Hq, N, d]; k, v [B, Hkv, N, d]; idx
 * [B, Hkv, N, K+3] int32 (-1 = empty slot); sel: nsel triples (b, h, t), or
 * NULL for every (b, h, t) in order; qrows != 0 (with sel): q holds only the
 * selected queries' head rows, [nsel, G, d].  out [nq, G, d] fp64.  Returns
 * -1 on a bad position or when some query has no attended key.           */
int po_sparse_attention(const po_params* p, const double* q, const double* k,
                        const double* v, const int32_t* idx, int64_t nsel,
                        const int64_t* sel, int qrows, double* out) {
  const int W = p->K + 3;
  const int d = p->d;
  if (p->Hkv <= 0 || p->Hq % p->Hkv != 0 || p->K < 1 || p->C < 1 || d < 1)
    return -1;
  const int32_t G = p->Hq / p->Hkv;
  const double s = po_scale(p);
  const int64_t nq = sel ? nsel : p->B * p->Hkv * p->N;
  int err = 0;
  if (qrows && !sel) return -1;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t i = 0; i < nq; ++i) {
    int64_t b, t;
    int32_t h;
    if (sel) { b = sel[3 * i]; h = (int32_t)sel[3 * i + 1]; t = sel[3 * i + 2]; }
    else {
      b = i / (p->Hkv * p->N); h = (int32_t)((i / p->N) % p->Hkv); t = i % p->N;
    }
    if (b < 0 || b >= p->B || h < 0 || h >= p->Hkv || t < 0 || t >= p->N) { err = 1; continue; }
    const int32_t* row = idx + ((b * p->Hkv + h) * p->N + t) * W;
    /* the attended key positions, each once, ascending */
    int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)W * (size_t)p->C);
    int64_t nk = 0;
    int64_t blocks[64];
    int nbk = 0;
    for (int j = 0; j < W && j < 64; ++j) {
      const int64_t blk = row[j];
      int seen = 0;
      if (blk < 0) continue;
      for (int u = 0; u < nbk; ++u) seen |= blocks[u] == blk;
      if (seen) continue;
      blocks[nbk++] = blk;
    }
    for (int u = 1; u < nbk; ++u) {  /* ascending block order */
      int64_t x = blocks[u];
      int w = u - 1;
      while (w >= 0 && blocks[w] > x) { blocks[w + 1] = blocks[w]; --w; }
      blocks[w + 1] = x;
    }
    for (int u = 0; u < nbk; ++u)
      for (int64_t c = 0; c < p->C; ++c) {
        const int64_t pos = blocks[u] * p->C + c;
        if (pos <= t && pos < p->N) keys[nk++] = pos;
      }
    if (nk == 0) { err = 1; free(keys); continue; }
    double* z = (double*)malloc(sizeof(double) * (size_t)nk);
    const double* kh = k + (b * p->Hkv + h) * p->N * d;
    const double* vh = v + (b * p->Hkv + h) * p->N * d;
    for (int32_t g = 0; g < G; ++g) {
      const double* qr = qrows ? q + (i * G + g) * d
                               : q + ((b * p->Hq + (int64_t)h * G + g) * p->N + t) * d;
      double* o = out + (i * G + g) * d;
      double m = -INFINITY, l = 0.0;
      for (int64_t u = 0; u < nk; ++u) {
        z[u] = s * po_dot(qr, kh + keys[u] * d, d);
        if (z[u] > m) m = z[u];
      }
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int64_t u = 0; u < nk; ++u) {
        const double w = exp(z[u] - m);
        const double* vr = vh + keys[u] * d;
        l += w;
        for (int c = 0; c < d; ++c) o[c] += w * vr[c];
      }
      for (int c = 0; c < d; ++c) o[c] /= l;
    }
    free(z);
    free(keys);
  }
  return err ? -1 : 0;
}

int po_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void po_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
