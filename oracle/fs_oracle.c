/*
 * fs_oracle.c -- plain, slow fp64 CPU oracle of the FreeSolo FS-L attention
 * forward pass, and of its backward pass with the hard indices held fixed.
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library; the product path (the CUDA
 * library under long_context_lm_gb300/csrc) never does, and the two share no
 * code, header, table or constant.
 *
 * Sources (web summaries of the paper, cited by page and section):
 *   [rainbus]  "FreeSolo:线性时间稀疏注意力实现零样本长度外推 FreeSolo: Linear-time
 *              Sparse Attention with Zero-Shot Length Extrapolation"
 *              (paper.rainbus.top summary), sections 前置知识, 核心方法,
 *              方法步骤详情 steps ①-⑥, 局限与改进.
 *   [ai.info]  "FreeSolo: Linear-time Sparse Attention with Zero-Shot Length
 *              Extrapolation" (ai.info AI summary), sections "Key
 *              Contributions", "Methodology in Plain English", "Why This
 *              Matters".
 *
 * The pages give the method in prose only; no formula is printed.  Where they
 * leave a step open the reading taken here is stated next to the code (and
 * listed in the design notes):
 *   - cell score      u_c = q.kbar_c + lambda_h * a_c * erf(sigma_h*(n - p_c)/s),
 *                     p_c = c*s + s/2 (cell midpoint), no 1/sqrt(d) on q.kbar;
 *   - availability    a cell is available to query block beta iff it ends at or
 *                     before the block start b0 = beta*Bq;
 *   - FS-L pool       the W newest available cells plus the top-P older cells
 *                     by (a_c desc, c asc); the two sets are disjoint;
 *   - selection       top-min(K,|pool|) by (u desc, c asc);
 *   - readout         softmax(q.k_t/sqrt(d)) over the selected cells' tokens,
 *                     no rotation, then RMSNorm without gain (eps), 0 if no
 *                     cell is available;
 *   - window          w keys including self, RoPE NeoX half-split
 *                     theta_i = base^(-2i/d), softmax scale 1/sqrt(d);
 *   - mix             out = o_win + m_h * o_long.
 *
 * Everything is computed in double precision from float inputs (the callers
 * pass bf16-rounded values, which float holds exactly).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Cell summaries.  [rainbus] 方法步骤详情 ③, 核心方法; [ai.info] "Key
 * Contributions" 2: kbar_c is the mean of the cell's s unrotated keys, a_c the
 * largest token-key L2 norm inside the cell.                                 */
/* ------------------------------------------------------------------------ */
static void cell_summaries(const float *k, int N, int d, int s, double *kbar,
                           double *amax) {
  int C = N / s;
  for (int c = 0; c < C; ++c) {
    double *kb = kbar + (size_t)c * d;
    for (int i = 0; i < d; ++i) kb[i] = 0.0;
    double best = -1.0;
    for (int t = c * s; t < (c + 1) * s; ++t) {
      const float *kt = k + (size_t)t * d;
      double sq = 0.0;
      for (int i = 0; i < d; ++i) {
        kb[i] += (double)kt[i];
        sq += (double)kt[i] * (double)kt[i];
      }
      double nrm = sqrt(sq);
      if (nrm > best) best = nrm;
    }
    for (int i = 0; i < d; ++i) kb[i] /= (double)s;
    amax[c] = best;
  }
}

/* ------------------------------------------------------------------------ */
/* Availability set (pool) of one query block.  [rainbus] 核心方法 and
 * 方法步骤详情 ④; [ai.info] "Methodology in Plain English": FS keeps the
 * whole available prefix; FS-L keeps the W most recent available cells plus
 * the P older cells with the largest a_c, a pool of at most P+W cells that
 * changes only at query-block boundaries.                                    */
/* ------------------------------------------------------------------------ */
typedef struct {
  double a;
  int c;
} cell_key;

/* (a desc, c asc): the cell with the larger norm ranks first; equal norms
 * rank the older (smaller index) cell first. */
static int cmp_cell_key(const void *x, const void *y) {
  const cell_key *p = (const cell_key *)x, *q = (const cell_key *)y;
  if (p->a > q->a) return -1;
  if (p->a < q->a) return 1;
  return (p->c < q->c) ? -1 : (p->c > q->c);
}

/* Definition form: sort the older cells from scratch.  Writes the pool as the
 * recent cells in ascending order followed by the kept older cells in rank
 * order; returns its size.  *gap_rel is the relative norm gap between the
 * P-th and (P+1)-th ranked older cell (the decision that fixes the pool), or
 * INFINITY when there are at most P older cells. */
static int pool_definition(const double *amax, int A, int P, int W, int mode,
                           int32_t *pool, double *gap_rel, cell_key *scratch) {
  *gap_rel = INFINITY;
  if (mode == 1) { /* FS: the whole available prefix */
    for (int c = 0; c < A; ++c) pool[c] = c;
    return A;
  }
  int nrec = A < W ? A : W;
  int nold = A - nrec;
  int n = 0;
  for (int c = nold; c < A; ++c) pool[n++] = c;
  for (int c = 0; c < nold; ++c) {
    scratch[c].a = amax[c];
    scratch[c].c = c;
  }
  qsort(scratch, (size_t)nold, sizeof(cell_key), cmp_cell_key);
  int keep = nold < P ? nold : P;
  for (int r = 0; r < keep; ++r) pool[n++] = scratch[r].c;
  if (nold > P) {
    double x = scratch[P - 1].a, y = scratch[P].a;
    double den = fabs(x) > fabs(y) ? fabs(x) : fabs(y);
    *gap_rel = den > 0 ? (x - y) / den : 0.0;
  }
  return n;
}

/* Running form of the same rule: a top-P list kept in rank order and updated
 * only when cells leave the recency window at a block boundary ([ai.info]
 * "Methodology in Plain English": the pool updates only at query-block
 * boundaries).  Fills pools[beta*cap ...] and counts[beta] for every block. */
static void pool_streaming(const double *amax, int nblk, int Bq, int s, int P,
                           int W, int32_t *pools, int32_t *counts, int cap,
                           cell_key *top /* P+1 entries */) {
  int ntop = 0, nold_prev = 0;
  for (int beta = 0; beta < nblk; ++beta) {
    int A = (beta * Bq) / s;
    int nrec = A < W ? A : W;
    int nold = A - nrec;
    for (int c = nold_prev; c < nold; ++c) { /* c leaves the recency window */
      cell_key nk = {amax[c], c};
      int pos = ntop;
      while (pos > 0 && cmp_cell_key(&nk, &top[pos - 1]) < 0) --pos;
      if (pos < P) {
        int last = ntop < P ? ntop : P - 1;
        for (int r = last; r > pos; --r) top[r] = top[r - 1];
        top[pos] = nk;
        if (ntop < P) ++ntop;
      }
    }
    nold_prev = nold;
    int32_t *pl = pools + (size_t)beta * cap;
    int n = 0;
    for (int c = nold; c < A; ++c) pl[n++] = c;
    for (int r = 0; r < ntop; ++r) pl[n++] = top[r].c;
    counts[beta] = n;
  }
}

/* ------------------------------------------------------------------------ */
/* RoPE.  [rainbus] 前置知识 "RoPE 旋转位置编码": q and k are rotated by R(i)
 * and R(j) so that their product depends only on the offset.  Half-split
 * pairing (x_i, x_{i+d/2}) with angle pos*theta_i, theta_i = base^(-2i/d).  */
/* ------------------------------------------------------------------------ */
static void rope_rotate(const float *x, double pos, int d, double base,
                        double *out) {
  int h = d / 2;
  for (int i = 0; i < h; ++i) {
    double theta = pow(base, -2.0 * (double)i / (double)d);
    double ang = pos * theta;
    double cs = cos(ang), sn = sin(ang);
    double x0 = (double)x[i], x1 = (double)x[i + h];
    out[i] = x0 * cs - x1 * sn;
    out[i + h] = x0 * sn + x1 * cs;
  }
}

/* ------------------------------------------------------------------------ */
/* Cell score.  [rainbus] 核心方法 ("内容匹配项加范数加权的 erf 相对位置偏置"),
 * 局限与改进 (available cells satisfy i - p_c > 0 and g_h >= erf(2));
 * [ai.info] "Methodology in Plain English" (content term plus a position bias
 * that grows with distance and is scaled by the norm; sigma_h, lambda_h).   */
/* ------------------------------------------------------------------------ */
static double cell_score(const float *qn, const double *kbar_c, double a_c,
                         int c, int n, int d, int s, double lambda,
                         double sigma) {
  double dot = 0.0;
  for (int i = 0; i < d; ++i) dot += (double)qn[i] * kbar_c[i];
  double p_c = (double)c * s + 0.5 * s;
  return dot + lambda * a_c * erf(sigma * ((double)n - p_c) / (double)s);
}

typedef struct {
  double u;
  int c;
} scored_cell;

/* (u desc, c asc) */
static int cmp_scored(const void *x, const void *y) {
  const scored_cell *p = (const scored_cell *)x, *q = (const scored_cell *)y;
  if (p->u > q->u) return -1;
  if (p->u < q->u) return 1;
  return (p->c < q->c) ? -1 : (p->c > q->c);
}

/* ------------------------------------------------------------------------ */
/* NoPE readout + RMSNorm.  [rainbus] 方法步骤详情 ⑥ ("选中 token 上做 NoPE
 * softmax 再 RMSNorm"), 前置知识 NoPE (position only affects selection);
 * [ai.info] "Key Contributions" 1 (unrotated queries and keys).             */
/* ------------------------------------------------------------------------ */
static void readout(const float *q, const float *k, const float *v, int d,
                    int s, int n, const int32_t *sel, int nsel, double eps,
                    double *o) {
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  if (nsel <= 0) return; /* no available cell: the branch contributes 0 */
  const float *qn = q + (size_t)n * d;
  double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int r = 0; r < nsel; ++r)
    for (int t = sel[r] * s; t < (sel[r] + 1) * s; ++t) {
      const float *kt = k + (size_t)t * d;
      double l = 0.0;
      for (int i = 0; i < d; ++i) l += (double)qn[i] * (double)kt[i];
      l *= scale;
      if (l > mx) mx = l;
    }
  double den = 0.0;
  for (int r = 0; r < nsel; ++r)
    for (int t = sel[r] * s; t < (sel[r] + 1) * s; ++t) {
      const float *kt = k + (size_t)t * d;
      const float *vt = v + (size_t)t * d;
      double l = 0.0;
      for (int i = 0; i < d; ++i) l += (double)qn[i] * (double)kt[i];
      double p = exp(l * scale - mx);
      den += p;
      for (int i = 0; i < d; ++i) o[i] += p * (double)vt[i];
    }
  double ms = 0.0;
  for (int i = 0; i < d; ++i) {
    o[i] /= den;
    ms += o[i] * o[i];
  }
  double r = 1.0 / sqrt(ms / (double)d + eps);
  for (int i = 0; i < d; ++i) o[i] *= r;
}

/* ------------------------------------------------------------------------ */
/* Sliding-window RoPE branch.  [rainbus] 方法步骤详情 ② ("在 w=512 窗口内做
 * RoPE 注意力"); [ai.info] "Methodology in Plain English" (ordinary sliding
 * window of 512 tokens with RoPE, fixed radius).  Keys j in
 * [max(0, n-w+1), n].  krot holds the rotated keys of this head.             */
/* ------------------------------------------------------------------------ */
static void window_branch(const float *qn, double pos_n, const double *krot,
                          const float *v, int d, int w, int n, double base,
                          double *o) {
  double qr[256];
  rope_rotate(qn, pos_n, d, base, qr);
  int j0 = n - w + 1 < 0 ? 0 : n - w + 1;
  double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int j = j0; j <= n; ++j) {
    const double *kj = krot + (size_t)j * d;
    double l = 0.0;
    for (int i = 0; i < d; ++i) l += qr[i] * kj[i];
    l *= scale;
    if (l > mx) mx = l;
  }
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  double den = 0.0;
  for (int j = j0; j <= n; ++j) {
    const double *kj = krot + (size_t)j * d;
    const float *vj = v + (size_t)j * d;
    double l = 0.0;
    for (int i = 0; i < d; ++i) l += qr[i] * kj[i];
    double p = exp(l * scale - mx);
    den += p;
    for (int i = 0; i < d; ++i) o[i] += p * (double)vj[i];
  }
  for (int i = 0; i < d; ++i) o[i] /= den;
}

/* ------------------------------------------------------------------------ */
/* Exported entry points (called through ctypes from the tests).             */
/* ------------------------------------------------------------------------ */

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

int fso_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* kbar [BH, N/s, d], amax [BH, N/s] for BH = batch*heads head slices. */
int fso_cells(const float *k, int BH, int N, int d, int s, double *kbar,
              double *amax, int nthreads) {
  if (N % s) return 1;
  int C = N / s;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int bh = 0; bh < BH; ++bh)
    cell_summaries(k + (size_t)bh * N * d, N, d, s, kbar + (size_t)bh * C * d,
                   amax + (size_t)bh * C);
  return 0;
}

/* Pools of every query block from per-cell norms amax [BH, C].
 * streaming = 0: definition (sort per block); 1: running top-P (FS-L only).
 * pool [BH, nblk, cap], count [BH, nblk], gap_rel [BH, nblk] (nullable). */
int fso_pools(const double *amax, int BH, int N, int s, int Bq, int P, int W,
              int mode, int streaming, int32_t *pool, int32_t *count,
              double *gap_rel, int cap, int nthreads) {
  if (N % Bq || Bq % s) return 1;
  int C = N / s, nblk = N / Bq;
  int need = mode == 1 ? (nblk - 1) * Bq / s : P + W;
  if (cap < need) return 2;
  if (streaming && mode != 0) return 3;
  set_threads(nthreads);
  if (streaming) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
      cell_key *top = (cell_key *)malloc(sizeof(cell_key) * (size_t)(P + 1));
      pool_streaming(amax + (size_t)bh * C, nblk, Bq, s, P, W,
                     pool + (size_t)bh * nblk * cap, count + (size_t)bh * nblk,
                     cap, top);
      free(top);
    }
    return 0;
  }
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
  for (int bh = 0; bh < BH; ++bh)
    for (int beta = 0; beta < nblk; ++beta) {
      cell_key *scratch = (cell_key *)malloc(sizeof(cell_key) * (size_t)(C + 1));
      double g;
      int A = beta * Bq / s;
      size_t o = (size_t)bh * nblk + beta;
      count[o] = pool_definition(amax + (size_t)bh * C, A, P, W, mode,
                                 pool + o * cap, &g, scratch);
      if (gap_rel) gap_rel[o] = g;
      free(scratch);
    }
  return 0;
}

/* Scores u of every cell of the pool of query n's block, one head slice.
 * Returns the pool size; writes pool ids and their scores (pool order). */
int fso_scores(const float *q, const float *k, int N, int d, int s, int Bq,
               int P, int W, int mode, double lambda, double sigma, int n,
               int32_t *pool_out, double *u_out) {
  int C = N / s;
  double *kbar = (double *)malloc(sizeof(double) * (size_t)C * d);
  double *amax = (double *)malloc(sizeof(double) * (size_t)C);
  cell_key *scratch = (cell_key *)malloc(sizeof(cell_key) * (size_t)(C + 1));
  cell_summaries(k, N, d, s, kbar, amax);
  int A = (n / Bq) * Bq / s;
  double g;
  int np = pool_definition(amax, A, P, W, mode, pool_out, &g, scratch);
  for (int r = 0; r < np; ++r) {
    int c = pool_out[r];
    u_out[r] = cell_score(q + (size_t)n * d, kbar + (size_t)c * d, amax[c], c,
                          n, d, s, lambda, sigma);
  }
  free(kbar);
  free(amax);
  free(scratch);
  return np;
}

/* NoPE readout + RMSNorm of query n over an explicit list of cells (one head
 * slice); used to check a kernel's output on the kernel's own selection where
 * a near-tie made two selections equally correct. */
int fso_readout(const float *q, const float *k, const float *v, int N, int d,
                int s, int n, const int32_t *sel, int nsel, double eps,
                double *o) {
  (void)N;
  readout(q, k, v, d, s, n, sel, nsel, eps, o);
  return 0;
}

/* Full forward for the requested rows of every head slice.
 *   q, k, v          [BH, N, d] float (bf16-rounded values)
 *   lambda, sigma,
 *   mix              [H] per-head routing weight, erf sharpness, branch mix
 *   rows             [nrows] query positions, or NULL for all N rows
 *   out              [BH, nrows, d]           (required)
 *   o_win, o_long    [BH, nrows, d]           (nullable)
 *   sel              [BH, nrows, K] int32, -1 padded, (u desc, c asc) order
 *   sel_score        [BH, nrows, K]           (nullable)
 *   gap_rel          [BH, nrows] relative gap between the K-th and (K+1)-th
 *                    ranked scores (INFINITY if |pool| <= K)   (nullable)
 *   pool_gap         [BH, nrows] relative norm gap that fixed the pool of the
 *                    row's block (INFINITY if no older cell was dropped)
 * pos_offset shifts every RoPE position by a constant (for the relative-
 * position check); it does not move cells or windows. */
int fso_forward(const float *q, const float *k, const float *v, int BH, int H,
                int N, int d, int w, int s, int K, int P, int W, int Bq,
                double rope_base, double rms_eps, int mode, double pos_offset,
                const double *lambda, const double *sigma, const double *mix,
                const int32_t *rows, int nrows, double *out, double *o_win,
                double *o_long, int32_t *sel, double *sel_score,
                double *gap_rel, double *pool_gap, int nthreads) {
  if (N % Bq || Bq % s || d > 256 || d % 2 || K < 0 || K > 64) return 1;
  if (rows == NULL) nrows = N;
  for (int r = 0; rows && r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return 4;
  int C = N / s, nblk = N / Bq;
  int cap = mode == 1 ? C : P + W;
  set_threads(nthreads);
  for (int bh = 0; bh < BH; ++bh) {
    int h = bh % H;
    const float *qh = q + (size_t)bh * N * d;
    const float *kh = k + (size_t)bh * N * d;
    const float *vh = v + (size_t)bh * N * d;
    double *kbar = (double *)malloc(sizeof(double) * (size_t)C * d);
    double *amax = (double *)malloc(sizeof(double) * (size_t)C);
    double *krot = (double *)malloc(sizeof(double) * (size_t)N * d);
    char *need_key = (char *)calloc((size_t)N, 1);
    char *need_blk = (char *)calloc((size_t)nblk, 1);
    int32_t *pools = (int32_t *)malloc(sizeof(int32_t) * (size_t)nblk * cap);
    int32_t *pcount = (int32_t *)malloc(sizeof(int32_t) * (size_t)nblk);
    double *pgap = (double *)malloc(sizeof(double) * (size_t)nblk);
    cell_summaries(kh, N, d, s, kbar, amax);
    for (int r = 0; r < nrows; ++r) {
      int n = rows ? rows[r] : r;
      need_blk[n / Bq] = 1;
      int j0 = n - w + 1 < 0 ? 0 : n - w + 1;
      for (int j = j0; j <= n; ++j) need_key[j] = 1;
    }
#pragma omp parallel for schedule(dynamic, 64)
    for (int j = 0; j < N; ++j)
      if (need_key[j])
        rope_rotate(kh + (size_t)j * d, (double)j + pos_offset, d, rope_base,
                    krot + (size_t)j * d);
#pragma omp parallel for schedule(dynamic, 1)
    for (int beta = 0; beta < nblk; ++beta) {
      if (!need_blk[beta]) continue;
      cell_key *scratch = (cell_key *)malloc(sizeof(cell_key) * (size_t)(C + 1));
      int A = beta * Bq / s;
      pcount[beta] = pool_definition(amax, A, P, W, mode,
                                     pools + (size_t)beta * cap, &pgap[beta],
                                     scratch);
      free(scratch);
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (int r = 0; r < nrows; ++r) {
      int n = rows ? rows[r] : r;
      int beta = n / Bq;
      int np = pcount[beta];
      const int32_t *pl = pools + (size_t)beta * cap;
      const float *qn = qh + (size_t)n * d;
      scored_cell *sc = (scored_cell *)malloc(sizeof(scored_cell) * (size_t)(np + 1));
      for (int t = 0; t < np; ++t) {
        int c = pl[t];
        sc[t].u = cell_score(qn, kbar + (size_t)c * d, amax[c], c, n, d, s,
                             lambda[h], sigma[h]);
        sc[t].c = c;
      }
      qsort(sc, (size_t)np, sizeof(scored_cell), cmp_scored);
      int nsel = np < K ? np : K;
      int32_t chosen[64];
      size_t ro = (size_t)bh * nrows + r;
      for (int t = 0; t < K; ++t) {
        chosen[t] = t < nsel ? sc[t].c : -1;
        if (sel) sel[ro * K + t] = chosen[t];
        if (sel_score) sel_score[ro * K + t] = t < nsel ? sc[t].u : 0.0;
      }
      if (gap_rel) {
        double g = INFINITY;
        if (np > K && K > 0) {
          double x = sc[K - 1].u, y = sc[K].u;
          double den = fabs(x) > fabs(y) ? fabs(x) : fabs(y);
          g = den > 0 ? (x - y) / den : 0.0;
        }
        gap_rel[ro] = g;
      }
      if (pool_gap) pool_gap[ro] = pgap[beta];
      free(sc);
      double ol[256], ow[256];
      readout(qh, kh, vh, d, s, n, chosen, nsel, rms_eps, ol);
      window_branch(qn, (double)n + pos_offset, krot, vh, d, w, n, rope_base,
                    ow);
      for (int i = 0; i < d; ++i) {
        out[ro * d + i] = ow[i] + mix[h] * ol[i];
        if (o_win) o_win[ro * d + i] = ow[i];
        if (o_long) o_long[ro * d + i] = ol[i];
      }
    }
    free(kbar);
    free(amax);
    free(krot);
    free(need_key);
    free(need_blk);
    free(pools);
    free(pcount);
    free(pgap);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward pass.  [rainbus] 方法步骤详情 (training: the hard top-P / top-K
 * indices carry no gradient), 核心方法 (the per-head mixing coefficient is
 * learned), 局限与改进 (sigma_h and lambda_h are fixed, without gradient);
 * [ai.info] "Methodology in Plain English" (training paragraph: hard top-P
 * and top-K indices receive no gradient, routing scalars stay fixed).
 *
 * Given g = dL/dout for a scalar loss L, the pool and the selection of every
 * row are held fixed, so the gradient reaches q, k and v only through the two
 * softmax reads (and the RMSNorm of the long branch), plus the mix weight
 * m_h; kbar_c, a_c, lambda_h and sigma_h receive none.  Per row n, with the
 * window probabilities p_j over the rotated q~ = R(n) q_n, k~_j = R(j) k_j
 * and the long probabilities p_t over the selected tokens (unrotated):
 *   window  dv_j += p_j g;  ds_j = p_j (g.v_j - g.o_win);
 *           dq~ = sum_j ds_j k~_j / sqrt(d);  dk~_j += ds_j q~ / sqrt(d);
 *           dq_n += R(n)^T dq~;  dk_j += R(j)^T dk~_j
 *   long    dm_h += g.o^;  do^ = m_h g;  rho = (mean(o^2) + eps)^(-1/2),
 *           o^ = rho o, so do = rho do^ - rho^3 (o.do^) o / d;
 *           dv_t += p_t do;  dl_t = p_t (do.v_t - do.o);
 *           dq_n += sum_t dl_t k_t / sqrt(d);  dk_t += dl_t q_n / sqrt(d)
 * (the softmax rule ds = p (dp - p.dp) with dp_j = g.v_j and p.dp = g.o).  */
/* ------------------------------------------------------------------------ */

/* out = R(pos)^T y: the inverse rotation of one vector (pairs i, i + d/2). */
static void rope_rotate_t(const double *y, double pos, int d, double base,
                          double *out) {
  int h = d / 2;
  for (int i = 0; i < h; ++i) {
    double theta = pow(base, -2.0 * (double)i / (double)d);
    double ang = pos * theta;
    double cs = cos(ang), sn = sin(ang);
    double y0 = y[i], y1 = y[i + h];
    out[i] = y0 * cs + y1 * sn;
    out[i + h] = -y0 * sn + y1 * cs;
  }
}

/* Gradients of one head slice.  dq, dk, dv [N, d] are accumulated into
 * (zeroed by the caller); returns g . o^ summed over the rows (dm_h). */
static double backward_head(const float *q, const float *k, const float *v,
                            const double *g, int N, int d, int w, int s, int K,
                            int P, int W, int Bq, double base, double eps,
                            int mode, double lambda, double sigma, double mix,
                            double *dq, double *dk, double *dv) {
  int C = N / s, nblk = N / Bq;
  int cap = mode == 1 ? C : P + W;
  double scale = 1.0 / sqrt((double)d);
  double *kbar = (double *)malloc(sizeof(double) * (size_t)C * d);
  double *amax = (double *)malloc(sizeof(double) * (size_t)C);
  double *krot = (double *)malloc(sizeof(double) * (size_t)N * d);
  double *dkrot = (double *)calloc((size_t)N * d, sizeof(double));
  int32_t *pools = (int32_t *)malloc(sizeof(int32_t) * (size_t)nblk * cap);
  int32_t *pcount = (int32_t *)malloc(sizeof(int32_t) * (size_t)nblk);
  cell_key *scratch = (cell_key *)malloc(sizeof(cell_key) * (size_t)(C + 1));
  scored_cell *sc = (scored_cell *)malloc(sizeof(scored_cell) * (size_t)(cap + 1));
  double *pw = (double *)malloc(sizeof(double) * (size_t)w);
  double *pt = (double *)malloc(sizeof(double) * (size_t)K * s + 1);
  double dmix = 0.0;
  cell_summaries(k, N, d, s, kbar, amax);
  for (int j = 0; j < N; ++j)
    rope_rotate(k + (size_t)j * d, (double)j, d, base, krot + (size_t)j * d);
  for (int beta = 0; beta < nblk; ++beta) {
    double gap;
    pcount[beta] = pool_definition(amax, beta * Bq / s, P, W, mode,
                                   pools + (size_t)beta * cap, &gap, scratch);
  }
  for (int n = 0; n < N; ++n) {
    const float *qn = q + (size_t)n * d;
    const double *gn = g + (size_t)n * d;
    double qr[256], dqr[256], dqn[256], ow[256], ol[256], dol[256], tmp[256];
    for (int i = 0; i < d; ++i) dqn[i] = 0.0;
    /* window branch: forward again, then its backward in rotated space */
    rope_rotate(qn, (double)n, d, base, qr);
    int j0 = n - w + 1 < 0 ? 0 : n - w + 1;
    double mx = -INFINITY, den = 0.0;
    for (int j = j0; j <= n; ++j) {
      double l = 0.0;
      for (int i = 0; i < d; ++i) l += qr[i] * krot[(size_t)j * d + i];
      pw[j - j0] = l * scale;
      if (pw[j - j0] > mx) mx = pw[j - j0];
    }
    for (int j = j0; j <= n; ++j) {
      pw[j - j0] = exp(pw[j - j0] - mx);
      den += pw[j - j0];
    }
    for (int i = 0; i < d; ++i) ow[i] = 0.0;
    for (int j = j0; j <= n; ++j) {
      pw[j - j0] /= den;
      for (int i = 0; i < d; ++i) ow[i] += pw[j - j0] * (double)v[(size_t)j * d + i];
    }
    double g_ow = 0.0;
    for (int i = 0; i < d; ++i) g_ow += gn[i] * ow[i];
    for (int i = 0; i < d; ++i) dqr[i] = 0.0;
    for (int j = j0; j <= n; ++j) {
      double p = pw[j - j0], g_vj = 0.0;
      for (int i = 0; i < d; ++i) {
        g_vj += gn[i] * (double)v[(size_t)j * d + i];
        dv[(size_t)j * d + i] += p * gn[i];
      }
      double ds = p * (g_vj - g_ow) * scale;
      for (int i = 0; i < d; ++i) {
        dqr[i] += ds * krot[(size_t)j * d + i];
        dkrot[(size_t)j * d + i] += ds * qr[i];
      }
    }
    rope_rotate_t(dqr, (double)n, d, base, tmp);
    for (int i = 0; i < d; ++i) dqn[i] += tmp[i];
    /* long branch: the row's selection (held fixed), forward, backward */
    int beta = n / Bq, np = pcount[beta];
    const int32_t *pl = pools + (size_t)beta * cap;
    for (int t = 0; t < np; ++t) {
      sc[t].c = pl[t];
      sc[t].u = cell_score(qn, kbar + (size_t)pl[t] * d, amax[pl[t]], pl[t], n,
                           d, s, lambda, sigma);
    }
    qsort(sc, (size_t)np, sizeof(scored_cell), cmp_scored);
    int nsel = np < K ? np : K;
    if (nsel > 0) {
      int ntok = nsel * s;
      mx = -INFINITY;
      den = 0.0;
      for (int r = 0; r < nsel; ++r)
        for (int e = 0; e < s; ++e) {
          int tk = sc[r].c * s + e;
          double l = 0.0;
          for (int i = 0; i < d; ++i) l += (double)qn[i] * (double)k[(size_t)tk * d + i];
          pt[r * s + e] = l * scale;
          if (pt[r * s + e] > mx) mx = pt[r * s + e];
        }
      for (int x = 0; x < ntok; ++x) {
        pt[x] = exp(pt[x] - mx);
        den += pt[x];
      }
      for (int i = 0; i < d; ++i) ol[i] = 0.0;
      for (int r = 0; r < nsel; ++r)
        for (int e = 0; e < s; ++e) {
          int tk = sc[r].c * s + e;
          pt[r * s + e] /= den;
          for (int i = 0; i < d; ++i) ol[i] += pt[r * s + e] * (double)v[(size_t)tk * d + i];
        }
      double ms = 0.0;
      for (int i = 0; i < d; ++i) ms += ol[i] * ol[i];
      double rho = 1.0 / sqrt(ms / (double)d + eps);
      /* mix weight and RMSNorm */
      double o_dohat = 0.0;
      for (int i = 0; i < d; ++i) {
        dmix += gn[i] * ol[i] * rho;
        o_dohat += ol[i] * mix * gn[i];
      }
      for (int i = 0; i < d; ++i)
        dol[i] = rho * mix * gn[i] - rho * rho * rho * o_dohat * ol[i] / (double)d;
      /* softmax read */
      double do_o = 0.0;
      for (int i = 0; i < d; ++i) do_o += dol[i] * ol[i];
      for (int r = 0; r < nsel; ++r)
        for (int e = 0; e < s; ++e) {
          int tk = sc[r].c * s + e;
          double p = pt[r * s + e], do_v = 0.0;
          for (int i = 0; i < d; ++i) {
            do_v += dol[i] * (double)v[(size_t)tk * d + i];
            dv[(size_t)tk * d + i] += p * dol[i];
          }
          double dl = p * (do_v - do_o) * scale;
          for (int i = 0; i < d; ++i) {
            dqn[i] += dl * (double)k[(size_t)tk * d + i];
            dk[(size_t)tk * d + i] += dl * (double)qn[i];
          }
        }
    }
    for (int i = 0; i < d; ++i) dq[(size_t)n * d + i] += dqn[i];
  }
  /* rotated-key gradients back to the unrotated keys */
  for (int j = 0; j < N; ++j) {
    double tmp[256];
    rope_rotate_t(dkrot + (size_t)j * d, (double)j, d, base, tmp);
    for (int i = 0; i < d; ++i) dk[(size_t)j * d + i] += tmp[i];
  }
  free(kbar);
  free(amax);
  free(krot);
  free(dkrot);
  free(pools);
  free(pcount);
  free(scratch);
  free(sc);
  free(pw);
  free(pt);
  return dmix;
}

/* Gradients of L = sum(g * out) for every head slice.
 *   g                [BH, N, d] upstream gradient dL/dout
 *   dq, dk, dv       [BH, N, d] (written)
 *   dmix             [H] (written): summed over the batch
 * Same parameters as fso_forward (all rows, no position offset). */
int fso_backward(const float *q, const float *k, const float *v, int BH, int H,
                 int N, int d, int w, int s, int K, int P, int W, int Bq,
                 double rope_base, double rms_eps, int mode,
                 const double *lambda, const double *sigma, const double *mix,
                 const double *g, double *dq, double *dk, double *dv,
                 double *dmix, int nthreads) {
  if (N % Bq || Bq % s || d > 256 || d % 2 || K < 0 || K > 64 || w < 1) return 1;
  if (BH % H) return 1;
  double *part = (double *)malloc(sizeof(double) * (size_t)BH);
  memset(dq, 0, sizeof(double) * (size_t)BH * N * d);
  memset(dk, 0, sizeof(double) * (size_t)BH * N * d);
  memset(dv, 0, sizeof(double) * (size_t)BH * N * d);
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int bh = 0; bh < BH; ++bh) {
    size_t o = (size_t)bh * N * d;
    int h = bh % H;
    part[bh] = backward_head(q + o, k + o, v + o, g + o, N, d, w, s, K, P, W, Bq,
                             rope_base, rms_eps, mode, lambda[h], sigma[h], mix[h],
                             dq + o, dk + o, dv + o);
  }
  for (int h = 0; h < H; ++h) dmix[h] = 0.0;
  for (int bh = 0; bh < BH; ++bh) dmix[bh % H] += part[bh];  /* fixed order */
  free(part);
  return 0;
}
