/*
 * fp64 CPU oracle for fused edge attention over a destination-sorted CSR graph.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links or calls this file;
 * only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code, header, table or helper with the CUDA path.
 *
 * Every function writes out the plain definition: an explicit loop over the
 * edges of one destination row, a dense softmax over that row's edge list
 * (maximum, exponentials, sum, divide), and plain chain-rule gradients.  No
 * online softmax, no recomputation from the log-sum-exp, no blocking.
 *
 * Sources (the web pages that define the method):
 *  - "On Efficient Scaling of GNNs via IO-Aware Layers Implementations"
 *    (mlsanity.com abstract and the Yandex Research blog post): attention layers
 *    of the GATv2 / Graph Transformer kind whose edge-level attention values are
 *    the softmax over each node's neighbourhood; the fused kernels must give the
 *    same result as materialising them ("Attention-based layers" paragraph).
 *  - Graph Transformer score q_i . k_j / sqrt(D) and GATv2 score
 *    a_h . LeakyReLU(W_l x_i + W_r x_j), both per head, as named in the layer
 *    definitions the pages cite ("Masked Label Prediction: Unified Message
 *    Passing Model" for the Graph Transformer, "How Attentive are Graph
 *    Attention Networks?" for GATv2).
 *
 * Conventions (readings where the pages are silent):
 *  - CSR row i is the destination; indices[indptr[i] .. indptr[i+1]) are the
 *    sources j.  Node tensors are [N, H, D] row-major.
 *  - lse[i,h] is the natural log-sum-exp of the row's scores; an empty row has
 *    out = 0 and lse = -inf and contributes to no gradient.
 *  - GATv2: W_l multiplies the destination features, W_r the source features;
 *    the aggregated value is the source projection FR_j = x_j W_r.
 *    LeakyReLU'(0) is taken as the negative slope.  The projections are layer
 *    outputs stored in the layer's dtype; the `store` argument rounds them
 *    the same way before the edge stage uses them.
 *
 * Parallelism: OpenMP over independent rows (or sources); each output element
 * is produced by one thread in a fixed order, so results do not depend on the
 * thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Graph preprocessing                                                       */
/* ------------------------------------------------------------------------ */

/* Transposed CSR by counting sort: t_indptr[j] .. t_indptr[j+1] lists the
 * destinations of source j.  Rows are visited in ascending order, so each
 * source's destination list comes out ascending.  Returns 0. */
int oracle_transpose(int64_t N, const int32_t *indptr, const int32_t *indices,
                     int32_t *t_indptr, int32_t *t_dst) {
    int64_t E = indptr[N];
    int64_t *cursor = (int64_t *)calloc((size_t)N + 1, sizeof(int64_t));
    if (!cursor) return -1;
    for (int64_t e = 0; e < E; ++e) cursor[indices[e] + 1] += 1;
    for (int64_t j = 0; j < N; ++j) cursor[j + 1] += cursor[j];
    for (int64_t j = 0; j <= N; ++j) t_indptr[j] = (int32_t)cursor[j];
    for (int64_t i = 0; i < N; ++i)
        for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e)
            t_dst[cursor[indices[e]]++] = (int32_t)i;
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Graph Transformer                                                         */
/* ------------------------------------------------------------------------ */

/* Scores of one row for head h: s[e - b] = (q_i . k_j) / sqrt(D), plus the
 * edge's bias B[e, h] when B is given (the Graph Transformer with an additive
 * per-edge, per-head score term; B is [E, H] in CSR edge order). */
static void gt_row_scores(int64_t i, int h, int H, int D, const int32_t *indptr,
                          const int32_t *indices, const double *Q, const double *K,
                          const double *B, double *s) {
    int64_t b = indptr[i], en = indptr[i + 1];
    const double *q = Q + ((size_t)i * H + h) * D;
    double inv = 1.0 / sqrt((double)D);
    for (int64_t e = b; e < en; ++e) {
        const double *k = K + ((size_t)indices[e] * H + h) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * k[d];
        s[e - b] = dot * inv + (B ? B[(size_t)e * H + h] : 0.0);
    }
}

/* Dense softmax over n scores: p = exp(s - max) / sum.  Returns the natural
 * log-sum-exp (max + log(sum)); -inf for n == 0. */
static double softmax(int64_t n, const double *s, double *p) {
    if (n == 0) return -INFINITY;
    double m = s[0];
    for (int64_t t = 1; t < n; ++t) if (s[t] > m) m = s[t];
    double z = 0.0;
    for (int64_t t = 0; t < n; ++t) { p[t] = exp(s[t] - m); z += p[t]; }
    for (int64_t t = 0; t < n; ++t) p[t] /= z;
    return m + log(z);
}

static int64_t max_degree(int64_t N, const int32_t *indptr) {
    int64_t mx = 0;
    for (int64_t i = 0; i < N; ++i) {
        int64_t d = (int64_t)indptr[i + 1] - indptr[i];
        if (d > mx) mx = d;
    }
    return mx;
}

/* GT forward for the listed rows.  out_rows[r] is [H, D], lse_rows[r] is [H];
 * B: optional [E, H] score bias (NULL: none). */
static int gt_fwd_rows_impl(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                            const double *Q, const double *K, const double *V, const double *B,
                            int64_t nrows, const int64_t *rows, double *out_rows, double *lse_rows) {
    int64_t md = max_degree(N, indptr);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        if (!s || !p) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (int64_t r = 0; r < nrows; ++r) {
                int64_t i = rows[r];
                int64_t b = indptr[i], n = indptr[i + 1] - b;
                for (int h = 0; h < H; ++h) {
                    gt_row_scores(i, h, H, D, indptr, indices, Q, K, B, s);
                    lse_rows[r * H + h] = softmax(n, s, p);
                    double *o = out_rows + ((size_t)r * H + h) * D;
                    for (int d = 0; d < D; ++d) o[d] = 0.0;
                    for (int64_t t = 0; t < n; ++t) {
                        const double *v = V + ((size_t)indices[b + t] * H + h) * D;
                        for (int d = 0; d < D; ++d) o[d] += p[t] * v[d];
                    }
                }
            }
        }
        free(s);
        free(p);
    }
    return err;
}

int oracle_gt_fwd_rows(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                       const double *Q, const double *K, const double *V,
                       int64_t nrows, const int64_t *rows, double *out_rows, double *lse_rows) {
    return gt_fwd_rows_impl(N, indptr, indices, H, D, Q, K, V, NULL, nrows, rows, out_rows, lse_rows);
}

/* GT forward of every row; B: optional [E, H] score bias (NULL: none). */
int oracle_gt_bias_fwd(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                       const double *Q, const double *K, const double *V, const double *B,
                       double *out, double *lse) {
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    if (!rows) return -1;
    for (int64_t i = 0; i < N; ++i) rows[i] = i;
    int rc = gt_fwd_rows_impl(N, indptr, indices, H, D, Q, K, V, B, N, rows, out, lse);
    free(rows);
    return rc;
}

int oracle_gt_fwd(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                  const double *Q, const double *K, const double *V, double *out, double *lse) {
    return oracle_gt_bias_fwd(N, indptr, indices, H, D, Q, K, V, NULL, out, lse);
}

/* Softmax Jacobian of one row, head h.  Fills p[t] (weights), ds[t]
 * (dL/ds = p (dP - sum_t' p dP)) with dP[t] = dO_i . v_j. */
static void gt_row_grad(int64_t i, int h, int H, int D, const int32_t *indptr,
                        const int32_t *indices, const double *Q, const double *K,
                        const double *V, const double *B, const double *dO, double *s, double *p,
                        double *ds) {
    int64_t b = indptr[i], n = indptr[i + 1] - b;
    gt_row_scores(i, h, H, D, indptr, indices, Q, K, B, s);
    softmax(n, s, p);
    const double *g = dO + ((size_t)i * H + h) * D;
    double sum_pdp = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        const double *v = V + ((size_t)indices[b + t] * H + h) * D;
        double dp = 0.0;
        for (int d = 0; d < D; ++d) dp += g[d] * v[d];
        ds[t] = dp;
        sum_pdp += p[t] * dp;
    }
    for (int64_t t = 0; t < n; ++t) ds[t] = p[t] * (ds[t] - sum_pdp);
}

/* dQ for the listed rows: dQ_i = sum_j dS_ij k_j / sqrt(D). */
int oracle_gt_bwd_dq_rows(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                          const double *Q, const double *K, const double *V, const double *dO,
                          int64_t nrows, const int64_t *rows, double *dq_rows) {
    int64_t md = max_degree(N, indptr);
    double inv = 1.0 / sqrt((double)D);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        double *ds = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        if (!s || !p || !ds) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (int64_t r = 0; r < nrows; ++r) {
                int64_t i = rows[r];
                int64_t b = indptr[i], n = indptr[i + 1] - b;
                for (int h = 0; h < H; ++h) {
                    double *o = dq_rows + ((size_t)r * H + h) * D;
                    for (int d = 0; d < D; ++d) o[d] = 0.0;
                    if (n == 0) continue;
                    gt_row_grad(i, h, H, D, indptr, indices, Q, K, V, NULL, dO, s, p, ds);
                    for (int64_t t = 0; t < n; ++t) {
                        const double *k = K + ((size_t)indices[b + t] * H + h) * D;
                        for (int d = 0; d < D; ++d) o[d] += ds[t] * k[d] * inv;
                    }
                }
            }
        }
        free(s);
        free(p);
        free(ds);
    }
    return err;
}

/* dK, dV for the listed source nodes.  For each edge (i <- j) the full row i
 * is re-solved (dense softmax), then dV_j += p_ij dO_i and
 * dK_j += dS_ij q_i / sqrt(D).  Edges of source j are visited in ascending
 * destination order.  t_indptr/t_dst come from oracle_transpose. */
int oracle_gt_bwd_dkdv_srcs(int64_t N, const int32_t *indptr, const int32_t *indices,
                            const int32_t *t_indptr, const int32_t *t_dst, int H, int D,
                            const double *Q, const double *K, const double *V, const double *dO,
                            int64_t nsrc, const int64_t *srcs, double *dk_rows, double *dv_rows) {
    int64_t md = max_degree(N, indptr);
    double inv = 1.0 / sqrt((double)D);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        double *ds = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        if (!s || !p || !ds) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < nsrc; ++r) {
                int64_t j = srcs[r];
                double *dk = dk_rows + (size_t)r * H * D;
                double *dv = dv_rows + (size_t)r * H * D;
                for (int64_t x = 0; x < (int64_t)H * D; ++x) { dk[x] = 0.0; dv[x] = 0.0; }
                for (int64_t te = t_indptr[j]; te < t_indptr[j + 1]; ++te) {
                    int64_t i = t_dst[te];
                    int64_t b = indptr[i], n = indptr[i + 1] - b;
                    for (int h = 0; h < H; ++h) {
                        gt_row_grad(i, h, H, D, indptr, indices, Q, K, V, NULL, dO, s, p, ds);
                        const double *q = Q + ((size_t)i * H + h) * D;
                        const double *g = dO + ((size_t)i * H + h) * D;
                        /* every occurrence of j in row i (duplicates are separate edges) */
                        for (int64_t t = 0; t < n; ++t) {
                            if (indices[b + t] != j) continue;
                            for (int d = 0; d < D; ++d) {
                                dv[h * D + d] += p[t] * g[d];
                                dk[h * D + d] += ds[t] * q[d] * inv;
                            }
                        }
                    }
                    /* a row holding j twice appears twice in t_dst: skip the repeat */
                    while (te + 1 < t_indptr[j + 1] && t_dst[te + 1] == i) ++te;
                }
            }
        }
        free(s);
        free(p);
        free(ds);
    }
    return err;
}

/* Full GT backward: per row, the softmax Jacobian gives p_e and dS_e for every
 * edge; dQ_i is summed per row; dK_j and dV_j are summed per source over its
 * edges in ascending edge order (the oracle's own edge grouping). */
int oracle_gt_bias_bwd(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                       const double *Q, const double *K, const double *V, const double *B,
                       const double *dO, double *dQ, double *dK, double *dV, double *dB);

int oracle_gt_bwd(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                  const double *Q, const double *K, const double *V, const double *dO,
                  double *dQ, double *dK, double *dV) {
    return oracle_gt_bias_bwd(N, indptr, indices, H, D, Q, K, V, NULL, dO, dQ, dK, dV, NULL);
}

/* As oracle_gt_bwd with the optional [E, H] score bias B; dB (if given,
 * [E, H]) receives dL/dB = dS of every edge (the bias enters the score with
 * unit weight). */
int oracle_gt_bias_bwd(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                       const double *Q, const double *K, const double *V, const double *B,
                       const double *dO, double *dQ, double *dK, double *dV, double *dB) {
    int64_t E = indptr[N];
    int64_t md = max_degree(N, indptr);
    double inv = 1.0 / sqrt((double)D);
    double *P = (double *)malloc(sizeof(double) * (size_t)(E * H + 1));
    double *DS = (double *)malloc(sizeof(double) * (size_t)(E * H + 1));
    int64_t *eptr = (int64_t *)calloc((size_t)N + 1, sizeof(int64_t));
    int64_t *eids = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E + 1));
    int32_t *erow = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int err = 0;
    if (!P || !DS || !eptr || !eids || !erow) err = -1;
    if (!err) {
#pragma omp parallel
        {
            double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
            double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
            double *ds = (double *)malloc(sizeof(double) * (size_t)(md + 1));
            if (!s || !p || !ds) {
#pragma omp atomic write
                err = -1;
            } else {
#pragma omp for schedule(dynamic, 64)
                for (int64_t i = 0; i < N; ++i) {
                    int64_t b = indptr[i], n = indptr[i + 1] - b;
                    for (int64_t e = b; e < b + n; ++e) erow[e] = (int32_t)i;
                    for (int h = 0; h < H; ++h) {
                        double *o = dQ + ((size_t)i * H + h) * D;
                        for (int d = 0; d < D; ++d) o[d] = 0.0;
                        if (n == 0) continue;
                        gt_row_grad(i, h, H, D, indptr, indices, Q, K, V, B, dO, s, p, ds);
                        for (int64_t t = 0; t < n; ++t) {
                            P[(b + t) * H + h] = p[t];
                            DS[(b + t) * H + h] = ds[t];
                            const double *k = K + ((size_t)indices[b + t] * H + h) * D;
                            for (int d = 0; d < D; ++d) o[d] += ds[t] * k[d] * inv;
                        }
                    }
                }
            }
            free(s);
            free(p);
            free(ds);
        }
    }
    if (!err) {
        /* group edge ids by source, ascending edge id within a source */
        for (int64_t e = 0; e < E; ++e) eptr[indices[e] + 1] += 1;
        for (int64_t j = 0; j < N; ++j) eptr[j + 1] += eptr[j];
        int64_t *cur = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N + 1));
        if (!cur) err = -1;
        if (!err) {
            memcpy(cur, eptr, sizeof(int64_t) * (size_t)(N + 1));
            for (int64_t e = 0; e < E; ++e) eids[cur[indices[e]]++] = e;
            free(cur);
#pragma omp parallel for schedule(dynamic, 64)
            for (int64_t j = 0; j < N; ++j) {
                double *dk = dK + (size_t)j * H * D;
                double *dv = dV + (size_t)j * H * D;
                for (int64_t x = 0; x < (int64_t)H * D; ++x) { dk[x] = 0.0; dv[x] = 0.0; }
                for (int64_t t = eptr[j]; t < eptr[j + 1]; ++t) {
                    int64_t e = eids[t];
                    int64_t i = erow[e];
                    for (int h = 0; h < H; ++h) {
                        const double *q = Q + ((size_t)i * H + h) * D;
                        const double *g = dO + ((size_t)i * H + h) * D;
                        double pe = P[e * H + h], dse = DS[e * H + h];
                        for (int d = 0; d < D; ++d) {
                            dv[h * D + d] += pe * g[d];
                            dk[h * D + d] += dse * q[d] * inv;
                        }
                    }
                }
            }
        }
    }
    if (!err && dB)
        for (int64_t x = 0; x < E * H; ++x) dB[x] = DS[x];
    free(P);
    free(DS);
    free(eptr);
    free(eids);
    free(erow);
    return err;
}

/* ------------------------------------------------------------------------ */
/* GATv2                                                                     */
/* ------------------------------------------------------------------------ */

static inline double lrelu(double z, double slope) { return z > 0.0 ? z : slope * z; }
static inline double lrelu_grad(double z, double slope) { return z > 0.0 ? 1.0 : slope; }

/* Round a double to the nearest bfloat16 (ties to even), returned as a
 * double: first to float (the projections are accumulated to a float), then
 * the float's 32-bit pattern to its upper 16 bits with round-half-even. */
double oracle_round_bf16(double x) {
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof(u));
    if ((u & 0x7f800000u) != 0x7f800000u) {  /* finite */
        u += 0x7fffu + ((u >> 16) & 1u);
        u &= 0xffff0000u;
    }
    memcpy(&f, &u, sizeof(f));
    return (double)f;
}

/* Storage rounding of the GATv2 projections: 0 keeps doubles, 1 rounds to
 * float, 2 to bfloat16.  The layer stores FL and FR in its tensor dtype and
 * the edge stage (forward and backward) consumes the stored values, so the
 * LeakyReLU branch is decided on the same numbers the kernels see. */
static void round_storage(int64_t n, double *x, int mode) {
    if (mode == 1)
        for (int64_t t = 0; t < n; ++t) x[t] = (double)(float)x[t];
    else if (mode == 2)
        for (int64_t t = 0; t < n; ++t) x[t] = oracle_round_bf16(x[t]);
}

/* Y[n, c] = sum_f X[n, f] W[f, c]   (X [N, F], W [F, C], Y [N, C]) */
int oracle_matmul(int64_t N, int F, int C, const double *X, const double *W, double *Y) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        double *y = Y + (size_t)n * C;
        for (int c = 0; c < C; ++c) y[c] = 0.0;
        for (int f = 0; f < F; ++f) {
            double x = X[(size_t)n * F + f];
            const double *w = W + (size_t)f * C;
            for (int c = 0; c < C; ++c) y[c] += x * w[c];
        }
    }
    return 0;
}

/* GATv2 scores of one row, head h:
 * e[t] = sum_d a[h,d] LeakyReLU(FL[i,h,d] + FR[j,h,d]). */
static void gatv2_row_scores(int64_t i, int h, int H, int D, const int32_t *indptr,
                             const int32_t *indices, const double *FL, const double *FR,
                             const double *a, double slope, double *e) {
    int64_t b = indptr[i], en = indptr[i + 1];
    const double *fl = FL + ((size_t)i * H + h) * D;
    const double *ah = a + (size_t)h * D;
    for (int64_t x = b; x < en; ++x) {
        const double *fr = FR + ((size_t)indices[x] * H + h) * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += ah[d] * lrelu(fl[d] + fr[d], slope);
        e[x - b] = acc;
    }
}

/* GATv2 forward on given projections FL = X W_l, FR = X W_r, for listed rows:
 * out_i = sum_j softmax_j(e_ij) FR_j. */
int oracle_gatv2_fwd_rows(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                          const double *FL, const double *FR, const double *a, double slope,
                          int64_t nrows, const int64_t *rows, double *out_rows, double *lse_rows) {
    int64_t md = max_degree(N, indptr);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        if (!s || !p) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (int64_t r = 0; r < nrows; ++r) {
                int64_t i = rows[r];
                int64_t b = indptr[i], n = indptr[i + 1] - b;
                for (int h = 0; h < H; ++h) {
                    gatv2_row_scores(i, h, H, D, indptr, indices, FL, FR, a, slope, s);
                    lse_rows[r * H + h] = softmax(n, s, p);
                    double *o = out_rows + ((size_t)r * H + h) * D;
                    for (int d = 0; d < D; ++d) o[d] = 0.0;
                    for (int64_t t = 0; t < n; ++t) {
                        const double *fr = FR + ((size_t)indices[b + t] * H + h) * D;
                        for (int d = 0; d < D; ++d) o[d] += p[t] * fr[d];
                    }
                }
            }
        }
        free(s);
        free(p);
    }
    return err;
}

/* Full GATv2 layer forward from X: FL = X W_l, FR = X W_r (stored with the
 * rounding `store`, see round_storage), then the edge stage. */
int oracle_gatv2_fwd(int64_t N, int F, int H, int D, const int32_t *indptr, const int32_t *indices,
                     const double *X, const double *Wl, const double *Wr, const double *a,
                     double slope, int store, double *FL, double *FR, double *out, double *lse) {
    int HD = H * D;
    oracle_matmul(N, F, HD, X, Wl, FL);
    oracle_matmul(N, F, HD, X, Wr, FR);
    round_storage(N * HD, FL, store);
    round_storage(N * HD, FR, store);
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    if (!rows) return -1;
    for (int64_t i = 0; i < N; ++i) rows[i] = i;
    int rc = oracle_gatv2_fwd_rows(N, indptr, indices, H, D, FL, FR, a, slope, N, rows, out, lse);
    free(rows);
    return rc;
}

/* Per-edge backward quantities of one GATv2 row, head h, given dO:
 *   p[t]  = softmax weight,   dp[t] = dO_i . FR_j,
 *   de[t] = p[t] (dp[t] - sum_t' p dp)   (gradient w.r.t. the score e). */
static void gatv2_row_grad(int64_t i, int h, int H, int D, const int32_t *indptr,
                           const int32_t *indices, const double *FL, const double *FR,
                           const double *a, double slope, const double *dO,
                           double *s, double *p, double *de) {
    int64_t b = indptr[i], n = indptr[i + 1] - b;
    gatv2_row_scores(i, h, H, D, indptr, indices, FL, FR, a, slope, s);
    softmax(n, s, p);
    const double *g = dO + ((size_t)i * H + h) * D;
    double sum_pdp = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        const double *fr = FR + ((size_t)indices[b + t] * H + h) * D;
        double dp = 0.0;
        for (int d = 0; d < D; ++d) dp += g[d] * fr[d];
        de[t] = dp;
        sum_pdp += p[t] * dp;
    }
    for (int64_t t = 0; t < n; ++t) de[t] = p[t] * (de[t] - sum_pdp);
}

/* Full GATv2 backward by the chain rule:
 *   out_i = sum_j p_ij FR_j,  p = softmax_j(e_ij),  e_ij = sum_d a_d LReLU(z_ijd),
 *   z_ij = FL_i + FR_j,  FL = X W_l,  FR = X W_r.
 * The rounding of the stored projections is treated as the identity in the
 * gradient (the projections' gradients pass straight to X, W_l, W_r).
 * Outputs dX [N, F], dWl, dWr [F, H*D], da [H, D], and the intermediate
 * dFL, dFR [N, H, D] (for inspection).  dFR_j gathers p_ij dO_i (value path)
 * plus dz_ij (score path) over the destinations of j in ascending order. */
int oracle_gatv2_bwd(int64_t N, int F, int H, int D, const int32_t *indptr, const int32_t *indices,
                     const double *X, const double *Wl, const double *Wr, const double *a,
                     double slope, int store, const double *dO, double *dX, double *dWl,
                     double *dWr, double *da, double *dFL, double *dFR) {
    int HD = H * D;
    int64_t E = indptr[N];
    int64_t md = max_degree(N, indptr);
    double *FL = (double *)malloc(sizeof(double) * (size_t)(N * HD + 1));
    double *FR = (double *)malloc(sizeof(double) * (size_t)(N * HD + 1));
    double *PE = (double *)malloc(sizeof(double) * (size_t)(E * H + 1));  /* p per edge */
    double *DE = (double *)malloc(sizeof(double) * (size_t)(E * H + 1));  /* dL/de per edge */
    int32_t *t_indptr = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N + 1));
    int32_t *t_dst = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int err = 0;
    if (!FL || !FR || !PE || !DE || !t_indptr || !t_dst) err = -1;
    if (!err) {
        oracle_matmul(N, F, HD, X, Wl, FL);
        oracle_matmul(N, F, HD, X, Wr, FR);
        round_storage(N * HD, FL, store);
        round_storage(N * HD, FR, store);
#pragma omp parallel
        {
            double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
            double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
            double *de = (double *)malloc(sizeof(double) * (size_t)(md + 1));
            if (!s || !p || !de) {
#pragma omp atomic write
                err = -1;
            } else {
#pragma omp for schedule(dynamic, 64)
                for (int64_t i = 0; i < N; ++i) {
                    int64_t b = indptr[i], n = indptr[i + 1] - b;
                    for (int h = 0; h < H; ++h) {
                        double *o = dFL + ((size_t)i * H + h) * D;
                        for (int d = 0; d < D; ++d) o[d] = 0.0;
                        if (n == 0) continue;
                        gatv2_row_grad(i, h, H, D, indptr, indices, FL, FR, a, slope, dO, s, p, de);
                        const double *fl = FL + ((size_t)i * H + h) * D;
                        const double *ah = a + (size_t)h * D;
                        for (int64_t t = 0; t < n; ++t) {
                            PE[(b + t) * H + h] = p[t];
                            DE[(b + t) * H + h] = de[t];
                            const double *fr = FR + ((size_t)indices[b + t] * H + h) * D;
                            /* dz = de * a * LReLU'(z) flows to FL_i */
                            for (int d = 0; d < D; ++d)
                                o[d] += de[t] * ah[d] * lrelu_grad(fl[d] + fr[d], slope);
                        }
                    }
                }
            }
            free(s);
            free(p);
            free(de);
        }
    }
    if (!err) {
        /* da[h,d] = sum over all edges (row order, then edge order) of de * LReLU(z) */
        for (int64_t x = 0; x < HD; ++x) da[x] = 0.0;
        for (int64_t i = 0; i < N; ++i) {
            for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e) {
                int64_t j = indices[e];
                for (int h = 0; h < H; ++h) {
                    const double *fl = FL + ((size_t)i * H + h) * D;
                    const double *fr = FR + ((size_t)j * H + h) * D;
                    double dee = DE[e * H + h];
                    for (int d = 0; d < D; ++d) da[h * D + d] += dee * lrelu(fl[d] + fr[d], slope);
                }
            }
        }
        /* dFR_j: value path p dO_i plus score path dz, over destinations of j */
        oracle_transpose(N, indptr, indices, t_indptr, t_dst);
#pragma omp parallel for schedule(dynamic, 64)
        for (int64_t j = 0; j < N; ++j) {
            double *o = dFR + (size_t)j * HD;
            for (int x = 0; x < HD; ++x) o[x] = 0.0;
            for (int64_t te = t_indptr[j]; te < t_indptr[j + 1]; ++te) {
                int64_t i = t_dst[te];
                /* locate the edge(s) of row i whose source is j */
                for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e) {
                    if (indices[e] != j) continue;
                    for (int h = 0; h < H; ++h) {
                        const double *fl = FL + ((size_t)i * H + h) * D;
                        const double *fr = FR + ((size_t)j * H + h) * D;
                        const double *g = dO + ((size_t)i * H + h) * D;
                        const double *ah = a + (size_t)h * D;
                        double pe = PE[e * H + h], dee = DE[e * H + h];
                        for (int d = 0; d < D; ++d)
                            o[h * D + d] += pe * g[d] + dee * ah[d] * lrelu_grad(fl[d] + fr[d], slope);
                    }
                }
                while (te + 1 < t_indptr[j + 1] && t_dst[te + 1] == i) ++te;
            }
        }
        /* dX = dFL W_l^T + dFR W_r^T */
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            for (int f = 0; f < F; ++f) {
                double acc = 0.0;
                for (int c = 0; c < HD; ++c)
                    acc += dFL[(size_t)n * HD + c] * Wl[(size_t)f * HD + c] +
                           dFR[(size_t)n * HD + c] * Wr[(size_t)f * HD + c];
                dX[(size_t)n * F + f] = acc;
            }
        }
        /* dW_l = X^T dFL, dW_r = X^T dFR */
#pragma omp parallel for schedule(static)
        for (int f = 0; f < F; ++f) {
            double *gl = dWl + (size_t)f * HD;
            double *gr = dWr + (size_t)f * HD;
            for (int c = 0; c < HD; ++c) { gl[c] = 0.0; gr[c] = 0.0; }
            for (int64_t n = 0; n < N; ++n) {
                double x = X[(size_t)n * F + f];
                for (int c = 0; c < HD; ++c) {
                    gl[c] += x * dFL[(size_t)n * HD + c];
                    gr[c] += x * dFR[(size_t)n * HD + c];
                }
            }
        }
    }
    free(FL);
    free(FR);
    free(PE);
    free(DE);
    free(t_indptr);
    free(t_dst);
    return err;
}

/* Slack of the GATv2 gradients due to LeakyReLU branches that the storage
 * precision of FL/FR leaves undecided.
 *
 * The branch of LeakyReLU'(z), z = FL_i + FR_j, is decided on the stored
 * projections.  Two correct implementations may store projections that differ
 * by a few units in the last place (they round differently accumulated
 * sums), so an element with |z| < tau_rel (|FL| + |FR|) may take either branch.
 * Flipping one such branch changes dz by de a (1 - slope), hence dFL_i and
 * dFR_j by that amount, da by de z (1 - slope), and dX, dW through the
 * projections.  This function sums the absolute values of those changes over
 * all undecided elements: any correct result lies within this slack of the
 * oracle's (plus rounding).  Outputs: sX [N, F], sWl, sWr [F, H*D], sda [H, D]. */
int oracle_gatv2_branch_slack(int64_t N, int F, int H, int D, const int32_t *indptr,
                              const int32_t *indices, const double *X, const double *Wl,
                              const double *Wr, const double *a, double slope, int store,
                              double tau_rel, const double *dO, double *sX, double *sWl,
                              double *sWr, double *sda) {
    int HD = H * D;
    int64_t md = max_degree(N, indptr);
    double *FL = (double *)malloc(sizeof(double) * (size_t)(N * HD + 1));
    double *FR = (double *)malloc(sizeof(double) * (size_t)(N * HD + 1));
    double *sFL = (double *)calloc((size_t)(N * HD + 1), sizeof(double));
    double *sFR = (double *)calloc((size_t)(N * HD + 1), sizeof(double));
    double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *de = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    int err = (!FL || !FR || !sFL || !sFR || !s || !p || !de) ? -1 : 0;
    if (!err) {
        oracle_matmul(N, F, HD, X, Wl, FL);
        oracle_matmul(N, F, HD, X, Wr, FR);
        round_storage(N * HD, FL, store);
        round_storage(N * HD, FR, store);
        for (int64_t x = 0; x < HD; ++x) sda[x] = 0.0;
        for (int64_t i = 0; i < N; ++i) {
            int64_t b = indptr[i], n = indptr[i + 1] - b;
            for (int h = 0; h < H; ++h) {
                if (n == 0) continue;
                gatv2_row_grad(i, h, H, D, indptr, indices, FL, FR, a, slope, dO, s, p, de);
                const double *fl = FL + ((size_t)i * H + h) * D;
                for (int64_t t = 0; t < n; ++t) {
                    int64_t j = indices[b + t];
                    const double *fr = FR + ((size_t)j * H + h) * D;
                    for (int d = 0; d < D; ++d) {
                        double z = fl[d] + fr[d];
                        /* open band: z exactly 0 is decided alike on equal inputs */
                        if (!(fabs(z) < tau_rel * (fabs(fl[d]) + fabs(fr[d])))) continue;
                        double v = fabs(de[t] * a[h * D + d]) * (1.0 - slope);
                        sFL[(size_t)i * HD + h * D + d] += v;
                        sFR[(size_t)j * HD + h * D + d] += v;
                        sda[h * D + d] += fabs(de[t] * z) * (1.0 - slope);
                    }
                }
            }
        }
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; ++n)
            for (int f = 0; f < F; ++f) {
                double acc = 0.0;
                for (int c = 0; c < HD; ++c)
                    acc += sFL[(size_t)n * HD + c] * fabs(Wl[(size_t)f * HD + c]) +
                           sFR[(size_t)n * HD + c] * fabs(Wr[(size_t)f * HD + c]);
                sX[(size_t)n * F + f] = acc;
            }
#pragma omp parallel for schedule(static)
        for (int f = 0; f < F; ++f)
            for (int c = 0; c < HD; ++c) {
                double gl = 0.0, gr = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    double x = fabs(X[(size_t)n * F + f]);
                    gl += x * sFL[(size_t)n * HD + c];
                    gr += x * sFR[(size_t)n * HD + c];
                }
                sWl[(size_t)f * HD + c] = gl;
                sWr[(size_t)f * HD + c] = gr;
            }
    }
    free(FL); free(FR); free(sFL); free(sFR); free(s); free(p); free(de);
    return err;
}

/* ------------------------------------------------------------------------ */
/* Min / max neighbourhood aggregation                                       */
/* ------------------------------------------------------------------------ */

/* The degree-aware reduction layer of "On Efficient Scaling of GNNs via
 * IO-Aware Layers Implementations" (arXiv abstract; Yandex Research blog post,
 * "Aggregation layers" paragraph), written from its definition: for every
 * destination row i and element f of the node rows (X [N, F]), walk the row's
 * edges in CSR order; the first edge is taken, a later edge replaces it only
 * when its value is strictly greater (is_max) or strictly smaller (min).
 * out[i, f] is the extreme value, arg[i, f] the source of its first
 * occurrence; an empty row gives out = 0 and arg = -1. */
int oracle_agg_fwd(int64_t N, const int32_t *indptr, const int32_t *indices, int F, int is_max,
                   const double *X, double *out, int32_t *arg) {
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < N; ++i) {
        for (int f = 0; f < F; ++f) {
            double best = 0.0;
            int32_t who = -1;
            for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e) {
                int32_t j = indices[e];
                double v = X[(size_t)j * F + f];
                if (who < 0 || (is_max ? v > best : v < best)) {
                    best = v;
                    who = j;
                }
            }
            out[(size_t)i * F + f] = who < 0 ? 0.0 : best;
            arg[(size_t)i * F + f] = who;
        }
    }
    return 0;
}

/* Backward of the aggregation: dX[j, f] = sum of dO[i, f] over the rows i
 * with arg[i, f] = j, rows taken in ascending order. */
int oracle_agg_bwd(int64_t N, int F, const int32_t *arg, const double *dO, double *dX) {
    for (int64_t x = 0; x < N * F; ++x) dX[x] = 0.0;
    for (int64_t i = 0; i < N; ++i)
        for (int f = 0; f < F; ++f) {
            int32_t j = arg[(size_t)i * F + f];
            if (j >= 0) dX[(size_t)j * F + f] += dO[(size_t)i * F + f];
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Graph reordering                                                          */
/* ------------------------------------------------------------------------ */

static const int32_t *g_sort_deg;   /* key of the comparator below (single-threaded use) */

static int cmp_deg_id(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    if (g_sort_deg[x] != g_sort_deg[y]) return g_sort_deg[x] < g_sort_deg[y] ? -1 : 1;
    return x < y ? -1 : (x > y ? 1 : 0);
}

/* Reverse Cuthill-McKee, the queue-based algorithm as it is usually stated:
 * degree(v) = row degree + transposed degree (CSR entries, self-loops and
 * duplicates included); the next start is the unvisited node of least
 * degree (least id on ties); a dequeued node appends its unvisited
 * neighbours over both edge directions (each once), in order of ascending
 * degree, then id; the final order is reversed: perm[v] = new id of v.  The
 * graph reordering the IO-aware layers abstract studies names no ordering;
 * this is the classic bandwidth-reducing one. */
int oracle_rcm(int64_t N, const int32_t *indptr, const int32_t *indices, int32_t *perm) {
    int64_t E = indptr[N];
    int32_t *deg = (int32_t *)calloc((size_t)(N + 1), sizeof(int32_t));
    int32_t *t_indptr = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N + 1));
    int32_t *t_dst = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int32_t *sorted = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N + 1));
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N + 1));
    char *visited = (char *)calloc((size_t)(N + 1), 1);
    int err = (!deg || !t_indptr || !t_dst || !sorted || !order || !visited) ? -1 : 0;
    if (!err) {
        oracle_transpose(N, indptr, indices, t_indptr, t_dst);
        for (int64_t v = 0; v < N; ++v)
            deg[v] = (indptr[v + 1] - indptr[v]) + (t_indptr[v + 1] - t_indptr[v]);
        for (int64_t v = 0; v < N; ++v) sorted[v] = (int32_t)v;
        g_sort_deg = deg;
        qsort(sorted, (size_t)N, sizeof(int32_t), cmp_deg_id);
        int64_t head = 0, tail = 0, next_start = 0;
        while (tail < N) {
            while (visited[sorted[next_start]]) ++next_start;
            int32_t s = sorted[next_start];
            visited[s] = 1;
            order[tail++] = s;
            while (head < tail) {
                int32_t u = order[head++];
                int64_t first = tail;
                for (int64_t e = indptr[u]; e < indptr[u + 1]; ++e) {
                    int32_t w = indices[e];
                    if (!visited[w]) { visited[w] = 1; order[tail++] = w; }
                }
                for (int64_t e = t_indptr[u]; e < t_indptr[u + 1]; ++e) {
                    int32_t w = t_dst[e];
                    if (!visited[w]) { visited[w] = 1; order[tail++] = w; }
                }
                qsort(order + first, (size_t)(tail - first), sizeof(int32_t), cmp_deg_id);
            }
        }
        for (int64_t p = 0; p < N; ++p) perm[order[p]] = (int32_t)(N - 1 - p);
    }
    free(deg); free(t_indptr); free(t_dst); free(sorted); free(order); free(visited);
    return err;
}

/* ------------------------------------------------------------------------ */
/* Rounding bound of the fp32 GATv2 backward                                 */
/* ------------------------------------------------------------------------ */

/* Rounding factor of a sum of n fp32 terms: |computed - exact| <= gam(n)
 * times the sum of the terms' magnitudes.  The deterministic factor is
 * n u / (1 - n u) (u = 2^-24), reached only when every rounding error has
 * the same sign; rounding errors of independent operations behave as
 * independent zero-mean variables, and the probabilistic analysis of Higham
 * and Mary ("A New Approach to Probabilistic Rounding Error Analysis", SIAM
 * J. Sci. Comput. 41, 2019) bounds the sum by lambda sqrt(n) u with
 * probability at least 1 - 2 exp(-lambda^2 / 2) per sum.  lambda = 6 (failure
 * probability below 3e-8 per sum); the smaller of the two factors is used. */
static double gam(double n) {
    const double u = 1.0 / 16777216.0, lambda = 6.0;
    double det = n * u / (1.0 - n * u), prob = lambda * sqrt(n > 1.0 ? n : 1.0) * u;
    return det < prob ? det : prob;
}

/* First-order bound on |fp32 result - exact result| of every GATv2 gradient
 * (dX, dW_l, dW_r, da), for float storage of the projections (store = 1),
 * derived for the arithmetic the layer performs in fp32:
 *   - projections by fp32 dot products of F terms (|dFL| <= gamma_F sum |x w|
 *     plus their storage rounding);
 *   - per edge: z = FL_i + FR_j, e = sum_d a_d LReLU(z_d) (D terms), the
 *     weight recomputed from the forward's lse as 2^(e log2 e - lse log2 e)
 *     (relative error <= |de| + u (2|e| + 2|lse|) + 4u, the last for the
 *     exponential) and normalised by the row sum Z (deg terms), and
 *     dp = dOut_i . FR_j (D terms);
 *   - row sums kept as sum p dp x - Delta sum p x (the destination pass),
 *     whose rounding is gamma_(deg+2) times the sums of |p dp x| and
 *     |Delta p x|, not of |de x|;
 *   - the source pass's direct sums of p dOut_i + de a LReLU'(z) over each
 *     source's destinations; da summed over all rows (gamma_N); dX over 2 H D
 *     products and dW over N nodes.
 * Every sum of n terms is bounded by gam(n) times the sum of the magnitudes
 * of its terms (any summation order; gam is the probabilistic factor above);
 * errors carried in are propagated to first order and add up worst-case.  LeakyReLU branches decided differently by the two sides are not
 * covered here (oracle_gatv2_branch_slack bounds them).  Outputs: bX [N, F],
 * bWl, bWr [F, H*D], bda [H, D]. */
int oracle_gatv2_bwd_bound(int64_t N, int F, int H, int D, const int32_t *indptr,
                           const int32_t *indices, const double *X, const double *Wl,
                           const double *Wr, const double *a, double slope, const double *dO,
                           double *bX, double *bWl, double *bWr, double *bda) {
    const double u = 1.0 / 16777216.0;
    int HD = H * D;
    int64_t E = indptr[N];
    int64_t md = max_degree(N, indptr);
    double *FL = (double *)malloc(sizeof(double) * (size_t)(N * HD + 1));
    double *FR = (double *)malloc(sizeof(double) * (size_t)(N * HD + 1));
    double *bFL = (double *)malloc(sizeof(double) * (size_t)(N * HD + 1));
    double *bFR = (double *)malloc(sizeof(double) * (size_t)(N * HD + 1));
    double *dFL = (double *)calloc((size_t)(N * HD + 1), sizeof(double));   /* |exact dFL| */
    double *dFR = (double *)calloc((size_t)(N * HD + 1), sizeof(double));   /* |exact dFR| */
    double *eFL = (double *)calloc((size_t)(N * HD + 1), sizeof(double));   /* bound on dFL */
    double *eFR = (double *)calloc((size_t)(N * HD + 1), sizeof(double));   /* bound on dFR */
    double *mFR = (double *)calloc((size_t)(N * HD + 1), sizeof(double));   /* sum of |terms| of dFR */
    double *lse = (double *)malloc(sizeof(double) * (size_t)(N * H + 1));
    double *delta = (double *)malloc(sizeof(double) * (size_t)(N * H + 1));
    double *bdelta = (double *)malloc(sizeof(double) * (size_t)(N * H + 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *rho = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *bdp = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *rowda = (double *)calloc((size_t)HD + 1, sizeof(double));      /* sum over rows of |row da| */
    int err = (!FL || !FR || !bFL || !bFR || !dFL || !dFR || !eFL || !eFR || !mFR || !lse ||
               !delta || !bdelta || !s || !p || !rho || !dp || !bdp || !rowda) ? -1 : 0;
    if (!err) {
        oracle_matmul(N, F, HD, X, Wl, FL);
        oracle_matmul(N, F, HD, X, Wr, FR);
        for (int64_t n = 0; n < N; ++n)
            for (int c = 0; c < HD; ++c) {
                double ml = 0.0, mr = 0.0;
                for (int f = 0; f < F; ++f) {
                    ml += fabs(X[(size_t)n * F + f] * Wl[(size_t)f * HD + c]);
                    mr += fabs(X[(size_t)n * F + f] * Wr[(size_t)f * HD + c]);
                }
                /* fp32 accumulation of F products, plus the storage rounding of both sides */
                bFL[(size_t)n * HD + c] = gam(F) * ml + 2.0 * u * fabs(FL[(size_t)n * HD + c]);
                bFR[(size_t)n * HD + c] = gam(F) * mr + 2.0 * u * fabs(FR[(size_t)n * HD + c]);
            }
        round_storage(N * HD, FL, 1);
        round_storage(N * HD, FR, 1);
        for (int x = 0; x < HD; ++x) bda[x] = 0.0;
        /* destination rows: dFL, Delta, da */
        for (int64_t i = 0; i < N; ++i) {
            int64_t b = indptr[i], n = indptr[i + 1] - b;
            for (int h = 0; h < H; ++h) {
                if (n == 0) { lse[i * H + h] = 0.0; delta[i * H + h] = 0.0; bdelta[i * H + h] = 0.0; continue; }
                const double *fl = FL + ((size_t)i * H + h) * D;
                const double *bfl = bFL + ((size_t)i * H + h) * D;
                const double *ah = a + (size_t)h * D;
                const double *g = dO + ((size_t)i * H + h) * D;
                double mx = -INFINITY;
                for (int64_t t = 0; t < n; ++t) {
                    const double *fr = FR + ((size_t)indices[b + t] * H + h) * D;
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d) acc += ah[d] * lrelu(fl[d] + fr[d], slope);
                    s[t] = acc;
                    if (acc > mx) mx = acc;
                }
                double Z = 0.0;
                for (int64_t t = 0; t < n; ++t) Z += exp(s[t] - mx);
                double L = mx + log(Z);
                lse[i * H + h] = L;
                double rmax = 0.0, C = 0.0, mC = 0.0, bC = 0.0;
                for (int64_t t = 0; t < n; ++t) {
                    int64_t j = indices[b + t];
                    const double *fr = FR + ((size_t)j * H + h) * D;
                    const double *bfr = bFR + ((size_t)j * H + h) * D;
                    double be = 0.0, me = 0.0, dpv = 0.0, mdp = 0.0, bd = 0.0;
                    for (int d = 0; d < D; ++d) {
                        double z = fl[d] + fr[d], lz = lrelu(z, slope);
                        double bz = bfl[d] + bfr[d] + u * fabs(z);
                        be += fabs(ah[d]) * (bz + u * fabs(lz));
                        me += fabs(ah[d] * lz);
                        dpv += g[d] * fr[d];
                        mdp += fabs(g[d] * fr[d]);
                        bd += fabs(g[d]) * bfr[d];
                    }
                    be += gam(D) * me;
                    p[t] = exp(s[t] - L);
                    rho[t] = be + u * (2.0 * fabs(s[t]) + 2.0 * fabs(L)) + 4.0 * u;
                    if (rho[t] > rmax) rmax = rho[t];
                    dp[t] = dpv;
                    bdp[t] = bd + gam(D) * mdp;
                    C += p[t] * dpv;
                    mC += p[t] * fabs(dpv);
                }
                /* normalisation by Z: every weight also carries Z's relative error */
                for (int64_t t = 0; t < n; ++t) rho[t] += rmax + gam((double)n) + u;
                for (int64_t t = 0; t < n; ++t) bC += rho[t] * p[t] * fabs(dp[t]) + p[t] * bdp[t];
                bC += gam((double)n) * mC;
                delta[i * H + h] = C;
                bdelta[i * H + h] = bC;
                /* dFL and da of this row from the decomposed sums */
                for (int d = 0; d < D; ++d) {
                    double eA = 0.0, magA = 0.0, magB = 0.0, ex = 0.0, gda = 0.0, ega = 0.0, mga = 0.0, mgb = 0.0;
                    for (int64_t t = 0; t < n; ++t) {
                        int64_t j = indices[b + t];
                        double fr = FR[((size_t)j * H + h) * D + d];
                        double z = fl[d] + fr, lp = lrelu_grad(z, slope), lz = lrelu(z, slope);
                        double bz = bfl[d] + bFR[((size_t)j * H + h) * D + d] + u * fabs(z);
                        double de = p[t] * (dp[t] - C);
                        double bde = rho[t] * p[t] * fabs(dp[t] - C) + p[t] * (bdp[t] + bC) +
                                     2.0 * u * p[t] * fabs(dp[t] - C);
                        ex += de * lp;
                        eA += bde * lp;
                        magA += p[t] * fabs(dp[t]) * lp;
                        magB += p[t] * lp;
                        gda += de * lz;
                        ega += bde * fabs(lz) + fabs(de) * bz;
                        mga += p[t] * fabs(dp[t] * lz);
                        mgb += p[t] * fabs(lz);
                    }
                    double gm = gam((double)n + 2.0);
                    double vFL = ah[d] * ex;
                    dFL[(size_t)i * HD + h * D + d] = fabs(vFL);
                    eFL[(size_t)i * HD + h * D + d] =
                        fabs(ah[d]) * (eA + gm * (magA + fabs(C) * magB)) + 2.0 * u * fabs(vFL);
                    rowda[h * D + d] += fabs(gda);
                    bda[h * D + d] += ega + gm * (mga + fabs(C) * mgb) + u * fabs(gda);
                }
            }
        }
        /* source columns: dFR = sum over destinations of p dOut_i + de a LReLU'(z) */
        for (int64_t i = 0; i < N; ++i) {
            int64_t b = indptr[i], n = indptr[i + 1] - b;
            for (int h = 0; h < H; ++h) {
                if (n == 0) continue;
                const double *fl = FL + ((size_t)i * H + h) * D;
                const double *bfl = bFL + ((size_t)i * H + h) * D;
                const double *ah = a + (size_t)h * D;
                const double *g = dO + ((size_t)i * H + h) * D;
                double L = lse[i * H + h], C = delta[i * H + h], bC = bdelta[i * H + h];
                double rmax = 0.0;
                for (int64_t t = 0; t < n; ++t) {
                    int64_t j = indices[b + t];
                    const double *fr = FR + ((size_t)j * H + h) * D;
                    const double *bfr = bFR + ((size_t)j * H + h) * D;
                    double e = 0.0, be = 0.0, me = 0.0;
                    for (int d = 0; d < D; ++d) {
                        double z = fl[d] + fr[d], lz = lrelu(z, slope);
                        e += ah[d] * lz;
                        be += fabs(ah[d]) * (bfl[d] + bfr[d] + u * fabs(z) + u * fabs(lz));
                        me += fabs(ah[d] * lz);
                    }
                    rho[t] = be + gam(D) * me + u * (2.0 * fabs(e) + 2.0 * fabs(L)) + 4.0 * u;
                    if (rho[t] > rmax) rmax = rho[t];
                    p[t] = exp(e - L);
                }
                for (int64_t t = 0; t < n; ++t) {
                    int64_t j = indices[b + t];
                    const double *fr = FR + ((size_t)j * H + h) * D;
                    const double *bfr = bFR + ((size_t)j * H + h) * D;
                    double dpv = 0.0, mdp = 0.0, bd = 0.0;
                    for (int d = 0; d < D; ++d) {
                        dpv += g[d] * fr[d];
                        mdp += fabs(g[d] * fr[d]);
                        bd += fabs(g[d]) * bfr[d];
                    }
                    double r = rho[t] + rmax + gam((double)n) + 2.0 * u;   /* lse + ln Z stored in fp32 */
                    double de = p[t] * (dpv - C);
                    double bde = r * p[t] * fabs(dpv - C) + p[t] * (bd + gam(D) * mdp + bC) +
                                 2.0 * u * p[t] * fabs(dpv - C);
                    for (int d = 0; d < D; ++d) {
                        double z = fl[d] + fr[d], lp = lrelu_grad(z, slope);
                        size_t o = (size_t)j * HD + h * D + d;
                        double term = p[t] * g[d] + de * ah[d] * lp;
                        dFR[o] += term;
                        mFR[o] += fabs(p[t] * g[d]) + fabs(de * ah[d] * lp);
                        eFR[o] += r * p[t] * fabs(g[d]) + fabs(ah[d]) * lp * bde +
                                  2.0 * u * (fabs(p[t] * g[d]) + fabs(de * ah[d]));
                    }
                }
            }
        }
        /* dFR sums over each source's destinations (t_deg terms, at most N) */
        int32_t *tdeg = (int32_t *)calloc((size_t)(N + 1), sizeof(int32_t));
        if (!tdeg) err = -1;
        else {
            for (int64_t e = 0; e < E; ++e) tdeg[indices[e]]++;
            for (int64_t j = 0; j < N; ++j)
                for (int c = 0; c < HD; ++c) {
                    size_t o = (size_t)j * HD + c;
                    eFR[o] += gam((double)tdeg[j]) * mFR[o] + u * fabs(dFR[o]);
                    dFR[o] = fabs(dFR[o]);
                }
            free(tdeg);
        }
        for (int x = 0; x < HD; ++x) bda[x] += gam((double)N) * rowda[x];
        /* dX = dFL W_l^T + dFR W_r^T (2 H D products), dW = X^T dF (N products) */
        for (int64_t n = 0; n < N; ++n)
            for (int f = 0; f < F; ++f) {
                double be = 0.0, mg = 0.0;
                for (int c = 0; c < HD; ++c) {
                    size_t o = (size_t)n * HD + c;
                    double wl = fabs(Wl[(size_t)f * HD + c]), wr = fabs(Wr[(size_t)f * HD + c]);
                    be += eFL[o] * wl + eFR[o] * wr;
                    mg += dFL[o] * wl + dFR[o] * wr;
                }
                bX[(size_t)n * F + f] = be + gam(2.0 * HD) * mg + u * mg;
            }
        for (int f = 0; f < F; ++f)
            for (int c = 0; c < HD; ++c) {
                double bl = 0.0, br = 0.0, ml = 0.0, mr = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    double x = fabs(X[(size_t)n * F + f]);
                    size_t o = (size_t)n * HD + c;
                    bl += x * eFL[o];
                    br += x * eFR[o];
                    ml += x * dFL[o];
                    mr += x * dFR[o];
                }
                bWl[(size_t)f * HD + c] = bl + gam((double)N) * ml + u * ml;
                bWr[(size_t)f * HD + c] = br + gam((double)N) * mr + u * mr;
            }
    }
    free(FL); free(FR); free(bFL); free(bFR); free(dFL); free(dFR); free(eFL); free(eFR); free(mFR);
    free(lse); free(delta); free(bdelta); free(s); free(p); free(rho); free(dp); free(bdp);
    free(rowda);
    return err;
}

/* ------------------------------------------------------------------------ */
/* GAT (the original graph attention score)                                  */
/* ------------------------------------------------------------------------ */

/* The GAT layer of the AT-GNN family named by "DF-GNN: Dynamic Fusion
 * Framework for Attention Graph Neural Networks on GPUs" (abstract), in its
 * usual per-head form: FL = X W ([N, F] x [F, H*D], stored with the rounding
 * `store`), el_i = a[h,0,:] . FL_i, er_j = a[h,1,:] . FL_j (a is [H, 2, D]:
 * the destination and source halves of the attention vector),
 * e_ij = LeakyReLU(el_i + er_j), p = softmax over the row, out_i =
 * sum_j p_ij FL_j, lse as for the other layers. */
static void gat_row(int64_t i, int h, int H, int D, const int32_t *indptr, const int32_t *indices,
                    const double *FL, const double *a, double slope, double *s) {
    const double *al = a + ((size_t)h * 2 + 0) * D, *ar = a + ((size_t)h * 2 + 1) * D;
    const double *fi = FL + ((size_t)i * H + h) * D;
    double el = 0.0;
    for (int d = 0; d < D; ++d) el += al[d] * fi[d];
    for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e) {
        const double *fj = FL + ((size_t)indices[e] * H + h) * D;
        double er = 0.0;
        for (int d = 0; d < D; ++d) er += ar[d] * fj[d];
        s[e - indptr[i]] = lrelu(el + er, slope);
    }
}

int oracle_gat_fwd(int64_t N, int F, int H, int D, const int32_t *indptr, const int32_t *indices,
                   const double *X, const double *W, const double *a, double slope, int store,
                   double *FL, double *out, double *lse) {
    int HD = H * D;
    int64_t md = max_degree(N, indptr);
    oracle_matmul(N, F, HD, X, W, FL);
    round_storage(N * HD, FL, store);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        if (!s || !p) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (int64_t i = 0; i < N; ++i) {
                int64_t b = indptr[i], n = indptr[i + 1] - b;
                for (int h = 0; h < H; ++h) {
                    gat_row(i, h, H, D, indptr, indices, FL, a, slope, s);
                    lse[i * H + h] = softmax(n, s, p);
                    double *o = out + ((size_t)i * H + h) * D;
                    for (int d = 0; d < D; ++d) o[d] = 0.0;
                    for (int64_t t = 0; t < n; ++t) {
                        const double *fj = FL + ((size_t)indices[b + t] * H + h) * D;
                        for (int d = 0; d < D; ++d) o[d] += p[t] * fj[d];
                    }
                }
            }
        }
        free(s);
        free(p);
    }
    return err;
}

/* GAT backward by the chain rule (the storage rounding of FL passes
 * gradients unchanged, as for GATv2):
 *   dp = dO_i . FL_j, Delta_i = sum p dp, de = p (dp - Delta_i),
 *   dz = de LeakyReLU'(el_i + er_j),
 *   del_i = sum_j dz (over the row), der_j = sum_i dz (over j's destinations),
 *   dFL_n = sum over edges with source n of p dO_i  +  a_l del_n  +  a_r der_n,
 *   da[h,0,:] = sum_n del_n FL_n,  da[h,1,:] = sum_n der_n FL_n,
 *   dX = dFL W^T,  dW = X^T dFL.
 * Edges are visited in CSR order; per-node sums are accumulated in that
 * order (serial).  Outputs dX [N, F], dW [F, H*D], da [H, 2, D], dFL. */
int oracle_gat_bwd(int64_t N, int F, int H, int D, const int32_t *indptr, const int32_t *indices,
                   const double *X, const double *W, const double *a, double slope, int store,
                   const double *dO, double *dX, double *dW, double *da, double *dFL) {
    int HD = H * D;
    int64_t md = max_degree(N, indptr);
    double *FL = (double *)malloc(sizeof(double) * (size_t)(N * HD + 1));
    double *del = (double *)calloc((size_t)(N * H + 1), sizeof(double));
    double *der = (double *)calloc((size_t)(N * H + 1), sizeof(double));
    double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    int err = (!FL || !del || !der || !s || !p || !dp) ? -1 : 0;
    if (!err) {
        oracle_matmul(N, F, HD, X, W, FL);
        round_storage(N * HD, FL, store);
        for (int64_t x = 0; x < N * HD; ++x) dFL[x] = 0.0;
        for (int64_t i = 0; i < N; ++i) {
            int64_t b = indptr[i], n = indptr[i + 1] - b;
            for (int h = 0; h < H; ++h) {
                if (n == 0) continue;
                gat_row(i, h, H, D, indptr, indices, FL, a, slope, s);
                softmax(n, s, p);
                const double *g = dO + ((size_t)i * H + h) * D;
                double delta = 0.0;
                for (int64_t t = 0; t < n; ++t) {
                    const double *fj = FL + ((size_t)indices[b + t] * H + h) * D;
                    double v = 0.0;
                    for (int d = 0; d < D; ++d) v += g[d] * fj[d];
                    dp[t] = v;
                    delta += p[t] * v;
                }
                /* recover the pre-activation el + er of each edge for LeakyReLU' */
                const double *al = a + ((size_t)h * 2 + 0) * D, *ar = a + ((size_t)h * 2 + 1) * D;
                const double *fi = FL + ((size_t)i * H + h) * D;
                double el = 0.0;
                for (int d = 0; d < D; ++d) el += al[d] * fi[d];
                for (int64_t t = 0; t < n; ++t) {
                    int64_t j = indices[b + t];
                    const double *fj = FL + ((size_t)j * H + h) * D;
                    double er = 0.0;
                    for (int d = 0; d < D; ++d) er += ar[d] * fj[d];
                    double de = p[t] * (dp[t] - delta);
                    double dz = de * lrelu_grad(el + er, slope);
                    del[i * H + h] += dz;
                    der[j * H + h] += dz;
                    double *dj = dFL + ((size_t)j * H + h) * D;
                    for (int d = 0; d < D; ++d) dj[d] += p[t] * g[d];
                }
            }
        }
        for (int64_t n = 0; n < N; ++n)
            for (int h = 0; h < H; ++h) {
                const double *al = a + ((size_t)h * 2 + 0) * D, *ar = a + ((size_t)h * 2 + 1) * D;
                double *dn = dFL + ((size_t)n * H + h) * D;
                for (int d = 0; d < D; ++d) dn[d] += al[d] * del[n * H + h] + ar[d] * der[n * H + h];
            }
        for (int64_t x = 0; x < 2 * HD; ++x) da[x] = 0.0;
        for (int64_t n = 0; n < N; ++n)
            for (int h = 0; h < H; ++h)
                for (int d = 0; d < D; ++d) {
                    double f = FL[((size_t)n * H + h) * D + d];
                    da[((size_t)h * 2 + 0) * D + d] += del[n * H + h] * f;
                    da[((size_t)h * 2 + 1) * D + d] += der[n * H + h] * f;
                }
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; ++n)
            for (int f = 0; f < F; ++f) {
                double acc = 0.0;
                for (int c = 0; c < HD; ++c) acc += dFL[(size_t)n * HD + c] * W[(size_t)f * HD + c];
                dX[(size_t)n * F + f] = acc;
            }
#pragma omp parallel for schedule(static)
        for (int f = 0; f < F; ++f) {
            double *gw = dW + (size_t)f * HD;
            for (int c = 0; c < HD; ++c) gw[c] = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double x = X[(size_t)n * F + f];
                for (int c = 0; c < HD; ++c) gw[c] += x * dFL[(size_t)n * HD + c];
            }
        }
    }
    free(FL); free(del); free(der); free(s); free(p); free(dp);
    return err;
}

/* GAT edge stage on given inputs: Fv [N, H, D] (the projected features),
 * el, er [N, H]: e_ij = LeakyReLU(el_i + er_j), p = softmax over the row,
 * out_i = sum_j p_ij Fv_j, lse.  Backward: dFv (the value path only:
 * dFv_j = sum over j's destinations of p dO_i), del_i = sum_j dz_ij,
 * der_j = sum_i dz_ij with dz = p (dO_i . Fv_j - Delta_i) LeakyReLU'(el_i + er_j);
 * the layer-level gradients follow by the chain rule through el = a_l . FL,
 * er = a_r . FL and FL = X W (oracle_gat_bwd). */
int oracle_gat_edge_fwd(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                        const double *Fv, const double *el, const double *er, double slope,
                        double *out, double *lse) {
    int64_t md = max_degree(N, indptr);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
        if (!s || !p) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (int64_t i = 0; i < N; ++i) {
                int64_t b = indptr[i], n = indptr[i + 1] - b;
                for (int h = 0; h < H; ++h) {
                    for (int64_t t = 0; t < n; ++t)
                        s[t] = lrelu(el[i * H + h] + er[(int64_t)indices[b + t] * H + h], slope);
                    lse[i * H + h] = softmax(n, s, p);
                    double *o = out + ((size_t)i * H + h) * D;
                    for (int d = 0; d < D; ++d) o[d] = 0.0;
                    for (int64_t t = 0; t < n; ++t) {
                        const double *v = Fv + ((size_t)indices[b + t] * H + h) * D;
                        for (int d = 0; d < D; ++d) o[d] += p[t] * v[d];
                    }
                }
            }
        }
        free(s);
        free(p);
    }
    return err;
}

int oracle_gat_edge_bwd(int64_t N, const int32_t *indptr, const int32_t *indices, int H, int D,
                        const double *Fv, const double *el, const double *er, double slope,
                        const double *dO, double *dFv, double *del, double *der) {
    int64_t md = max_degree(N, indptr);
    double *s = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(md + 1));
    if (!s || !p || !dp) { free(s); free(p); free(dp); return -1; }
    for (int64_t x = 0; x < N * H * D; ++x) dFv[x] = 0.0;
    for (int64_t x = 0; x < N * H; ++x) { del[x] = 0.0; der[x] = 0.0; }
    for (int64_t i = 0; i < N; ++i) {
        int64_t b = indptr[i], n = indptr[i + 1] - b;
        for (int h = 0; h < H; ++h) {
            if (n == 0) continue;
            for (int64_t t = 0; t < n; ++t)
                s[t] = lrelu(el[i * H + h] + er[(int64_t)indices[b + t] * H + h], slope);
            softmax(n, s, p);
            const double *g = dO + ((size_t)i * H + h) * D;
            double delta = 0.0;
            for (int64_t t = 0; t < n; ++t) {
                const double *v = Fv + ((size_t)indices[b + t] * H + h) * D;
                double x = 0.0;
                for (int d = 0; d < D; ++d) x += g[d] * v[d];
                dp[t] = x;
                delta += p[t] * x;
            }
            for (int64_t t = 0; t < n; ++t) {
                int64_t j = indices[b + t];
                double dz = p[t] * (dp[t] - delta) * lrelu_grad(el[i * H + h] + er[j * H + h], slope);
                del[i * H + h] += dz;
                der[j * H + h] += dz;
                double *dj = dFv + ((size_t)j * H + h) * D;
                for (int d = 0; d < D; ++d) dj[d] += p[t] * g[d];
            }
        }
    }
    free(s); free(p); free(dp);
    return 0;
}
