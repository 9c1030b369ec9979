/*
 * attn_oracle.c -- float64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the package's smoke check and the CPU-baseline
 * leg of the benchmark load this file's shared object; the GPU library never links,
 * loads or calls it, and this file includes nothing from the GPU library.
 *
 * What it computes is the plain definition of the operator, written out row by row with
 * the row of logits materialised (no tiling, no online state):
 *
 *   "How Does FlashAttention Preserve Global Softmax Across Tiles?", section 1 (the
 *   operator: logits = scale * <q_i, k_j> + b_ij over the visible set J_i; weights sum to
 *   one on a nonempty row, masked positions weigh zero; scale independent of tiling),
 *   section 6 (global positions; rectangular causal masks align the two sequences' ends,
 *   "bottom-right": key j is visible to query i iff j <= i + (N_k - N_q); an empty row
 *   returns zero), section 7 (the saved per-row log-sum-exp L_i).
 *   "Reducing Memory Traffic with Output Accumulation in FlashAttention", "Computing the
 *   Value Weighted Sum First" (stable softmax subtracts the row maximum before exp;
 *   weighted sum first, one division by the exponential sum).
 *
 * Readings taken where the pages leave a step open:
 *   - bias is added after scaling and is not itself scaled;
 *   - with per-sequence key lengths kv_len[b], the causal alignment uses the sequence's
 *     own key end: j <= i + kv_len[b] - N_q;
 *   - a bias of -inf marks a position as masked; masked positions are never read for
 *     arithmetic, so any value stored there (NaN included) cannot change the result;
 *   - an empty row gives o = +0.0 and lse = -inf exactly.
 *
 * The per-key-subset state (m, l, u) and the merge of states follow the same page,
 * section 3 (a maximum, a shifted exponential sum and an unnormalised weighted value sum
 * per key subset; merging disjoint subsets puts both maxima into a common coordinate and
 * scales both l and u of each subset by exp(m_X - m)), and "Flash attention and
 * efficient attention: Visual walkthrough", Step 5.
 *
 * Inputs are float32 arrays holding the exact values the GPU path sees (bfloat16 values
 * widen to float32 without rounding); every operation here is done in float64.
 *
 * Layouts (all contiguous, row-major):
 *   q    [B, Nq, H, dk]      k [B, Nk, H, dk]      v [B, Nk, H, dv]
 *   bias [B, H, Nq, Nk] or NULL
 *   kv_lens [B] or NULL (NULL means Nk for every sequence; values are clamped to [0, Nk])
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_EXPORT __attribute__((visibility("default")))

typedef struct {
    int64_t B, H, Nq, Nk, dk, dv;
    const float *q, *k, *v, *bias;
    const int32_t *kv_lens;
    int causal;
    double scale;
} problem_t;

static int64_t key_len(const problem_t *p, int64_t b) {
    if (!p->kv_lens) return p->Nk;
    int64_t n = p->kv_lens[b];
    if (n < 0) n = 0;
    if (n > p->Nk) n = p->Nk;
    return n;
}

static double bias_at(const problem_t *p, int64_t b, int64_t h, int64_t i, int64_t j) {
    return (double)p->bias[((b * p->H + h) * p->Nq + i) * p->Nk + j];
}

/* Is key j in the visible set J_i of query row i of (b, h)? */
static int visible(const problem_t *p, int64_t b, int64_t h, int64_t i, int64_t j) {
    int64_t n = key_len(p, b);
    if (j >= n) return 0;                                 /* padding */
    if (p->causal && j > i + n - p->Nq) return 0;         /* bottom-right causal */
    if (p->bias) {                                        /* bias -inf masks */
        float bij = p->bias[((b * p->H + h) * p->Nq + i) * p->Nk + j];
        if (isinf(bij) && bij < 0) return 0;
    }
    return 1;
}

/* Logit x_ij = scale * <q_i, k_j> + b_ij, only ever evaluated for visible (i, j). */
static double logit(const problem_t *p, int64_t b, int64_t h, int64_t i, int64_t j) {
    const float *qi = p->q + ((b * p->Nq + i) * p->H + h) * p->dk;
    const float *kj = p->k + ((b * p->Nk + j) * p->H + h) * p->dk;
    double dot = 0.0;
    for (int64_t c = 0; c < p->dk; ++c) dot += (double)qi[c] * (double)kj[c];
    double x = p->scale * dot;
    if (p->bias) x += bias_at(p, b, h, i, j);
    return x;
}

static const float *value_row(const problem_t *p, int64_t b, int64_t h, int64_t j) {
    return p->v + ((b * p->Nk + j) * p->H + h) * p->dv;
}

/*
 * One row, by definition: materialise x_j for j in J_i, take m = max_j x_j,
 * w_j = exp(x_j - m), l = sum_j w_j, o = sum_j w_j v_j / l, lse = m + ln l.
 * xbuf holds Nk doubles.  Empty row: o = +0.0, lse = -inf.
 */
static void one_row(const problem_t *p, int64_t b, int64_t h, int64_t i, double *xbuf,
                    double *o, double *lse) {
    int64_t nvis = 0;
    double m = -INFINITY;
    for (int64_t j = 0; j < p->Nk; ++j) {
        if (!visible(p, b, h, i, j)) continue;
        double x = logit(p, b, h, i, j);
        xbuf[j] = x;
        if (nvis == 0 || x > m) m = x;
        ++nvis;
    }
    for (int64_t c = 0; c < p->dv; ++c) o[c] = 0.0;
    if (nvis == 0) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < p->Nk; ++j) {
        if (!visible(p, b, h, i, j)) continue;
        double w = exp(xbuf[j] - m);
        l += w;
        const float *vj = value_row(p, b, h, j);
        for (int64_t c = 0; c < p->dv; ++c) o[c] += w * (double)vj[c];
    }
    for (int64_t c = 0; c < p->dv; ++c) o[c] /= l;
    *lse = m + log(l);
}

static int check_problem(const problem_t *p) {
    if (p->B < 0 || p->H < 0 || p->Nq < 0 || p->Nk < 0 || p->dk < 1 || p->dv < 1) return -1;
    if (p->Nq > 0 && !p->q) return -1;
    if (p->Nk > 0 && (!p->k || !p->v)) return -1;
    return 0;
}

/*
 * O and lse for every row (rows == NULL) or for the listed rows.
 * A row index r is the flat index (b * H + h) * Nq + i.
 * rows == NULL: o is [B, Nq, H, dv], lse is [B, H, Nq].
 * rows != NULL: o is [n_rows, dv], lse is [n_rows], in the order listed.
 * Returns the number of threads used, or -1 on bad arguments.
 */
ORACLE_EXPORT int oracle_attn_fwd(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t dk,
                                  int64_t dv, const float *q, const float *k, const float *v,
                                  const float *bias, const int32_t *kv_lens, int causal,
                                  double scale, const int64_t *rows, int64_t n_rows,
                                  double *o, double *lse, int n_threads) {
    problem_t p = {B, H, Nq, Nk, dk, dv, q, k, v, bias, kv_lens, causal, scale};
    if (check_problem(&p)) return -1;
    int64_t total = rows ? n_rows : B * H * Nq;
    int used = 1;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
    {
#pragma omp single
        used = omp_get_num_threads();
#else
    {
#endif
        double *xbuf = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (int64_t t = 0; t < total; ++t) {
            int64_t r = rows ? rows[t] : t;
            int64_t b = r / (H * Nq), h = (r / Nq) % H, i = r % Nq;
            double *orow = rows ? o + t * dv : o + ((b * Nq + i) * H + h) * dv;
            double *lrow = rows ? lse + t : lse + r;
            one_row(&p, b, h, i, xbuf, orow, lrow);
        }
        free(xbuf);
    }
    return used;
}

/*
 * The full weight matrix P [B, H, Nq, Nk] (small inputs only): p_ij = exp(x_ij - m_i) / l_i
 * on visible positions, exactly 0 on masked ones and on every entry of an empty row.
 */
ORACLE_EXPORT int oracle_attn_probs(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t dk,
                                    int64_t dv, const float *q, const float *k, const float *v,
                                    const float *bias, const int32_t *kv_lens, int causal,
                                    double scale, double *probs) {
    problem_t p = {B, H, Nq, Nk, dk, dv, q, k, v, bias, kv_lens, causal, scale};
    if (check_problem(&p)) return -1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < Nq; ++i) {
                double *prow = probs + ((b * H + h) * Nq + i) * Nk;
                double m = -INFINITY;
                int64_t nvis = 0;
                for (int64_t j = 0; j < Nk; ++j) {
                    prow[j] = 0.0;
                    if (!visible(&p, b, h, i, j)) continue;
                    double x = logit(&p, b, h, i, j);
                    if (nvis == 0 || x > m) m = x;
                    ++nvis;
                }
                if (nvis == 0) continue;
                double l = 0.0;
                for (int64_t j = 0; j < Nk; ++j) {
                    if (!visible(&p, b, h, i, j)) continue;
                    prow[j] = exp(logit(&p, b, h, i, j) - m);
                    l += prow[j];
                }
                for (int64_t j = 0; j < Nk; ++j) prow[j] /= l;
            }
    return 0;
}

/*
 * The state (m, l, u) of one query row over the visible keys in [j0, j1):
 *   m = max x_j,  l = sum exp(x_j - m),  u = sum exp(x_j - m) v_j.
 * Rows are all (b, h, i) in order; state is [B, H, Nq, 2 + dv] laid out (m, l, u[0..dv)).
 * An empty subset gives the empty state (m = -inf, l = 0, u = 0).
 */
ORACLE_EXPORT int oracle_key_state(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t dk,
                                   int64_t dv, const float *q, const float *k, const float *v,
                                   const float *bias, const int32_t *kv_lens, int causal,
                                   double scale, int64_t j0, int64_t j1, double *state) {
    problem_t p = {B, H, Nq, Nk, dk, dv, q, k, v, bias, kv_lens, causal, scale};
    if (check_problem(&p) || j0 < 0 || j1 > Nk || j0 > j1) return -1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < Nq; ++i) {
                double *s = state + ((b * H + h) * Nq + i) * (2 + dv);
                double m = -INFINITY;
                int64_t nvis = 0;
                for (int64_t j = j0; j < j1; ++j) {
                    if (!visible(&p, b, h, i, j)) continue;
                    double x = logit(&p, b, h, i, j);
                    if (nvis == 0 || x > m) m = x;
                    ++nvis;
                }
                s[0] = m;
                s[1] = 0.0;
                for (int64_t c = 0; c < dv; ++c) s[2 + c] = 0.0;
                if (nvis == 0) continue;
                for (int64_t j = j0; j < j1; ++j) {
                    if (!visible(&p, b, h, i, j)) continue;
                    double w = exp(logit(&p, b, h, i, j) - m);
                    s[1] += w;
                    const float *vj = value_row(&p, b, h, j);
                    for (int64_t c = 0; c < dv; ++c) s[2 + c] += w * (double)vj[c];
                }
            }
    return 0;
}

/*
 * Merge n_states states per row and finalise.
 * states [n_rows, n_states, 2 + dv] as (m, l, u); empty states (l == 0) are skipped.
 *   m = max over nonempty s of m_s;  l = sum exp(m_s - m) l_s;  u = sum exp(m_s - m) u_s;
 *   o = u / l,  lse = m + ln l.   A row whose states are all empty: o = +0.0, lse = -inf.
 * o [n_rows, dv], lse [n_rows].
 */
ORACLE_EXPORT int oracle_merge_states(int64_t n_rows, int64_t n_states, int64_t dv,
                                      const double *states, double *o, double *lse) {
    if (n_rows < 0 || n_states < 0 || dv < 1) return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        const double *st = states + r * n_states * (2 + dv);
        double *orow = o + r * dv;
        double m = -INFINITY;
        int any = 0;
        for (int64_t s = 0; s < n_states; ++s) {
            const double *x = st + s * (2 + dv);
            if (!(x[1] > 0.0)) continue;
            if (!any || x[0] > m) m = x[0];
            any = 1;
        }
        for (int64_t c = 0; c < dv; ++c) orow[c] = 0.0;
        if (!any) {
            lse[r] = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (int64_t s = 0; s < n_states; ++s) {
            const double *x = st + s * (2 + dv);
            if (!(x[1] > 0.0)) continue;
            double a = exp(x[0] - m);
            l += a * x[1];
            for (int64_t c = 0; c < dv; ++c) orow[c] += a * x[2 + c];
        }
        for (int64_t c = 0; c < dv; ++c) orow[c] /= l;
        lse[r] = m + log(l);
    }
    return 0;
}

/*
 * Gradients of the loss through O, by definition ("How Does FlashAttention Preserve Global
 * Softmax Across Tiles?", section 7: with g_i the upstream gradient of row i, the softmax
 * Jacobian's row reduction is c_i = sum_j p_ij (g_i . v_j), which equals g_i . o_i; the
 * gradient with respect to the scaled logits is p_ij (g_i . v_j - c_i); the Q and K gradients
 * carry the original scale).  Written out row by row with the probability row materialised:
 *
 *   p_ij  = exp(x_ij - m_i) / l_i on visible (i, j), 0 elsewhere (as in the forward)
 *   dV_j  = sum_i p_ij g_i
 *   dP_ij = g_i . v_j,   c_i = sum_j p_ij dP_ij,   dS_ij = p_ij (dP_ij - c_i)
 *   dQ_i  = scale * sum_j dS_ij k_j,   dK_j = scale * sum_i dS_ij q_i
 *
 * Readings: the bias is fixed input (no gradient is formed for it); an empty row has a
 * constant zero output, so it passes no gradient (its p row is all zero).
 * dout [B, Nq, H, dv]; dq [B, Nq, H, dk], dk [B, Nk, H, dk], dv [B, Nk, H, dv], float64.
 * Returns the number of threads used, or -1 on bad arguments.
 */
ORACLE_EXPORT int oracle_attn_bwd(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t dk,
                                  int64_t dv, const float *q, const float *k, const float *v,
                                  const float *bias, const int32_t *kv_lens, int causal,
                                  double scale, const float *dout, double *dq, double *dkey,
                                  double *dval, int n_threads) {
    problem_t p = {B, H, Nq, Nk, dk, dv, q, k, v, bias, kv_lens, causal, scale};
    if (check_problem(&p) || (Nq > 0 && !dout)) return -1;
    memset(dq, 0, sizeof(double) * (size_t)(B * Nq * H * dk));
    memset(dkey, 0, sizeof(double) * (size_t)(B * Nk * H * dk));
    memset(dval, 0, sizeof(double) * (size_t)(B * Nk * H * dv));
    int used = 1;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
    {
#pragma omp single
        used = omp_get_num_threads();
#else
    {
#endif
        double *prow = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double *dprow = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        /* one (b, h) per iteration: its dK and dV rows are written by this thread only */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t bh = 0; bh < B * H; ++bh) {
            const int64_t b = bh / H, h = bh % H;
            for (int64_t i = 0; i < Nq; ++i) {
                /* the probability row */
                double m = -INFINITY;
                int64_t nvis = 0;
                for (int64_t j = 0; j < Nk; ++j) {
                    prow[j] = 0.0;
                    if (!visible(&p, b, h, i, j)) continue;
                    double x = logit(&p, b, h, i, j);
                    prow[j] = x;
                    if (nvis == 0 || x > m) m = x;
                    ++nvis;
                }
                if (nvis == 0) continue; /* empty row: no gradient */
                double l = 0.0;
                for (int64_t j = 0; j < Nk; ++j) {
                    if (!visible(&p, b, h, i, j)) continue;
                    prow[j] = exp(prow[j] - m);
                    l += prow[j];
                }
                for (int64_t j = 0; j < Nk; ++j) prow[j] /= l;
                /* dP_ij = g_i . v_j and the row reduction c_i */
                const float *gi = dout + ((b * Nq + i) * H + h) * dv;
                double c = 0.0;
                for (int64_t j = 0; j < Nk; ++j) {
                    dprow[j] = 0.0;
                    if (!visible(&p, b, h, i, j)) continue;
                    const float *vj = value_row(&p, b, h, j);
                    double d = 0.0;
                    for (int64_t t = 0; t < dv; ++t) d += (double)gi[t] * (double)vj[t];
                    dprow[j] = d;
                    c += prow[j] * d;
                }
                const float *qi = q + ((b * Nq + i) * H + h) * dk;
                double *dqi = dq + ((b * Nq + i) * H + h) * dk;
                for (int64_t j = 0; j < Nk; ++j) {
                    if (!visible(&p, b, h, i, j)) continue;
                    const double ds = prow[j] * (dprow[j] - c);
                    const float *kj = k + ((b * Nk + j) * H + h) * dk;
                    double *dkj = dkey + ((b * Nk + j) * H + h) * dk;
                    double *dvj = dval + ((b * Nk + j) * H + h) * dv;
                    for (int64_t t = 0; t < dv; ++t) dvj[t] += prow[j] * (double)gi[t];
                    for (int64_t t = 0; t < dk; ++t) {
                        dqi[t] += scale * ds * (double)kj[t];
                        dkj[t] += scale * ds * (double)qi[t];
                    }
                }
            }
        }
        free(prow);
        free(dprow);
    }
    return used;
}

ORACLE_EXPORT int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
