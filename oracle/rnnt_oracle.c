/*
 * rnnt_oracle.c -- plain float64 CPU oracle for the RNN-T (transducer) loss
 * and its gradient on the compact 2D logit layout.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or constant with the CUDA path.
 *
 * What it computes (sources are the four pages the project is specified by):
 *   - rnnt-loss-ascend README ("optimized_transducer"), sections
 *     "参数说明" (parameters), "约束说明" (constraints), "核心梯度融合公式"
 *     (the fused-gradient formula) and "精度保证" (alpha/beta loss check):
 *     logits of one sample occupy T*(U+1) consecutive rows of a (rows, V)
 *     matrix; blank in [-V, V-1] with negatives counted from the end;
 *     clamp <= 0 disables gradient clipping; fused_log_softmax selects
 *     whether rows are raw logits (softmax applied here) or log-probs.
 *   - ESPnet GPURNNT docs (cost_and_grad / score_forward): the loss is the
 *     negative log-likelihood given by the forward variable, the gradient is
 *     taken with respect to the activation tensor.
 *   - warp-transducer blog, section 5.2: targets must not contain blank.
 *
 * Readings of points the pages leave open (each restated in the tests):
 *   - FastEmit (the fastemit_lambda argument of the GPURNNT docs and of
 *     compute_multiblank_grad_kernel, after the FastEmit paper they cite):
 *     the gradient with respect to every label-emission log-probability is
 *     scaled by (1 + lambda); blank terms and the reported loss are not
 *     changed;
 *   - rows of one sample are ordered (t, u) with u fastest;
 *   - target_lengths may be 0 (lattice width U+1 >= 1);
 *   - the terminal step is the blank emitted at (T-1, U);
 *   - clamp is applied to the per-sample gradient before the reduction scale
 *     (1/B for "mean"), which is passed in as `scale`.
 *
 * Everything is the textbook definition written out with plain loops in
 * double precision: log-softmax per node, the forward (alpha) and backward
 * (beta) recursions over the (t, u) lattice, the arc posteriors, and the
 * chain rule through log-softmax.  No blocking, no reordering, no fusion.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#else
static inline int omp_in_parallel(void) { return 0; }
#endif

#define ORACLE_F32 0
#define ORACLE_F16 1
#define ORACLE_F64 2

#define ORACLE_RED_NONE 0
#define ORACLE_RED_SUM 1
#define ORACLE_RED_MEAN 2

/* IEEE binary16 -> double, exact. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);
    return sign ? -v : v;
}

static double element(const void *x, int dtype, int64_t i)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)x)[i];
    if (dtype == ORACLE_F64)
        return ((const double *)x)[i];
    return half_bits_to_double(((const uint16_t *)x)[i]);
}

/* log(exp(a) + exp(b)) */
static double log_add(double a, double b)
{
    if (a == -INFINITY)
        return b;
    if (b == -INFINITY)
        return a;
    double m = a > b ? a : b;
    return m + log1p(exp(-fabs(a - b)));
}

/* Log-probabilities of the V outputs at one lattice node (one row). */
static void node_logprobs(const void *x, int dtype, int64_t row, int V, int fused, double *lp)
{
    for (int k = 0; k < V; ++k)
        lp[k] = element(x, dtype, row * (int64_t)V + k);
    if (!fused)
        return;
    double m = -INFINITY;
    for (int k = 0; k < V; ++k)
        if (lp[k] > m)
            m = lp[k];
    double s = 0.0;
    for (int k = 0; k < V; ++k)
        s += exp(lp[k] - m);
    double lse = m + log(s);
    for (int k = 0; k < V; ++k)
        lp[k] -= lse;
}

int rnnt_oracle_normalize_blank(int blank, int V)
{
    return blank < 0 ? blank + V : blank;
}

/* Labels y[0..U) must be output indices other than blank (warp-transducer
 * blog 4.4 / 5.2: a target equal to blank, or outside the vocabulary, is an
 * invalid input).  Returns 0 when every label is valid, -1 otherwise. */
static int labels_valid(const int32_t *y, int U, int V, int blank)
{
    for (int u = 0; u < U; ++u)
        if (y[u] < 0 || y[u] >= V || y[u] == blank)
            return -1;
    return 0;
}

/* Exclusive prefix sum of T_b*(U_b+1): first row of each sample. off has B+1 entries. */
void rnnt_oracle_offsets(int B, const int32_t *T, const int32_t *U, int64_t *off)
{
    off[0] = 0;
    for (int b = 0; b < B; ++b)
        off[b + 1] = off[b] + (int64_t)T[b] * (int64_t)(U[b] + 1);
}

/*
 * One sample: x points at its first row (T*(U+1) rows of V values), y at its
 * U labels.  Outputs (all T*(U+1), row order t*(U+1)+u):
 *   lpb[r]   log P(blank | t,u)
 *   lpy[r]   log P(y_{u+1} | t,u) for u < U, -inf at u = U
 *   alpha[r] log forward variable, alpha(0,0) = 0
 *   beta[r]  log backward variable, beta(T-1,U) = lpb(T-1,U)
 *   losses[0] = -(alpha(T-1,U) + lpb(T-1,U)),  losses[1] = -beta(0,0)
 * Returns 0, or -1 on a bad argument.
 */
int rnnt_oracle_forward(const void *x, int dtype, int V, int T, int U, const int32_t *y, int blank,
                        int fused, double *lpb, double *lpy, double *alpha, double *beta,
                        double *losses)
{
    if (T < 1 || U < 0 || V < 1)
        return -1;
    blank = rnnt_oracle_normalize_blank(blank, V);
    if (blank < 0 || blank >= V || labels_valid(y, U, V, blank) != 0)
        return -1;
    const int W = U + 1;
    double *lp = (double *)malloc(sizeof(double) * (size_t)V);
    if (!lp)
        return -1;
    for (int t = 0; t < T; ++t) {
        for (int u = 0; u <= U; ++u) {
            int64_t r = (int64_t)t * W + u;
            node_logprobs(x, dtype, r, V, fused, lp);
            lpb[r] = lp[blank];
            lpy[r] = (u < U) ? lp[y[u]] : -INFINITY;
        }
    }
    free(lp);

    for (int t = 0; t < T; ++t) {
        for (int u = 0; u <= U; ++u) {
            int64_t r = (int64_t)t * W + u;
            if (t == 0 && u == 0) {
                alpha[r] = 0.0;
                continue;
            }
            double from_blank = (t > 0) ? alpha[r - W] + lpb[r - W] : -INFINITY;
            double from_label = (u > 0) ? alpha[r - 1] + lpy[r - 1] : -INFINITY;
            alpha[r] = log_add(from_blank, from_label);
        }
    }

    for (int t = T - 1; t >= 0; --t) {
        for (int u = U; u >= 0; --u) {
            int64_t r = (int64_t)t * W + u;
            if (t == T - 1 && u == U) {
                beta[r] = lpb[r];
                continue;
            }
            double via_blank = (t < T - 1) ? beta[r + W] + lpb[r] : -INFINITY;
            double via_label = (u < U) ? beta[r + 1] + lpy[r] : -INFINITY;
            beta[r] = log_add(via_blank, via_label);
        }
    }

    int64_t last = (int64_t)(T - 1) * W + U;
    losses[0] = -(alpha[last] + lpb[last]);
    losses[1] = -beta[0];
    return 0;
}

/*
 * Gradient rows [r0, r1) of one sample, written to grad ((r1-r0) x V, double).
 * Uses the forward() outputs.  Per node (t,u):
 *   dL/dlp(blank) = -exp(alpha + lpb + beta(after blank) - ll)
 *   dL/dlp(y_u+1) = -(1 + lambda) * exp(alpha + lpy + beta(t,u+1) - ll)   (u < U)
 * where ll = alpha(T-1,U) + lpb(T-1,U), beta after the terminal blank is
 * log 1 = 0, a blank from t = T-1 with u < U leaves the lattice (-inf), and
 * lambda is the FastEmit weight (0 for the plain transducer loss).
 * With fused log-softmax the chain rule through lp = h - logsumexp(h) gives
 *   dL/dh_k = dL/dlp_k - p_k * sum_j dL/dlp_j.
 * Then clamp (if clamp > 0) and multiply by scale.
 */
int rnnt_oracle_grad(const void *x, int dtype, int V, int T, int U, const int32_t *y, int blank,
                     int fused, const double *lpb, const double *lpy, const double *alpha,
                     const double *beta, double clamp, double scale, double fastemit_lambda,
                     int64_t r0, int64_t r1, double *grad)
{
    if (T < 1 || U < 0 || V < 1)
        return -1;
    blank = rnnt_oracle_normalize_blank(blank, V);
    if (blank < 0 || blank >= V || labels_valid(y, U, V, blank) != 0)
        return -1;
    const int W = U + 1;
    const int64_t rows = (int64_t)T * W;
    if (r0 < 0 || r1 > rows || r0 > r1)
        return -1;
    const int64_t last = rows - 1;
    const double ll = alpha[last] + lpb[last];
    int failed = 0;

#pragma omp parallel for schedule(static) if (!omp_in_parallel() && (r1 - r0) * V > 65536)
    for (int64_t r = r0; r < r1; ++r) {
        double *g = grad + (r - r0) * (int64_t)V;
        int t = (int)(r / W), u = (int)(r % W);
        double beta_after_blank;
        if (t < T - 1)
            beta_after_blank = beta[r + W];
        else if (u == U)
            beta_after_blank = 0.0;
        else
            beta_after_blank = -INFINITY;
        double post_blank = exp(alpha[r] + lpb[r] + beta_after_blank - ll);
        double post_label = (u < U) ? exp(alpha[r] + lpy[r] + beta[r + 1] - ll) : 0.0;

        for (int k = 0; k < V; ++k)
            g[k] = 0.0;
        g[blank] -= post_blank;
        if (u < U)
            g[y[u]] -= (1.0 + fastemit_lambda) * post_label;

        if (fused) {
            double *lp = (double *)malloc(sizeof(double) * (size_t)V);
            if (!lp) {
                failed = 1;
                continue;
            }
            node_logprobs(x, dtype, r, V, 1, lp);
            double s = 0.0;
            for (int k = 0; k < V; ++k)
                s += g[k];
            for (int k = 0; k < V; ++k)
                g[k] -= exp(lp[k]) * s;
            free(lp);
        }
        for (int k = 0; k < V; ++k) {
            double v = g[k];
            if (clamp > 0.0)
                v = v < -clamp ? -clamp : (v > clamp ? clamp : v);
            g[k] = v * scale;
        }
    }
    return failed ? -1 : 0;
}

/*
 * Whole batch, samples processed in parallel (OpenMP).  logits is the
 * compact (rows, V) matrix, targets is (B, S) row-major.  Writes per-sample
 * losses (from alpha), losses_beta (from beta), the reduced loss (sum, or
 * mean over B; "none" reports the sum) and, if grad is not NULL, the full
 * (rows, V) gradient in double.  Returns 0, or -1 on a bad argument or
 * inconsistent lengths.
 */
int rnnt_oracle_batch(const void *logits, int dtype, int64_t rows, int V, const int32_t *targets,
                      int S, const int32_t *T, const int32_t *U, int B, int blank, double clamp,
                      int fused, int reduction, double fastemit_lambda, double *losses,
                      double *losses_beta, double *reduced, double *grad)
{
    if (B < 1 || V < 1)
        return -1;
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(B + 1));
    if (!off)
        return -1;
    rnnt_oracle_offsets(B, T, U, off);
    if (off[B] != rows) {
        free(off);
        return -1;
    }
    const double scale = (reduction == ORACLE_RED_MEAN) ? 1.0 / (double)B : 1.0;
    const size_t es = (dtype == ORACLE_F32) ? 4 : (dtype == ORACLE_F64 ? 8 : 2);
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        int64_t n = (int64_t)T[b] * (U[b] + 1);
        double *buf = (double *)malloc(sizeof(double) * (size_t)n * 4);
        if (!buf) {
            failed = 1;
            continue;
        }
        double *lpb = buf, *lpy = buf + n, *al = buf + 2 * n, *be = buf + 3 * n;
        const char *xb = (const char *)logits + (size_t)off[b] * (size_t)V * es;
        double ls[2];
        if (rnnt_oracle_forward(xb, dtype, V, T[b], U[b], targets + (int64_t)b * S, blank, fused,
                                lpb, lpy, al, be, ls) != 0)
            failed = 1;
        losses[b] = ls[0];
        losses_beta[b] = ls[1];
        if (grad && rnnt_oracle_grad(xb, dtype, V, T[b], U[b], targets + (int64_t)b * S, blank,
                                     fused, lpb, lpy, al, be, clamp, scale, fastemit_lambda, 0, n,
                                     grad + off[b] * (int64_t)V) != 0)
            failed = 1;
        free(buf);
    }
    double s = 0.0;
    for (int b = 0; b < B; ++b)
        s += losses[b];
    *reduced = (reduction == ORACLE_RED_MEAN) ? s / (double)B : s;
    free(off);
    return failed ? -1 : 0;
}

int rnnt_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Multi-blank transducer (ESPnet compute_multiblank_grad_kernel docs, after
 * the multi-blank transducer paper they cite).  Besides the standard blank
 * (one frame), K big blanks: big blank i is output bb_id[i] and advances
 * bb_dur[i] >= 2 frames.  sigma >= 0 is subtracted from every log-probability
 * used by the lattice (logit under-normalisation).  Readings of what the docs
 * leave open:
 *   - a path starts at (0,0) and ends when a blank-type step reaches frame T
 *     with all U labels emitted: the standard blank from (T-1,U) or big
 *     blank i from (T-bb_dur[i], U); no step may jump past frame T, and a
 *     blank-type step reaching frame T with labels left is not a path;
 *   - the gradient follows the same chain rule as the standard loss: arc
 *     posteriors at their output index, minus p_k times their sum through
 *     log-softmax; FastEmit scales label arcs by 1 + lambda.
 * One sample, rows t*(U+1)+u of x.  losses[0] from alpha, losses[1] = -beta(0,0).
 * grad (T*(U+1) x V, may be NULL) receives the clamped, scaled gradient.
 */
int rnnt_oracle_mb_sample(const void *x, int dtype, int V, int T, int U, const int32_t *y,
                          int blank, int fused, int K, const int32_t *bb_id,
                          const int32_t *bb_dur, double sigma, double fastemit_lambda,
                          double clamp, double scale, double *losses, double *grad)
{
    if (T < 1 || U < 0 || V < 1 || K < 0 || K > 8)
        return -1;
    blank = rnnt_oracle_normalize_blank(blank, V);
    if (blank < 0 || blank >= V || labels_valid(y, U, V, blank) != 0)
        return -1;
    for (int i = 0; i < K; ++i) {
        if (bb_dur[i] < 2 || bb_id[i] < 0 || bb_id[i] >= V || bb_id[i] == blank)
            return -1;
        for (int u = 0; u < U; ++u)   /* a big blank is never a label */
            if (y[u] == bb_id[i])
                return -1;
    }
    const int W = U + 1;
    const int64_t n = (int64_t)T * W;
    /* per node: lp'(blank), lp'(label), lp'(big blank i); then alpha, beta */
    double *lpb = (double *)malloc(sizeof(double) * (size_t)n * (4 + K));
    double *lp = (double *)malloc(sizeof(double) * (size_t)V);
    if (!lpb || !lp) {
        free(lpb);
        free(lp);
        return -1;
    }
    double *lpy = lpb + n, *alpha = lpb + 2 * n, *beta = lpb + 3 * n, *lpg = lpb + 4 * n;
    for (int64_t r = 0; r < n; ++r) {
        int u = (int)(r % W);
        node_logprobs(x, dtype, r, V, fused, lp);
        lpb[r] = lp[blank] - sigma;
        lpy[r] = (u < U) ? lp[y[u]] - sigma : -INFINITY;
        for (int i = 0; i < K; ++i)
            lpg[(int64_t)i * n + r] = lp[bb_id[i]] - sigma;
    }
    for (int t = 0; t < T; ++t) {
        for (int u = 0; u <= U; ++u) {
            int64_t r = (int64_t)t * W + u;
            if (t == 0 && u == 0) {
                alpha[r] = 0.0;
                continue;
            }
            double a = (t > 0) ? alpha[r - W] + lpb[r - W] : -INFINITY;
            if (u > 0)
                a = log_add(a, alpha[r - 1] + lpy[r - 1]);
            for (int i = 0; i < K; ++i) {
                int t0 = t - bb_dur[i];
                if (t0 >= 0) {
                    int64_t r0 = (int64_t)t0 * W + u;
                    a = log_add(a, alpha[r0] + lpg[(int64_t)i * n + r0]);
                }
            }
            alpha[r] = a;
        }
    }
    /* beta(t,u): log-probability of finishing from (t,u); frame T is the end. */
    for (int t = T - 1; t >= 0; --t) {
        for (int u = U; u >= 0; --u) {
            int64_t r = (int64_t)t * W + u;
            double b = -INFINITY;
            if (t + 1 < T)
                b = beta[r + W] + lpb[r];
            else if (u == U)
                b = lpb[r];
            if (u < U)
                b = log_add(b, beta[r + 1] + lpy[r]);
            for (int i = 0; i < K; ++i) {
                int t1 = t + bb_dur[i];
                double g = lpg[(int64_t)i * n + r];
                if (t1 < T)
                    b = log_add(b, beta[(int64_t)t1 * W + u] + g);
                else if (t1 == T && u == U)
                    b = log_add(b, g);
            }
            beta[r] = b;
        }
    }
    double ll = alpha[n - 1] + lpb[n - 1];
    for (int i = 0; i < K; ++i) {
        int t0 = T - bb_dur[i];
        if (t0 >= 0) {
            int64_t r0 = (int64_t)t0 * W + U;
            ll = log_add(ll, alpha[r0] + lpg[(int64_t)i * n + r0]);
        }
    }
    losses[0] = -ll;
    losses[1] = -beta[0];

    if (grad) {
        for (int64_t r = 0; r < n; ++r) {
            int t = (int)(r / W), u = (int)(r % W);
            double *g = grad + r * (int64_t)V;
            for (int k = 0; k < V; ++k)
                g[k] = 0.0;
            double bn = (t + 1 < T) ? beta[r + W] : (u == U ? 0.0 : -INFINITY);
            g[blank] -= exp(alpha[r] + lpb[r] + bn - ll);
            if (u < U)
                g[y[u]] -= (1.0 + fastemit_lambda) * exp(alpha[r] + lpy[r] + beta[r + 1] - ll);
            for (int i = 0; i < K; ++i) {
                int t1 = t + bb_dur[i];
                double bb = (t1 < T) ? beta[(int64_t)t1 * W + u]
                                     : ((t1 == T && u == U) ? 0.0 : -INFINITY);
                g[bb_id[i]] -= exp(alpha[r] + lpg[(int64_t)i * n + r] + bb - ll);
            }
            if (fused) {
                node_logprobs(x, dtype, r, V, 1, lp);
                double s = 0.0;
                for (int k = 0; k < V; ++k)
                    s += g[k];
                for (int k = 0; k < V; ++k)
                    g[k] -= exp(lp[k]) * s;
            }
            for (int k = 0; k < V; ++k) {
                double v = g[k];
                if (clamp > 0.0)
                    v = v < -clamp ? -clamp : (v > clamp ? clamp : v);
                g[k] = v * scale;
            }
        }
    }
    free(lpb);
    free(lp);
    return 0;
}
