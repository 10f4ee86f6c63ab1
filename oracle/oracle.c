/*
 * fp64 CPU oracle for the three row-wise reductions: softmax forward,
 * RMSNorm forward and cross-entropy forward over a row-major M x N matrix.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the definition that the CUDA
 * library is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Source.  The QbitAI article on QuACK ("无需CUDA代码，给H100加速33%-50%",
 * ramisays.com / senqingzn.com) names the three operators in its section
 * "让内存密集型内核达到“光速”" (making memory-bound kernels reach speed of light):
 * RMSNorm, softmax and cross-entropy loss, the reductions of large-language-
 * model layers.  The article never writes the formulas down, so each function
 * below is the textbook definition that those operator names denote, written
 * out with no blocking, fusion or reordering:
 *
 *   softmax   m = max_j x_j,  y_j = exp(x_j - m) / sum_k exp(x_k - m)
 *   RMSNorm   rstd = 1 / sqrt((1/N) sum_j x_j^2 + eps),  y_j = x_j * rstd * w_j
 *   x-entropy lse = m + log sum_j exp(x_j - m),  loss = lse - x_t
 *
 * and, further down, their gradients (softmax dx; RMSNorm dx and dw;
 * cross-entropy dlogits), the textbook derivatives of the same definitions.
 *
 * All inputs arrive already widened to double (exact for fp32 and bf16 data);
 * every operation is done in double with libm's exp, log and sqrt.  Each row
 * is handled on its own, one element at a time, in index order.
 *
 * Readings where the article is silent:
 *   - RMSNorm: eps is added to the mean of squares inside the square root; the
 *     mean divides by N; the weight multiplies plainly (no 1+w, no bias);
 *     rstd = 1/sqrt(ms + eps) is the per-row scalar returned.
 *   - Cross-entropy: no reduction over rows, no ignore index, no smoothing;
 *     a target outside [0, N) gives a NaN loss for that row.
 *   - Softmax max-shift: the shift by the row maximum is part of the textbook
 *     definition used here; mathematically it changes nothing, and it keeps
 *     exp() finite for the large-magnitude rows the tests use.
 *
 * Compiled with -ffp-contract=off so that no multiply-add is fused and the
 * results are the same on x86-64 and aarch64 hosts.
 */
#include <math.h>
#include <stdint.h>

/* Softmax forward, one row after another (article section
 * "让内存密集型内核达到“光速”": softmax named as a reduction operator; section
 * "内存吞吐量": the conventional three sweeps over the row -- row maximum, sum of
 * shifted exponentials, normalisation -- which is the order taken here). */
void oracle_softmax_fwd(const double *x, double *y, int64_t M, int64_t N)
{
    for (int64_t i = 0; i < M; ++i) {
        const double *xi = x + i * N;
        double *yi = y + i * N;

        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j)
            if (xi[j] > m) m = xi[j];

        double s = 0.0;
        for (int64_t j = 0; j < N; ++j)
            s += exp(xi[j] - m);

        for (int64_t j = 0; j < N; ++j)
            yi[j] = exp(xi[j] - m) / s;
    }
}

/* RMSNorm forward (article section "让内存密集型内核达到“光速”": RMSNorm named
 * as a reduction operator; the section "内存吞吐量" benchmarks it).  rstd may be
 * NULL when the caller does not want it. */
void oracle_rmsnorm_fwd(const double *x, const double *w, double *y,
                        double *rstd, int64_t M, int64_t N, double eps)
{
    for (int64_t i = 0; i < M; ++i) {
        const double *xi = x + i * N;
        double *yi = y + i * N;

        double sum_sq = 0.0;
        for (int64_t j = 0; j < N; ++j)
            sum_sq += xi[j] * xi[j];
        double ms = sum_sq / (double)N;
        double r = 1.0 / sqrt(ms + eps);

        for (int64_t j = 0; j < N; ++j)
            yi[j] = xi[j] * r * w[j];
        if (rstd) rstd[i] = r;
    }
}

/* Cross-entropy loss forward (article section "让内存密集型内核达到“光速”":
 * cross-entropy loss named as the third reduction operator).  Per row:
 * lse = log sum_j exp(x_j) computed with the max shift, loss = lse - x_t.
 * lse may be NULL when the caller does not want it. */
void oracle_xent_fwd(const double *x, const int64_t *target, double *loss,
                     double *lse, int64_t M, int64_t N)
{
    for (int64_t i = 0; i < M; ++i) {
        const double *xi = x + i * N;

        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j)
            if (xi[j] > m) m = xi[j];

        double s = 0.0;
        for (int64_t j = 0; j < N; ++j)
            s += exp(xi[j] - m);

        double l = m + log(s);
        int64_t t = target[i];
        loss[i] = (t >= 0 && t < N) ? l - xi[t] : NAN;
        if (lse) lse[i] = l;
    }
}

/* ------------------------------------------------------------------------
 * Backward passes (gradients of the three forward operators above).  The
 * article benchmarks forward passes only; these are the textbook derivatives
 * of the same definitions, written out the same plain way.
 * ------------------------------------------------------------------------ */

/* Softmax backward: given y = softmax(x) and dy = dL/dy, per row
 *   dx_j = y_j * (dy_j - sum_k dy_k * y_k). */
void oracle_softmax_bwd(const double *y, const double *dy, double *dx, int64_t M, int64_t N)
{
    for (int64_t i = 0; i < M; ++i) {
        const double *yi = y + i * N, *gi = dy + i * N;
        double *di = dx + i * N;

        double dot = 0.0;
        for (int64_t j = 0; j < N; ++j)
            dot += gi[j] * yi[j];

        for (int64_t j = 0; j < N; ++j)
            di[j] = yi[j] * (gi[j] - dot);
    }
}

/* RMSNorm backward: given x, w, r = rstd (as returned by the forward pass) and
 * dy = dL/dy for y_j = x_j * r * w_j, per row
 *   dx_j = r * dy_j * w_j - x_j * r^3 * (1/N) sum_k dy_k * w_k * x_k,
 * and over all rows dw_j = sum_i dy_ij * x_ij * r_i.  (d r / d x_j = -r^3 x_j / N.) */
void oracle_rmsnorm_bwd(const double *x, const double *w, const double *rstd,
                        const double *dy, double *dx, double *dw, int64_t M, int64_t N)
{
    for (int64_t j = 0; j < N; ++j)
        dw[j] = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        const double *xi = x + i * N, *gi = dy + i * N;
        double *di = dx + i * N;
        double r = rstd[i];

        double dot = 0.0;
        for (int64_t j = 0; j < N; ++j)
            dot += gi[j] * w[j] * xi[j];
        double c = r * r * r * dot / (double)N;

        for (int64_t j = 0; j < N; ++j) {
            di[j] = r * gi[j] * w[j] - xi[j] * c;
            dw[j] += gi[j] * xi[j] * r;
        }
    }
}

/* Cross-entropy backward: given the logits, the targets, lse (as returned by
 * the forward pass) and dloss_i = dL/dloss_i, per row
 *   dx_j = dloss_i * (exp(x_j - lse_i) - [j == t_i]);
 * a row whose target is outside [0, N) gets NaN gradients (its loss is NaN). */
void oracle_xent_bwd(const double *x, const int64_t *target, const double *lse,
                     const double *dloss, double *dx, int64_t M, int64_t N)
{
    for (int64_t i = 0; i < M; ++i) {
        const double *xi = x + i * N;
        double *di = dx + i * N;
        int64_t t = target[i];
        int ok = (t >= 0 && t < N);

        for (int64_t j = 0; j < N; ++j) {
            double p = exp(xi[j] - lse[i]);
            di[j] = ok ? dloss[i] * (p - (j == t ? 1.0 : 0.0)) : NAN;
        }
    }
}

/* ------------------------------------------------------------------------
 * Cross-entropy variants (ignore index, z-loss, mean over rows).
 * A row is ignored when has_ignore is nonzero and t_i == ignore_index; with
 * has_ignore == 0 no row is ignored, whatever its target (no target value
 * stands for "none", so INT64_MIN is an ordinary out-of-range target).
 *   loss_i = lse_i - x_{i,t_i} + z * lse_i^2      for a row not ignored,
 *   loss_i = 0                                    for an ignored row,
 *   mean   = sum of loss_i over the rows not ignored / their number
 *            (NaN when every row is ignored: 0 / 0);
 *   dx_ij  = dloss_i * ((1 + 2 z lse_i) exp(x_ij - lse_i) - [j == t_i]),
 *            0 on ignored rows.  d(z lse^2)/dx_j = 2 z lse softmax_j.
 * A target that is neither ignored nor inside [0, N) gives NaN, as before.
 * ------------------------------------------------------------------------ */
void oracle_xent_fwd_ex(const double *x, const int64_t *target, double *loss, double *lse,
                        double *mean, int64_t M, int64_t N, int has_ignore, int64_t ignore_index,
                        double z)
{
    double total = 0.0;
    int64_t counted = 0;
    for (int64_t i = 0; i < M; ++i) {
        const double *xi = x + i * N;

        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j)
            if (xi[j] > m) m = xi[j];

        double s = 0.0;
        for (int64_t j = 0; j < N; ++j)
            s += exp(xi[j] - m);

        double l = m + log(s);
        int64_t t = target[i];
        double li;
        if (has_ignore && t == ignore_index) {
            li = 0.0;
        } else {
            li = (t >= 0 && t < N) ? l - xi[t] + z * l * l : NAN;
            total += li;
            counted += 1;
        }
        loss[i] = li;
        if (lse) lse[i] = l;
    }
    if (mean) *mean = total / (double)counted;
}

void oracle_xent_bwd_ex(const double *x, const int64_t *target, const double *lse,
                        const double *dloss, double *dx, int64_t M, int64_t N,
                        int has_ignore, int64_t ignore_index, double z)
{
    for (int64_t i = 0; i < M; ++i) {
        const double *xi = x + i * N;
        double *di = dx + i * N;
        int64_t t = target[i];

        for (int64_t j = 0; j < N; ++j) {
            if (has_ignore && t == ignore_index) {
                di[j] = 0.0;
            } else if (t >= 0 && t < N) {
                double p = exp(xi[j] - lse[i]);
                di[j] = dloss[i] * ((1.0 + 2.0 * z * lse[i]) * p - (j == t ? 1.0 : 0.0));
            } else {
                di[j] = NAN;
            }
        }
    }
}

/* ------------------------------------------------------------------------
 * LayerNorm forward (the article's claim that the same row-reduction template
 * carries over to other normalisations; LayerNorm itself is not named there).
 * Per row, with the population variance (divide by N) and eps inside the root:
 *   mean = (1/N) sum_j x_j,  var = (1/N) sum_j (x_j - mean)^2,
 *   rstd = 1 / sqrt(var + eps),  y_j = (x_j - mean) * rstd * w_j + b_j
 * b may be NULL (no bias).  mean and rstd may be NULL.
 * ------------------------------------------------------------------------ */
void oracle_layernorm_fwd(const double *x, const double *w, const double *b, double *y,
                          double *mean, double *rstd, int64_t M, int64_t N, double eps)
{
    for (int64_t i = 0; i < M; ++i) {
        const double *xi = x + i * N;
        double *yi = y + i * N;

        double sum = 0.0;
        for (int64_t j = 0; j < N; ++j)
            sum += xi[j];
        double mu = sum / (double)N;

        double sq = 0.0;
        for (int64_t j = 0; j < N; ++j)
            sq += (xi[j] - mu) * (xi[j] - mu);
        double var = sq / (double)N;
        double r = 1.0 / sqrt(var + eps);

        for (int64_t j = 0; j < N; ++j)
            yi[j] = (xi[j] - mu) * r * w[j] + (b ? b[j] : 0.0);
        if (mean) mean[i] = mu;
        if (rstd) rstd[i] = r;
    }
}
