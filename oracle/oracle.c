/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the six per-row
 * FP32 reduction operators.  TEST INFRASTRUCTURE ONLY: the product library
 * never links, loads or calls this file; only the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg do.
 *
 * Every function works one row at a time with scalar loops.  Inputs are FP32
 * (as the GPU receives them); every intermediate is held in double and the
 * outputs are returned in double, i.e. the exact-as-possible value before the
 * single rounding to FP32 that the GPU path performs at its store.  This is
 * the reading of "FP32 reduction and epilogue arithmetic, rounding only on
 * the output store" (Thread Ownership and Software Staging,
 * §Register-tiled reductions, the rmsnorm_register paragraph), carried one
 * precision higher so that it bounds the GPU's FP32 rounding error.
 *
 * Formulas (n = cols, all sums over the n entries of one row):
 *   rmsnorm     ms = sum(x^2)/n;  y = x / sqrt(ms + eps) * w
 *   layernorm   mu = sum(x)/n; var = sum((x-mu)^2)/n (biased, two-pass);
 *               y = (x - mu) / sqrt(var + eps) * gamma + beta
 *   residual LN h = x + r; y = layernorm(h); h_out = fl32(x + r)
 *   softmax     m = max(x); e = exp(x - m); y = e / sum(e)
 *   row sum     s = sum(x)
 *   cross-ent.  loss = m + log(sum(exp(x - m))) - x[label]; mean = sum(loss)/R
 * Fused variants on the same rows (the pages name none of them; they are
 * the plain compositions of the definitions above):
 *   residual RMSNorm  h = x + r; y = rmsnorm(h); h_out = fl32(x + r)
 *   log-softmax       y = (x - m) - log(sum(exp(x - m)))
 *   cross-entropy with an ignore index: rows whose label equals it have
 *                     loss 0 and are left out of the mean, which divides by
 *                     the number of other rows (NaN when there are none)
 * The operator family is named in "Consecutive-worker reduction layout
 * checkpoint", §Evidence and what remains (the generic V=4 operator coverage
 * run: sum, softmax, RMSNorm, LayerNorm, residual LayerNorm, cross-entropy).
 * The pages give no formula for LayerNorm, residual LayerNorm or
 * cross-entropy; the plain textbook definitions above are the reading used.
 *
 * NULL weight / gamma means 1, NULL beta means 0.  A label outside [0, n)
 * gives a NaN loss for that row (and a NaN mean).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#define ORACLE_API __attribute__((visibility("default")))

ORACLE_API void oracle_rmsnorm_f64(const float *x, const float *w,
                                   int64_t rows, int64_t cols, double eps,
                                   double *y)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        double *yr = y + r * cols;
        double ss = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double v = (double)xr[j];
            ss += v * v;
        }
        double ms = ss / (double)cols;
        double denom = sqrt(ms + eps);
        for (int64_t j = 0; j < cols; ++j) {
            double wj = w ? (double)w[j] : 1.0;
            yr[j] = (double)xr[j] / denom * wj;
        }
    }
}

/* LayerNorm of one row held in double. */
static void layernorm_row(const double *h, const float *gamma,
                          const float *beta, int64_t cols, double eps,
                          double *y)
{
    double s = 0.0;
    for (int64_t j = 0; j < cols; ++j)
        s += h[j];
    double mu = s / (double)cols;
    double sq = 0.0;
    for (int64_t j = 0; j < cols; ++j) {
        double d = h[j] - mu;
        sq += d * d;
    }
    double var = sq / (double)cols;
    double denom = sqrt(var + eps);
    for (int64_t j = 0; j < cols; ++j) {
        double g = gamma ? (double)gamma[j] : 1.0;
        double b = beta ? (double)beta[j] : 0.0;
        y[j] = (h[j] - mu) / denom * g + b;
    }
}

/* `scratch` holds one row of doubles (cols entries), owned by the caller. */
ORACLE_API void oracle_layernorm_f64(const float *x, const float *gamma,
                                     const float *beta, int64_t rows,
                                     int64_t cols, double eps, double *y,
                                     double *scratch)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        for (int64_t j = 0; j < cols; ++j)
            scratch[j] = (double)xr[j];
        layernorm_row(scratch, gamma, beta, cols, eps, y + r * cols);
    }
}

ORACLE_API void oracle_residual_layernorm_f64(
    const float *x, const float *res, const float *gamma, const float *beta,
    int64_t rows, int64_t cols, double eps, double *y, float *h_out,
    double *scratch)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        const float *rr = res + r * cols;
        for (int64_t j = 0; j < cols; ++j) {
            /* The sum of two floats is exact in double for the magnitudes
             * used here; its single rounding to float is then the correctly
             * rounded FP32 sum. */
            double h = (double)xr[j] + (double)rr[j];
            scratch[j] = h;
            if (h_out)
                h_out[r * cols + j] = (float)h;
        }
        layernorm_row(scratch, gamma, beta, cols, eps, y + r * cols);
    }
}

ORACLE_API void oracle_softmax_f64(const float *x, int64_t rows, int64_t cols,
                                   double *y)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        double *yr = y + r * cols;
        double m = -INFINITY;
        int has_nan = 0;
        for (int64_t j = 0; j < cols; ++j) {
            double v = (double)xr[j];
            if (v != v)
                has_nan = 1;
            if (v > m)
                m = v;
        }
        if (has_nan) {
            for (int64_t j = 0; j < cols; ++j)
                yr[j] = NAN;
            continue;
        }
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            yr[j] = exp((double)xr[j] - m);
            s += yr[j];
        }
        for (int64_t j = 0; j < cols; ++j)
            yr[j] = yr[j] / s;
    }
}

ORACLE_API void oracle_row_sum_f64(const float *x, int64_t rows, int64_t cols,
                                   double *out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            s += (double)xr[j];
        out[r] = s;
    }
}

ORACLE_API void oracle_cross_entropy_f64(const float *logits,
                                         const int32_t *labels, int64_t rows,
                                         int64_t cols, double *loss,
                                         double *mean)
{
    double total = 0.0;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = logits + r * cols;
        int32_t lab = labels[r];
        if (lab < 0 || (int64_t)lab >= cols) {
            loss[r] = NAN;
            total += NAN;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < cols; ++j)
            if ((double)xr[j] > m)
                m = (double)xr[j];
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            s += exp((double)xr[j] - m);
        loss[r] = m + log(s) - (double)xr[lab];
        total += loss[r];
    }
    if (mean)
        *mean = rows > 0 ? total / (double)rows : NAN;
}

ORACLE_API void oracle_residual_rmsnorm_f64(const float *x, const float *res,
                                            const float *w, int64_t rows,
                                            int64_t cols, double eps,
                                            double *y, float *h_out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        const float *rr = res + r * cols;
        double *yr = y + r * cols;
        double ss = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double h = (double)xr[j] + (double)rr[j];
            yr[j] = h; /* keep h until the scale is known */
            ss += h * h;
            if (h_out)
                h_out[r * cols + j] = (float)h;
        }
        double denom = sqrt(ss / (double)cols + eps);
        for (int64_t j = 0; j < cols; ++j) {
            double wj = w ? (double)w[j] : 1.0;
            yr[j] = yr[j] / denom * wj;
        }
    }
}

ORACLE_API void oracle_log_softmax_f64(const float *x, int64_t rows,
                                       int64_t cols, double *y)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        double *yr = y + r * cols;
        double m = -INFINITY;
        int has_nan = 0;
        for (int64_t j = 0; j < cols; ++j) {
            double v = (double)xr[j];
            if (v != v)
                has_nan = 1;
            if (v > m)
                m = v;
        }
        if (has_nan) {
            for (int64_t j = 0; j < cols; ++j)
                yr[j] = NAN;
            continue;
        }
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            s += exp((double)xr[j] - m);
        double ls = log(s);
        for (int64_t j = 0; j < cols; ++j)
            yr[j] = ((double)xr[j] - m) - ls;
    }
}

ORACLE_API void oracle_cross_entropy_ignore_f64(const float *logits,
                                                const int32_t *labels,
                                                int32_t ignore_index,
                                                int64_t rows, int64_t cols,
                                                double *loss, double *mean)
{
    double total = 0.0;
    int64_t counted = 0;
    for (int64_t r = 0; r < rows; ++r) {
        if (labels[r] == ignore_index) {
            loss[r] = 0.0;
            continue;
        }
        /* one row through the plain definition */
        oracle_cross_entropy_f64(logits + r * cols, labels + r, 1, cols,
                                 loss + r, NULL);
        total += loss[r];
        counted += 1;
    }
    if (mean)
        *mean = counted > 0 ? total / (double)counted : NAN;
}
