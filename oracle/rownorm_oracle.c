/*
 * Plain C float64 oracle for row-wise LayerNorm / RMSNorm forward.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the test suite, the smoke check
 * and the CPU-baseline leg of the benchmark load this file's library. It
 * shares no code, header or constant with the CUDA library.
 *
 * Every input is the exact FP32 value the GPU receives, widened to double.
 * One row at a time, in the order the definitions are written; no blocking,
 * no fusion, no reordering.
 */
#include <math.h>
#include <stdint.h>

/*
 * LayerNorm forward.
 * Statistics: "Rewriting the layer norm and matmul kernels", section
 * "A reduction has to meet somewhere" (displayed equation):
 *   mu_i = (1/d) sum_j x_ij,   sigma_i^2 = (1/d) sum_j (x_ij - mu_i)^2.
 * Output: the affine layer-normalization map with eps inside the root,
 *   rstd_i = (sigma_i^2 + eps)^(-1/2),  y_ij = (x_ij - mu_i) rstd_i gamma_j + beta_j.
 * y is [rows*d], mean and rstd are [rows]; all float64.
 */
void oracle_layer_norm(const float *x, const float *gamma, const float *beta,
                       int64_t rows, int64_t d, float eps,
                       double *y, double *mean, double *rstd)
{
    for (int64_t i = 0; i < rows; ++i) {
        const float *xi = x + i * d;
        double sum = 0.0;
        for (int64_t j = 0; j < d; ++j)
            sum += (double)xi[j];
        double mu = sum / (double)d;

        double sq = 0.0;
        for (int64_t j = 0; j < d; ++j) {
            double c = (double)xi[j] - mu;
            sq += c * c;
        }
        double var = sq / (double)d;
        double rs = 1.0 / sqrt(var + (double)eps);

        for (int64_t j = 0; j < d; ++j)
            y[i * d + j] = ((double)xi[j] - mu) * rs * (double)gamma[j] + (double)beta[j];
        mean[i] = mu;
        rstd[i] = rs;
    }
}

/*
 * RMSNorm forward: "RMSNorm on an RTX 5070 ...", section "The operator and
 * the change" (displayed equation):
 *   y_rc = x_rc w_c ( (1/D) sum_j x_rj^2 + eps )^(-1/2).
 * y is [rows*d] and r (the per-row scale) is [rows]; all float64.
 */
void oracle_rms_norm(const float *x, const float *w, int64_t rows, int64_t d,
                     float eps, double *y, double *r)
{
    for (int64_t i = 0; i < rows; ++i) {
        const float *xi = x + i * d;
        double sq = 0.0;
        for (int64_t j = 0; j < d; ++j)
            sq += (double)xi[j] * (double)xi[j];
        double ms = sq / (double)d;
        double ri = 1.0 / sqrt(ms + (double)eps);
        for (int64_t j = 0; j < d; ++j)
            y[i * d + j] = (double)xi[j] * (double)w[j] * ri;
        r[i] = ri;
    }
}
