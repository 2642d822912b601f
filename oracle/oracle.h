/*
 * CPU oracle for the FP32 row reductions: TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this code. The CUDA library never includes, links or calls it, and
 * it shares no code with the CUDA path.
 *
 * Two families:
 *   oracle_*_f64  the plain definitions, evaluated serially in FP64 (every
 *                 input widened to double, one rounding at the very end is
 *                 left to the caller: outputs are returned as double);
 *   ot_*_f32      a bit-exact FP32 emulation of the ordered fixed-tree policy
 *                 ("OT-1024"), including its own exp/log.
 *
 * All tensors are row-major contiguous: x[r*cols + c]. Weight/bias pointers
 * may be NULL (weight 1, bias 0). Labels are int64; a label outside [0, cols)
 * selects the fill value 0. Every function returns 0, or -1 for bad sizes.
 */
#ifndef FP32_ROW_REDUCTION_ORACLE_H
#define FP32_ROW_REDUCTION_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int oracle_softmax_f64(const float *x, double *y, int64_t rows, int64_t cols);
int oracle_rmsnorm_f64(const float *x, const float *w, double *y,
                       int64_t rows, int64_t cols, float eps);
int oracle_layernorm_f64(const float *x, const float *gamma, const float *beta,
                         double *y, int64_t rows, int64_t cols, float eps);
int oracle_cross_entropy_f64(const float *logits, const int64_t *labels,
                             double *loss, int64_t rows, int64_t cols);

float ot_expf(float x);
float ot_logf(float x);
void ot_expf_n(const float *x, float *y, int64_t n);
void ot_logf_n(const float *x, float *y, int64_t n);
float ot_sum_f32(const float *v, int64_t n);
float ot_max_f32(const float *v, int64_t n);
float ot_min_f32(const float *v, int64_t n);
int ot_softmax_f32(const float *x, float *y, int64_t rows, int64_t cols);
int ot_rmsnorm_f32(const float *x, const float *w, float *y,
                   int64_t rows, int64_t cols, float eps);
int ot_layernorm_f32(const float *x, const float *gamma, const float *beta,
                     float *y, int64_t rows, int64_t cols, float eps);
int ot_cross_entropy_f32(const float *logits, const int64_t *labels,
                         float *loss, int64_t rows, int64_t cols);

int oracle_softmax_bwd_f64(const float *y, const float *dy, double *dx, int64_t rows, int64_t cols);
int oracle_cross_entropy_bwd_f64(const float *logits, const int64_t *labels, const float *dloss, double *dx,
                                 int64_t rows, int64_t cols);
int oracle_rmsnorm_bwd_f64(const float *x, const float *w, const float *dy, double *dx, double *dw,
                           int64_t rows, int64_t cols, float eps);
int oracle_layernorm_bwd_f64(const float *x, const float *gamma, const float *dy, double *dx, double *dgamma,
                             double *dbeta, int64_t rows, int64_t cols, float eps);
int ot_softmax_bwd_f32(const float *y, const float *dy, float *dx, int64_t rows, int64_t cols);
int ot_cross_entropy_bwd_f32(const float *logits, const int64_t *labels, const float *dloss, float *dx,
                             int64_t rows, int64_t cols);
int ot_rmsnorm_bwd_f32(const float *x, const float *w, const float *dy, float *dx, float *dw,
                       int64_t rows, int64_t cols, float eps);
int ot_layernorm_bwd_f32(const float *x, const float *gamma, const float *dy, float *dx, float *dgamma,
                         float *dbeta, int64_t rows, int64_t cols, float eps);

float fold_sum_f32(const float *v, int64_t n, int right);
float fold_max_f32(const float *v, int64_t n, int right);
float fold_min_f32(const float *v, int64_t n, int right);
int fold_softmax_f32(const float *x, float *y, int64_t rows, int64_t cols, int right);
int fold_rmsnorm_f32(const float *x, const float *w, float *y, int64_t rows, int64_t cols, float eps, int right);
int fold_layernorm_f32(const float *x, const float *gamma, const float *beta, float *y, int64_t rows, int64_t cols,
                       float eps, int right);
int fold_cross_entropy_f32(const float *logits, const int64_t *labels, float *loss, int64_t rows, int64_t cols,
                           int right);

/* Unordered maximum / minimum: NaN elements skipped (NaN only when all are NaN). */
int skipnan_row_max_f32(const float *x, float *out, int64_t rows, int64_t cols);
int skipnan_row_min_f32(const float *x, float *out, int64_t rows, int64_t cols);
int skipnan_axis_max_f32(const float *x, float *out, int64_t outer, int64_t extent, int64_t inner);
int skipnan_axis_min_f32(const float *x, float *out, int64_t outer, int64_t extent, int64_t inner);

#ifdef __cplusplus
}
#endif
#endif
