/*
 * CPU oracle for the FP32 row reductions: TEST INFRASTRUCTURE ONLY.
 * (Only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * it; the CUDA library never includes, links or calls this file.)
 *
 * Part 1, oracle_*_f64: the plain definitions of the four row operators,
 * serial, in FP64. Sources ("TIRx Metal reduction lowering" page):
 *   softmax        §1 "The frontend stays execution-first", row softmax
 *                  program: exp(value - reduce(value, max)) / reduce(., add)
 *   cross-entropy  §1, cross-entropy program: log(total) + peak - selected,
 *                  and §5.2 "Guarded immutable views and dynamic gather":
 *                  selected = (0 <= label < N) ? logits[row, label] : 0
 *   LayerNorm      §5.1 "Shared SSA is not a physical allocation decision":
 *                  mean = sum/width, centered = x - mean,
 *                  variance = sum(centered^2)/width, centered/sqrt(var+eps);
 *                  the affine (gamma, beta) is the "affine outputs" of the
 *                  §8 LayerNorm test, applied as (c/sigma)*gamma + beta
 *   RMSNorm        named as an operator on the "Whole-launch reduction cost
 *                  policy" page (held-out results) but never written out.
 *                  Reading: y = x / sqrt(mean(x^2) + eps) * w (eps inside the
 *                  root, as for LayerNorm).
 * §8 "Correctness and structural verification" checks every output against
 * an FP64 formula; this file is that formula.
 *
 * Part 2, ot_*_f32: bit-exact FP32 emulation of the ordered policy. The page
 * (§1, ReductionPolicy: unordered_tree / ordered_tree / fold_left /
 * fold_right; "an ordered tree ... stays ordered"; precise math required)
 * names an ordered tree but fixes no shape, so this library defines one,
 * "OT-1024", independent of how a kernel maps it:
 *   leaf k in [0,1024): fold_left over the columns e with e % 1024 == k in
 *                       increasing e, starting from the identity;
 *   partial t in [0,256): (leaf[4t] (+) leaf[4t+1]) (+) (leaf[4t+2] (+) leaf[4t+3]);
 *   32 partials of a group g (partials 32g..32g+31): xor butterfly with
 *                       offsets 16, 8, 4, 2, 1 (v_l = v_l (+) v_{l^o});
 *   8 group results:    ((g0 (+) g1) (+) (g2 (+) g3)) (+) ((g4 (+) g5) (+) (g6 (+) g7)).
 * All arithmetic is IEEE binary32 round-to-nearest-even with no FMA
 * contraction (this file is compiled with -ffp-contract=off), no flush to
 * zero, IEEE division and square root, and the exp/log defined below.
 * A row is divided by its normaliser (softmax sum, RMS, LayerNorm sigma) as a
 * multiplication by the correctly rounded reciprocal of that normaliser: one
 * IEEE division per row, then one rounded product per element.
 */
#include "oracle.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Part 1: FP64 definitions                                                   */
/* ------------------------------------------------------------------------- */

static int bad_sizes(int64_t rows, int64_t cols) { return rows < 0 || cols < 1; }

int oracle_softmax_f64(const float *x, double *y, int64_t rows, int64_t cols) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        double *yr = y + r * cols;
        double peak = -INFINITY;
        for (int64_t c = 0; c < cols; ++c)
            if ((double)xr[c] > peak) peak = (double)xr[c];
        double total = 0.0;
        for (int64_t c = 0; c < cols; ++c) total += exp((double)xr[c] - peak);
        for (int64_t c = 0; c < cols; ++c) yr[c] = exp((double)xr[c] - peak) / total;
    }
    return 0;
}

int oracle_rmsnorm_f64(const float *x, const float *w, double *y,
                       int64_t rows, int64_t cols, float eps) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        double *yr = y + r * cols;
        double sumsq = 0.0;
        for (int64_t c = 0; c < cols; ++c) sumsq += (double)xr[c] * (double)xr[c];
        double rms = sqrt(sumsq / (double)cols + (double)eps);
        for (int64_t c = 0; c < cols; ++c)
            yr[c] = (double)xr[c] / rms * (w ? (double)w[c] : 1.0);
    }
    return 0;
}

int oracle_layernorm_f64(const float *x, const float *gamma, const float *beta,
                         double *y, int64_t rows, int64_t cols, float eps) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        double *yr = y + r * cols;
        double sum = 0.0;
        for (int64_t c = 0; c < cols; ++c) sum += (double)xr[c];
        double mean = sum / (double)cols;
        double sq = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            double centered = (double)xr[c] - mean;
            sq += centered * centered;
        }
        double sigma = sqrt(sq / (double)cols + (double)eps);
        for (int64_t c = 0; c < cols; ++c) {
            double v = ((double)xr[c] - mean) / sigma;
            if (gamma) v *= (double)gamma[c];
            if (beta) v += (double)beta[c];
            yr[c] = v;
        }
    }
    return 0;
}

int oracle_cross_entropy_f64(const float *logits, const int64_t *labels,
                             double *loss, int64_t rows, int64_t cols) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = logits + r * cols;
        double peak = -INFINITY;
        for (int64_t c = 0; c < cols; ++c)
            if ((double)xr[c] > peak) peak = (double)xr[c];
        double total = 0.0;
        for (int64_t c = 0; c < cols; ++c) total += exp((double)xr[c] - peak);
        int64_t label = labels[r];
        double selected = (label >= 0 && label < cols) ? (double)xr[label] : 0.0;
        loss[r] = log(total) + peak - selected;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Part 2: OT-1024 emulation                                                  */
/* ------------------------------------------------------------------------- */

/* Float helpers on bit patterns (no library rounding involved). */
static float bits_to_f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
/* 2^n as a float for n in [-126, 127]. */
static float pow2i(int n) { return bits_to_f((uint32_t)(n + 127) << 23); }

/*
 * ot_expf: exp on binary32, defined step by step so that a host and a GPU
 * computing it with IEEE operations get identical bits.
 * Method: Cody & Waite argument reduction (W. J. Cody, W. Waite, "Software
 * Manual for the Elementary Functions", 1980) x = k ln2 + r with ln2 split in
 * two floats, then the Taylor series of e^r through r^7/7! (remainder below
 * 5e-9 relative for |r| <= ln2/2), then scaling by 2^k in two exact halves.
 * Constants are the binary32 roundings of the mathematical values:
 *   L2E = RN(1/ln2), LN2_HI = RN(ln2), LN2_LO = RN(ln2 - LN2_HI), C_i = RN(1/i!).
 */
#define OT_L2E 0x1.715476p+0f
#define OT_LN2_HI 0x1.62e430p-1f
#define OT_LN2_LO -0x1.05c610p-29f
#define OT_C2 0x1.000000p-1f
#define OT_C3 0x1.555556p-3f
#define OT_C4 0x1.555556p-5f
#define OT_C5 0x1.111112p-7f
#define OT_C6 0x1.6c16c2p-10f
#define OT_C7 0x1.a01a02p-13f

float ot_expf(float x) {
    if (x != x) return x + x;          /* NaN */
    if (x > 100.0f) return INFINITY;   /* far beyond ln(FLT_MAX) */
    if (x < -110.0f) return 0.0f;      /* far below ln(min subnormal) */
    float kf = rintf(x * OT_L2E);      /* nearest integer, ties to even */
    int k = (int)kf;
    float r = fmaf(-kf, OT_LN2_HI, x);
    r = fmaf(-kf, OT_LN2_LO, r);
    float p = OT_C7;
    p = fmaf(p, r, OT_C6);
    p = fmaf(p, r, OT_C5);
    p = fmaf(p, r, OT_C4);
    p = fmaf(p, r, OT_C3);
    p = fmaf(p, r, OT_C2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int k1 = k >> 1;                   /* floor(k/2): both factors stay normal */
    int k2 = k - k1;
    return (p * pow2i(k1)) * pow2i(k2);
}

/*
 * ot_logf: natural log on binary32 (only positive finite arguments matter to
 * the ordered cross-entropy, whose argument is a sum >= 1).
 * Method: x = 2^e * m with m in (sqrt(1/2), sqrt(2)], f = m - 1 (exact), and
 * log m = 2 atanh(s) with s = f / (2 + f), |s| <= 0.1716.  Since 2s = f - s*f,
 *   2 atanh(s) = f - s * (f - R),  R = (2/3)s^2 + (2/5)s^4 + (2/7)s^6 + (2/9)s^8
 * (next term below 3e-10 relative), so the leading term f is exact and only
 * the small correction s*(f - R) carries rounding error.  Finally
 * log x = e*LN2_HI + (e*LN2_LO + log m).
 * Constants: RN(2/3), RN(2/5), RN(2/7), RN(2/9), RN(sqrt 2).
 */
#define OT_T3 0x1.555556p-1f
#define OT_T5 0x1.99999ap-2f
#define OT_T7 0x1.24924ap-2f
#define OT_T9 0x1.c71c72p-3f
#define OT_SQRT2 0x1.6a09e6p+0f

float ot_logf(float x) {
    if (x != x) return x + x;
    if (x < 0.0f) return NAN;
    if (x == 0.0f) return -INFINITY;
    if (x == INFINITY) return x;
    int e = 0;
    if (x < 0x1p-126f) { x = x * 0x1p23f; e = -23; }   /* subnormal: exact scale */
    uint32_t u = f_to_bits(x);
    e += (int)((u >> 23) & 0xffu) - 127;
    float m = bits_to_f((u & 0x007fffffu) | 0x3f800000u);  /* [1, 2) */
    if (m > OT_SQRT2) { m = m * 0.5f; e += 1; }
    float f = m - 1.0f;
    float s = f / (2.0f + f);
    float z = s * s;
    float q = OT_T9;
    q = fmaf(q, z, OT_T7);
    q = fmaf(q, z, OT_T5);
    q = fmaf(q, z, OT_T3);
    float big_r = z * q;
    float lm = fmaf(-s, f - big_r, f);
    float ef = (float)e;
    return fmaf(ef, OT_LN2_HI, fmaf(ef, OT_LN2_LO, lm));
}

void ot_expf_n(const float *x, float *y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = ot_expf(x[i]);
}
void ot_logf_n(const float *x, float *y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = ot_logf(x[i]);
}

/* Canonical max: commutative for all non-NaN pairs (+0 beats -0). */
static float ot_max2(float a, float b) {
    if (a != a) return a;
    if (b != b) return b;
    if (a > b) return a;
    if (b > a) return b;
    return signbit(a) ? b : a;
}
/* Canonical min: NaN in the first operand wins, then NaN in the second, then
 * the smaller value, -0 over +0 (commutative for all non-NaN pairs). */
static float ot_min2(float a, float b) {
    if (a != a) return a;
    if (b != b) return b;
    if (a < b) return a;
    if (b < a) return b;
    return signbit(a) ? a : b;
}
static float ot_add2(float a, float b) { return a + b; }

enum { OT_LEAVES = 1024, OT_PARTIALS = 256, OT_GROUPS = 8, OT_LANES = 32 };

/* The fixed tree above the 1024 leaves. */
static float ot_tree(const float *leaf, float (*op)(float, float)) {
    float part[OT_PARTIALS];
    for (int t = 0; t < OT_PARTIALS; ++t)
        part[t] = op(op(leaf[4 * t], leaf[4 * t + 1]), op(leaf[4 * t + 2], leaf[4 * t + 3]));
    float g[OT_GROUPS];
    for (int w = 0; w < OT_GROUPS; ++w) {
        float v[OT_LANES], nv[OT_LANES];
        for (int l = 0; l < OT_LANES; ++l) v[l] = part[w * OT_LANES + l];
        for (int o = 16; o >= 1; o >>= 1) {
            for (int l = 0; l < OT_LANES; ++l) nv[l] = op(v[l], v[l ^ o]);
            memcpy(v, nv, sizeof v);
        }
        g[w] = v[0];
    }
    return op(op(op(g[0], g[1]), op(g[2], g[3])), op(op(g[4], g[5]), op(g[6], g[7])));
}

float ot_sum_f32(const float *v, int64_t n) {
    float leaf[OT_LEAVES];
    for (int k = 0; k < OT_LEAVES; ++k) leaf[k] = 0.0f;
    for (int64_t e = 0; e < n; ++e) leaf[e % OT_LEAVES] = leaf[e % OT_LEAVES] + v[e];
    return ot_tree(leaf, ot_add2);
}

float ot_max_f32(const float *v, int64_t n) {
    float leaf[OT_LEAVES];
    for (int k = 0; k < OT_LEAVES; ++k) leaf[k] = -INFINITY;
    for (int64_t e = 0; e < n; ++e) leaf[e % OT_LEAVES] = ot_max2(leaf[e % OT_LEAVES], v[e]);
    return ot_tree(leaf, ot_max2);
}

float ot_min_f32(const float *v, int64_t n) {
    float leaf[OT_LEAVES];
    for (int k = 0; k < OT_LEAVES; ++k) leaf[k] = INFINITY;
    for (int64_t e = 0; e < n; ++e) leaf[e % OT_LEAVES] = ot_min2(leaf[e % OT_LEAVES], v[e]);
    return ot_tree(leaf, ot_min2);
}

/* Sum over the row of a per-element contribution, in OT-1024 order. */
typedef float (*ot_elem_fn)(float x, float a);
static float ot_sum_of(const float *xr, int64_t n, ot_elem_fn f, float a) {
    float leaf[OT_LEAVES];
    for (int k = 0; k < OT_LEAVES; ++k) leaf[k] = 0.0f;
    for (int64_t e = 0; e < n; ++e) leaf[e % OT_LEAVES] = leaf[e % OT_LEAVES] + f(xr[e], a);
    return ot_tree(leaf, ot_add2);
}
static float el_identity(float x, float a) { (void)a; return x; }
static float el_square(float x, float a) { (void)a; return x * x; }
static float el_centered_square(float x, float mean) { float c = x - mean; return c * c; }
static float el_exp_shifted(float x, float peak) { return ot_expf(x - peak); }

int ot_softmax_f32(const float *x, float *y, int64_t rows, int64_t cols) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        float *yr = y + r * cols;
        float peak = ot_max_f32(xr, cols);
        float total = ot_sum_of(xr, cols, el_exp_shifted, peak);
        float inv = 1.0f / total;
        for (int64_t c = 0; c < cols; ++c) yr[c] = ot_expf(xr[c] - peak) * inv;
    }
    return 0;
}

int ot_rmsnorm_f32(const float *x, const float *w, float *y,
                   int64_t rows, int64_t cols, float eps) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        float *yr = y + r * cols;
        float sumsq = ot_sum_of(xr, cols, el_square, 0.0f);
        float rms = sqrtf(sumsq / (float)cols + eps);
        float inv = 1.0f / rms;
        for (int64_t c = 0; c < cols; ++c) {
            float v = xr[c] * inv;
            yr[c] = w ? v * w[c] : v;
        }
    }
    return 0;
}

int ot_layernorm_f32(const float *x, const float *gamma, const float *beta,
                     float *y, int64_t rows, int64_t cols, float eps) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        float *yr = y + r * cols;
        float mean = ot_sum_of(xr, cols, el_identity, 0.0f) / (float)cols;
        float var = ot_sum_of(xr, cols, el_centered_square, mean) / (float)cols;
        float sigma = sqrtf(var + eps);
        float inv = 1.0f / sigma;
        for (int64_t c = 0; c < cols; ++c) {
            float v = (xr[c] - mean) * inv;
            if (gamma) v = v * gamma[c];
            if (beta) v = v + beta[c];
            yr[c] = v;
        }
    }
    return 0;
}

int ot_cross_entropy_f32(const float *logits, const int64_t *labels,
                         float *loss, int64_t rows, int64_t cols) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = logits + r * cols;
        float peak = ot_max_f32(xr, cols);
        float total = ot_sum_of(xr, cols, el_exp_shifted, peak);
        int64_t label = labels[r];
        float selected = (label >= 0 && label < cols) ? xr[label] : 0.0f;
        loss[r] = (ot_logf(total) + peak) - selected;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Part 3: backward passes (the gradients of the four row operators)          */
/* ------------------------------------------------------------------------- */
/*
 * Not on the pages (the next rows of the same row-reduction family). The FP64
 * functions are the derivatives of the Part 1 definitions, written out:
 *   softmax        dx_c = y_c (dy_c - sum_j dy_j y_j)
 *   cross-entropy  dx_c = dloss (p_c - [c == label]), p = softmax(logits); a
 *                  label outside [0, N) selects nothing, so no one-hot term;
 *                  dloss = 1 when no per-row upstream gradient is given
 *   RMSNorm        r = 1 / sqrt(mean(x^2) + eps), g = dy w:
 *                  dx_c = r (g_c - x_c r^2 mean(g x)), dw_c = sum_rows dy_c x_c r
 *   LayerNorm      xh = (x - mean) r, r = 1 / sqrt(var + eps), g = dy gamma:
 *                  dx_c = r (g_c - mean(g) - xh_c mean(g xh)),
 *                  dgamma_c = sum_rows dy_c xh_c, dbeta_c = sum_rows dy_c
 * The ot_*_bwd_f32 functions emulate the ordered policy: every row sum is
 * OT-1024 over the row's terms, every column sum (dw, dgamma, dbeta) is
 * OT-1024 over that column's per-row terms, and each step is the binary32
 * operation written below, in that order.
 */

int oracle_softmax_bwd_f64(const float *y, const float *dy, double *dx, int64_t rows, int64_t cols) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *yr = y + r * cols, *gr = dy + r * cols;
        double dot = 0.0;
        for (int64_t c = 0; c < cols; ++c) dot += (double)gr[c] * (double)yr[c];
        for (int64_t c = 0; c < cols; ++c) dx[r * cols + c] = (double)yr[c] * ((double)gr[c] - dot);
    }
    return 0;
}

int oracle_cross_entropy_bwd_f64(const float *logits, const int64_t *labels, const float *dloss, double *dx,
                                 int64_t rows, int64_t cols) {
    if (bad_sizes(rows, cols)) return -1;
    double *p = (double *)malloc((size_t)cols * sizeof(double));
    if (!p) return -2;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = logits + r * cols;
        double peak = -INFINITY;
        for (int64_t c = 0; c < cols; ++c) if ((double)xr[c] > peak) peak = (double)xr[c];
        double total = 0.0;
        for (int64_t c = 0; c < cols; ++c) { p[c] = exp((double)xr[c] - peak); total += p[c]; }
        const double scale = dloss ? (double)dloss[r] : 1.0;
        for (int64_t c = 0; c < cols; ++c) {
            double d = p[c] / total - (c == labels[r] ? 1.0 : 0.0);
            dx[r * cols + c] = scale * d;
        }
    }
    free(p);
    return 0;
}

int oracle_rmsnorm_bwd_f64(const float *x, const float *w, const float *dy, double *dx, double *dw,
                           int64_t rows, int64_t cols, float eps) {
    if (bad_sizes(rows, cols)) return -1;
    if (dw) for (int64_t c = 0; c < cols; ++c) dw[c] = 0.0;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols, *gr = dy + r * cols;
        double ss = 0.0, gx = 0.0;
        for (int64_t c = 0; c < cols; ++c) ss += (double)xr[c] * (double)xr[c];
        const double inv = 1.0 / sqrt(ss / (double)cols + (double)eps);
        for (int64_t c = 0; c < cols; ++c) gx += (double)gr[c] * (w ? (double)w[c] : 1.0) * (double)xr[c];
        const double k = gx / (double)cols * inv * inv;
        for (int64_t c = 0; c < cols; ++c) {
            const double g = (double)gr[c] * (w ? (double)w[c] : 1.0);
            dx[r * cols + c] = inv * (g - (double)xr[c] * k);
            if (dw) dw[c] += (double)gr[c] * (double)xr[c] * inv;
        }
    }
    return 0;
}

int oracle_layernorm_bwd_f64(const float *x, const float *gamma, const float *dy, double *dx, double *dgamma,
                             double *dbeta, int64_t rows, int64_t cols, float eps) {
    if (bad_sizes(rows, cols)) return -1;
    if (dgamma) for (int64_t c = 0; c < cols; ++c) dgamma[c] = 0.0;
    if (dbeta) for (int64_t c = 0; c < cols; ++c) dbeta[c] = 0.0;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols, *gr = dy + r * cols;
        double sum = 0.0, sq = 0.0, sg = 0.0, sgx = 0.0;
        for (int64_t c = 0; c < cols; ++c) sum += (double)xr[c];
        const double mean = sum / (double)cols;
        for (int64_t c = 0; c < cols; ++c) sq += ((double)xr[c] - mean) * ((double)xr[c] - mean);
        const double inv = 1.0 / sqrt(sq / (double)cols + (double)eps);
        for (int64_t c = 0; c < cols; ++c) {
            const double g = (double)gr[c] * (gamma ? (double)gamma[c] : 1.0);
            sg += g;
            sgx += g * ((double)xr[c] - mean) * inv;
        }
        const double a = sg / (double)cols, b = sgx / (double)cols;
        for (int64_t c = 0; c < cols; ++c) {
            const double g = (double)gr[c] * (gamma ? (double)gamma[c] : 1.0);
            const double xh = ((double)xr[c] - mean) * inv;
            dx[r * cols + c] = inv * (g - a - xh * b);
            if (dgamma) dgamma[c] += (double)gr[c] * xh;
            if (dbeta) dbeta[c] += (double)gr[c];
        }
    }
    return 0;
}

/* OT-1024 over the columns of a rows x cols term matrix: out[c] = OT_sum(t[., c]). */
static int ot_column_sums(const float *t, float *out, int64_t rows, int64_t cols) {
    float *col = (float *)malloc((size_t)(rows > 0 ? rows : 1) * sizeof(float));
    if (!col) return -2;
    for (int64_t c = 0; c < cols; ++c) {
        for (int64_t r = 0; r < rows; ++r) col[r] = t[r * cols + c];
        out[c] = ot_sum_f32(col, rows);
    }
    free(col);
    return 0;
}

int ot_softmax_bwd_f32(const float *y, const float *dy, float *dx, int64_t rows, int64_t cols) {
    if (bad_sizes(rows, cols)) return -1;
    float *t = (float *)malloc((size_t)cols * sizeof(float));
    if (!t) return -2;
    for (int64_t r = 0; r < rows; ++r) {
        const float *yr = y + r * cols, *gr = dy + r * cols;
        for (int64_t c = 0; c < cols; ++c) t[c] = gr[c] * yr[c];
        const float s = ot_sum_f32(t, cols);
        for (int64_t c = 0; c < cols; ++c) dx[r * cols + c] = yr[c] * (gr[c] - s);
    }
    free(t);
    return 0;
}

int ot_cross_entropy_bwd_f32(const float *logits, const int64_t *labels, const float *dloss, float *dx,
                             int64_t rows, int64_t cols) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = logits + r * cols;
        const float peak = ot_max_f32(xr, cols);
        const float total = ot_sum_of(xr, cols, el_exp_shifted, peak);
        const float inv = 1.0f / total;
        for (int64_t c = 0; c < cols; ++c) {
            const float p = ot_expf(xr[c] - peak) * inv;
            const float d = c == labels[r] ? p - 1.0f : p;
            dx[r * cols + c] = dloss ? d * dloss[r] : d;
        }
    }
    return 0;
}

int ot_rmsnorm_bwd_f32(const float *x, const float *w, const float *dy, float *dx, float *dw,
                       int64_t rows, int64_t cols, float eps) {
    if (bad_sizes(rows, cols)) return -1;
    float *t = (float *)malloc((size_t)cols * sizeof(float));
    float *terms = dw ? (float *)malloc((size_t)(rows > 0 ? rows : 1) * (size_t)cols * sizeof(float)) : NULL;
    if (!t || (dw && !terms)) { free(t); free(terms); return -2; }
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols, *gr = dy + r * cols;
        const float ss = ot_sum_of(xr, cols, el_square, 0.0f);
        const float rms = sqrtf(ss / (float)cols + eps);
        const float inv = 1.0f / rms;
        for (int64_t c = 0; c < cols; ++c) t[c] = (w ? gr[c] * w[c] : gr[c]) * xr[c];
        const float cs = ot_sum_f32(t, cols);
        const float k = ((cs / (float)cols) * inv) * inv;
        for (int64_t c = 0; c < cols; ++c) {
            const float g = w ? gr[c] * w[c] : gr[c];
            dx[r * cols + c] = inv * (g - xr[c] * k);
            if (terms) terms[r * cols + c] = (gr[c] * xr[c]) * inv;
        }
    }
    int rc = terms ? ot_column_sums(terms, dw, rows, cols) : 0;
    free(t);
    free(terms);
    return rc;
}

int ot_layernorm_bwd_f32(const float *x, const float *gamma, const float *dy, float *dx, float *dgamma,
                         float *dbeta, int64_t rows, int64_t cols, float eps) {
    if (bad_sizes(rows, cols)) return -1;
    const size_t n = (size_t)(rows > 0 ? rows : 1) * (size_t)cols;
    float *t = (float *)malloc((size_t)cols * sizeof(float));
    float *xh = (float *)malloc((size_t)cols * sizeof(float));
    float *tg = dgamma ? (float *)malloc(n * sizeof(float)) : NULL;
    float *tb = dbeta ? (float *)malloc(n * sizeof(float)) : NULL;
    if (!t || !xh || (dgamma && !tg) || (dbeta && !tb)) { free(t); free(xh); free(tg); free(tb); return -2; }
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols, *gr = dy + r * cols;
        const float mean = ot_sum_of(xr, cols, el_identity, 0.0f) / (float)cols;
        const float var = ot_sum_of(xr, cols, el_centered_square, mean) / (float)cols;
        const float sigma = sqrtf(var + eps);
        const float inv = 1.0f / sigma;
        for (int64_t c = 0; c < cols; ++c) {
            xh[c] = (xr[c] - mean) * inv;
            t[c] = gamma ? gr[c] * gamma[c] : gr[c];
        }
        const float sa = ot_sum_f32(t, cols);
        for (int64_t c = 0; c < cols; ++c) t[c] = (gamma ? gr[c] * gamma[c] : gr[c]) * xh[c];
        const float sb = ot_sum_f32(t, cols);
        const float a = sa / (float)cols, b = sb / (float)cols;
        for (int64_t c = 0; c < cols; ++c) {
            const float g = gamma ? gr[c] * gamma[c] : gr[c];
            dx[r * cols + c] = inv * ((g - a) - xh[c] * b);
            if (tg) tg[r * cols + c] = gr[c] * xh[c];
            if (tb) tb[r * cols + c] = gr[c];
        }
    }
    int rc = 0;
    if (tg) rc = ot_column_sums(tg, dgamma, rows, cols);
    if (!rc && tb) rc = ot_column_sums(tb, dbeta, rows, cols);
    free(t);
    free(xh);
    free(tg);
    free(tb);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Part 4: the fold policies                                                  */
/* ------------------------------------------------------------------------- */
/*
 * "TIRx Metal reduction lowering" §1 (ReductionPolicy): besides the trees, a
 * reduction may be restricted to fold_left or fold_right, and "stays ordered".
 * Reading: fold_left visits the columns in increasing order with the
 * accumulator as the left operand, acc = acc (+) t_c, starting from the
 * identity; fold_right visits them in decreasing order with the accumulator as
 * the right operand, acc = t_c (+) acc. Max and min are the canonical selects
 * of Part 2. The operators keep the op sequences of Part 2 with every
 * OT-1024 reduction replaced by the fold (the same exp/log).
 */
static float fold_sum_of(const float *xr, int64_t n, ot_elem_fn f, float a, int right) {
    float acc = 0.0f;
    if (!right)
        for (int64_t e = 0; e < n; ++e) acc = acc + f(xr[e], a);
    else
        for (int64_t e = n - 1; e >= 0; --e) acc = f(xr[e], a) + acc;
    return acc;
}

float fold_sum_f32(const float *v, int64_t n, int right) { return fold_sum_of(v, n, el_identity, 0.0f, right); }

float fold_max_f32(const float *v, int64_t n, int right) {
    float acc = -INFINITY;
    if (!right)
        for (int64_t e = 0; e < n; ++e) acc = ot_max2(acc, v[e]);
    else
        for (int64_t e = n - 1; e >= 0; --e) acc = ot_max2(v[e], acc);
    return acc;
}

float fold_min_f32(const float *v, int64_t n, int right) {
    float acc = INFINITY;
    if (!right)
        for (int64_t e = 0; e < n; ++e) acc = ot_min2(acc, v[e]);
    else
        for (int64_t e = n - 1; e >= 0; --e) acc = ot_min2(v[e], acc);
    return acc;
}

int fold_softmax_f32(const float *x, float *y, int64_t rows, int64_t cols, int right) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        const float peak = fold_max_f32(xr, cols, right);
        const float inv = 1.0f / fold_sum_of(xr, cols, el_exp_shifted, peak, right);
        for (int64_t c = 0; c < cols; ++c) y[r * cols + c] = ot_expf(xr[c] - peak) * inv;
    }
    return 0;
}

int fold_rmsnorm_f32(const float *x, const float *w, float *y, int64_t rows, int64_t cols, float eps, int right) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        const float rms = sqrtf(fold_sum_of(xr, cols, el_square, 0.0f, right) / (float)cols + eps);
        const float inv = 1.0f / rms;
        for (int64_t c = 0; c < cols; ++c) {
            const float v = xr[c] * inv;
            y[r * cols + c] = w ? v * w[c] : v;
        }
    }
    return 0;
}

int fold_layernorm_f32(const float *x, const float *gamma, const float *beta, float *y, int64_t rows, int64_t cols,
                       float eps, int right) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        const float mean = fold_sum_of(xr, cols, el_identity, 0.0f, right) / (float)cols;
        const float var = fold_sum_of(xr, cols, el_centered_square, mean, right) / (float)cols;
        const float inv = 1.0f / sqrtf(var + eps);
        for (int64_t c = 0; c < cols; ++c) {
            float v = (xr[c] - mean) * inv;
            if (gamma) v = v * gamma[c];
            if (beta) v = v + beta[c];
            y[r * cols + c] = v;
        }
    }
    return 0;
}

int fold_cross_entropy_f32(const float *logits, const int64_t *labels, float *loss, int64_t rows, int64_t cols,
                           int right) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = logits + r * cols;
        const float peak = fold_max_f32(xr, cols, right);
        const float total = fold_sum_of(xr, cols, el_exp_shifted, peak, right);
        const int64_t label = labels[r];
        const float selected = (label >= 0 && label < cols) ? xr[label] : 0.0f;
        loss[r] = (ot_logf(total) + peak) - selected;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Part 5: the unordered maximum and minimum                                 */
/* ------------------------------------------------------------------------- */
/*
 * "TIRx Metal reduction lowering" §8 lists minimum and maximum among the row
 * reductions and fixes only their reducers; the page leaves NaN undefined
 * (§3). The unordered policy's reading: a NaN element is skipped, so a vector
 * gives NaN only when every element is NaN; otherwise the result is the
 * largest (smallest) non-NaN value, infinities included. When the extreme is
 * a zero that occurs with both signs the sign is not fixed (either zero is a
 * correct result), and this definition returns the first one met. Written as
 * the plain serial scan: start from "nothing seen" (NaN) and replace it by
 * each non-NaN element that is larger (smaller).
 */
static float skipnan_extreme(const float *v, int64_t n, int64_t stride, int want_max) {
    float best = NAN;
    for (int64_t i = 0; i < n; ++i) {
        const float e = v[i * stride];
        if (isnan(e)) continue;
        if (isnan(best) || (want_max ? e > best : e < best)) best = e;
    }
    return best;
}

int skipnan_row_max_f32(const float *x, float *out, int64_t rows, int64_t cols) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) out[r] = skipnan_extreme(x + r * cols, cols, 1, 1);
    return 0;
}

int skipnan_row_min_f32(const float *x, float *out, int64_t rows, int64_t cols) {
    if (bad_sizes(rows, cols)) return -1;
    for (int64_t r = 0; r < rows; ++r) out[r] = skipnan_extreme(x + r * cols, cols, 1, 0);
    return 0;
}

/* The same over the middle axis of a contiguous [outer, extent, inner] array:
 * out[o * inner + i] is the extreme of x[o, :, i]. */
int skipnan_axis_max_f32(const float *x, float *out, int64_t outer, int64_t extent, int64_t inner) {
    if (outer < 0 || extent < 1 || inner < 1) return -1;
    for (int64_t o = 0; o < outer; ++o)
        for (int64_t i = 0; i < inner; ++i)
            out[o * inner + i] = skipnan_extreme(x + o * extent * inner + i, extent, inner, 1);
    return 0;
}

int skipnan_axis_min_f32(const float *x, float *out, int64_t outer, int64_t extent, int64_t inner) {
    if (outer < 0 || extent < 1 || inner < 1) return -1;
    for (int64_t o = 0; o < outer; ++o)
        for (int64_t i = 0; i < inner; ++i)
            out[o * inner + i] = skipnan_extreme(x + o * extent * inner + i, extent, inner, 0);
    return 0;
}
