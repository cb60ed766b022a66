/*
 * Oracle: float32 variance.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Source: "Variance in float32 with a first-element shift, a local centring
 * and a compensated tree sum", section 2 ("The kernel"), all steps in
 * float32 with round-to-nearest:
 *   1. shift:      y_i = x_i - x_0
 *   2. centring:   m = sum(y) / n;  d_i = y_i - m
 *   3. compensated tree over d_i^2: each level adds pairs with TwoSum, the
 *      rounding errors are carried up in a second array, the result is the
 *      final sum plus the final carry (s2); s1 = sum(d)
 *   4. two-term:   var = max(s2/n - (s1/n)^2, 0), rescaled by n/(n - ddof);
 *      mean = x_0 + m.
 * Readings taken (the note leaves these open):
 *   - tree topology: adjacent pairs (2i, 2i+1) per level, an unpaired last
 *     node passed up unchanged; the same tree for sum(y) and sum(d);
 *   - carry combine at a node: c = (c_left + c_right) + e;
 *   - "/n" is an IEEE division; (s1/n)^2 is one rounded product;
 *   - max(., 0) propagates NaN; the rescale multiplies by RN(n / (n - ddof))
 *     and is skipped for ddof = 0.
 * TwoSum is the six-operation error-free sum (Knuth; Ogita-Rump-Oishi
 * Algorithm 3.1 as the note cites it): s = a + b, bb = s - a,
 * e = (a - (s - bb)) + (b - bb).
 *
 * The formula of reference (section 1, tf.nn.moments) and the naive formula
 * use mean(v) = RN(RN(sum v) * RN(1/n)): that reading is pinned by the
 * identical-value table of section 3 (naive 1.04858e+06, 6.71089e+07,
 * 4.5036e+15, inf; reference 0, 0, 0, nan), which true division does not
 * reproduce.  The float64 two-pass variance is the accuracy reference, as the
 * note's numpy.var in float64 is.
 *
 * Pins: identical values give exactly 0.0 (kernel), the section 3 table
 * (reference and naive), the complex check 6.421875, Sterbenz exactness of
 * the shift, and closeness to the float64 two-pass value.
 */
#include "oracle.h"
#include <math.h>
#include <stdlib.h>
#include <string.h>

static float tree_plain(float* a, int64_t n) {
    /* in place, destroys a */
    int64_t m = n;
    while (m > 1) {
        int64_t h = m / 2;
        for (int64_t i = 0; i < h; ++i) a[i] = a[2 * i] + a[2 * i + 1];
        if (m & 1) a[h] = a[m - 1];
        m = h + (m & 1);
    }
    return a[0];
}

static void two_sum(float a, float b, float* s, float* e) {
    float ss = a + b;
    float bb = ss - a;
    *e = (a - (ss - bb)) + (b - bb);
    *s = ss;
}

static float tree_twosum(float* s, float* c, int64_t n) {
    int64_t m = n;
    while (m > 1) {
        int64_t h = m / 2;
        for (int64_t i = 0; i < h; ++i) {
            float sl = s[2 * i], sr = s[2 * i + 1];
            float cl = c[2 * i], cr = c[2 * i + 1];
            float sn, e;
            two_sum(sl, sr, &sn, &e);
            s[i] = sn;
            c[i] = (cl + cr) + e;
        }
        if (m & 1) { s[h] = s[m - 1]; c[h] = c[m - 1]; }
        m = h + (m & 1);
    }
    return s[0] + c[0];
}

static float max_nan(float v) {
    if (v != v) return v;
    return v > 0.0f ? v : 0.0f;
}

static float rescale(float v, int64_t n, int ddof) {
    if (ddof == 0) return v;
    float f = (float)n / (float)(n - ddof);
    return v * f;
}

static void kernel_slice(const float* x, int64_t n, int ddof, float* var, float* mean) {
    if (n <= 0) { *var = 0.0f; if (mean) *mean = 0.0f; return; }
    float* y = (float*)malloc(sizeof(float) * (size_t)n);
    float* t = (float*)malloc(sizeof(float) * (size_t)n);
    float* s = (float*)malloc(sizeof(float) * (size_t)n);
    float* c = (float*)malloc(sizeof(float) * (size_t)n);
    float x0 = x[0];
    for (int64_t i = 0; i < n; ++i) y[i] = x[i] - x0;           /* step 1 */
    memcpy(t, y, sizeof(float) * (size_t)n);
    float nf = (float)n;
    float m = tree_plain(t, n) / nf;                             /* step 2 */
    for (int64_t i = 0; i < n; ++i) y[i] = y[i] - m;             /* y now holds d */
    for (int64_t i = 0; i < n; ++i) { s[i] = y[i] * y[i]; c[i] = 0.0f; }
    float s2 = tree_twosum(s, c, n);                             /* step 3 */
    float s1 = tree_plain(y, n);
    float tm = s1 / nf;                                          /* step 4 */
    float v = (s2 / nf) - (tm * tm);
    *var = rescale(max_nan(v), n, ddof);
    if (mean) *mean = x0 + m;
    free(y); free(t); free(s); free(c);
}

static float mean_recip(const float* v, int64_t n, float* work) {
    memcpy(work, v, sizeof(float) * (size_t)n);
    float inv = 1.0f / (float)n;
    return tree_plain(work, n) * inv;
}

static void twoterm_slice(const float* x, int64_t n, int ddof, float* var) {
    float* d = (float*)malloc(sizeof(float) * (size_t)n);
    float* d2 = (float*)malloc(sizeof(float) * (size_t)n);
    float* w = (float*)malloc(sizeof(float) * (size_t)n);
    float m = mean_recip(x, n, w);
    for (int64_t i = 0; i < n; ++i) { d[i] = x[i] - m; d2[i] = d[i] * d[i]; }
    float md = mean_recip(d, n, w);
    float v = mean_recip(d2, n, w) - (md * md);
    *var = rescale(max_nan(v), n, ddof);
    free(d); free(d2); free(w);
}

static void naive_slice(const float* x, int64_t n, int ddof, float* var) {
    float* d2 = (float*)malloc(sizeof(float) * (size_t)n);
    float* w = (float*)malloc(sizeof(float) * (size_t)n);
    float m = mean_recip(x, n, w);
    for (int64_t i = 0; i < n; ++i) { float d = x[i] - m; d2[i] = d * d; }
    *var = rescale(mean_recip(d2, n, w), n, ddof);
    free(d2); free(w);
}

static void f64_slice(const float* x, int64_t n, int ddof, double* var, double* mean) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += (double)x[i];
    double m = s / (double)n;
    double q = 0.0;
    for (int64_t i = 0; i < n; ++i) { double d = (double)x[i] - m; q += d * d; }
    *var = q / (double)(n - ddof);
    if (mean) *mean = m;
}

/* Gather slice s of a row-major [rows, cols] array into buf. */
static int64_t gather(const float* x, int64_t rows, int64_t cols, int axis, int64_t s, float* buf) {
    int64_t len = axis == 1 ? cols : rows;
    for (int64_t i = 0; i < len; ++i) buf[i] = axis == 1 ? x[s * cols + i] : x[i * cols + s];
    return len;
}

void orc_var_kernel_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof,
                        float* var_out, float* mean_out) {
    int64_t ns = axis == 1 ? rows : cols, len = axis == 1 ? cols : rows;
    float* buf = (float*)malloc(sizeof(float) * (size_t)len);
    for (int64_t s = 0; s < ns; ++s) {
        gather(x, rows, cols, axis, s, buf);
        float mn;
        kernel_slice(buf, len, ddof, &var_out[s], &mn);
        if (mean_out) mean_out[s] = mn;
    }
    free(buf);
}

void orc_var_twoterm_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof,
                         float* var_out) {
    int64_t ns = axis == 1 ? rows : cols, len = axis == 1 ? cols : rows;
    float* buf = (float*)malloc(sizeof(float) * (size_t)len);
    for (int64_t s = 0; s < ns; ++s) {
        gather(x, rows, cols, axis, s, buf);
        twoterm_slice(buf, len, ddof, &var_out[s]);
    }
    free(buf);
}

void orc_var_naive_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof,
                       float* var_out) {
    int64_t ns = axis == 1 ? rows : cols, len = axis == 1 ? cols : rows;
    float* buf = (float*)malloc(sizeof(float) * (size_t)len);
    for (int64_t s = 0; s < ns; ++s) {
        gather(x, rows, cols, axis, s, buf);
        naive_slice(buf, len, ddof, &var_out[s]);
    }
    free(buf);
}

void orc_var_f64(const float* x, int64_t rows, int64_t cols, int axis, int ddof,
                 double* var_out, double* mean_out) {
    int64_t ns = axis == 1 ? rows : cols, len = axis == 1 ? cols : rows;
    float* buf = (float*)malloc(sizeof(float) * (size_t)len);
    for (int64_t s = 0; s < ns; ++s) {
        gather(x, rows, cols, axis, s, buf);
        double mn;
        f64_slice(buf, len, ddof, &var_out[s], &mn);
        if (mean_out) mean_out[s] = mn;
    }
    free(buf);
}

/* Section 2, last paragraph: a complex input is split into real and imaginary
   parts and the two variances are added. */
void orc_var_kernel_c64(const float* re, const float* im, int64_t n, int ddof, float* var_out) {
    float vr, vi, mr, mi;
    kernel_slice(re, n, ddof, &vr, &mr);
    kernel_slice(im, n, ddof, &vi, &mi);
    *var_out = vr + vi;
}
