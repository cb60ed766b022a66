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
 * the shift, closeness to the float64 two-pass value, TwoSum's exact error
 * (s + e = a + b), and s2 equal to the correctly rounded sum of the leaves on
 * integer slices where the carries are exact and a plain tree rounds.
 */
#include "oracle.h"
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* The kernel's pieces, for float (the pages' precision) and double (the
   same steps in the input dtype, "all in the input dtype"). */
#define DEFINE_VAR_PIECES(T, SFX)                                                \
static T tree_plain_##SFX(T* a, int64_t n) {                                     \
    /* in place, destroys a */                                                   \
    int64_t m = n;                                                               \
    while (m > 1) {                                                              \
        int64_t h = m / 2;                                                       \
        for (int64_t i = 0; i < h; ++i) a[i] = a[2 * i] + a[2 * i + 1];          \
        if (m & 1) a[h] = a[m - 1];                                              \
        m = h + (m & 1);                                                         \
    }                                                                            \
    return a[0];                                                                 \
}                                                                                \
                                                                                 \
static void two_sum_##SFX(T a, T b, T* s, T* e) {                                \
    T ss = a + b;                                                                \
    T bb = ss - a;                                                               \
    *e = (a - (ss - bb)) + (b - bb);                                             \
    *s = ss;                                                                     \
}                                                                                \
                                                                                 \
static T tree_twosum_##SFX(T* s, T* c, int64_t n) {                              \
    int64_t m = n;                                                               \
    while (m > 1) {                                                              \
        int64_t h = m / 2;                                                       \
        for (int64_t i = 0; i < h; ++i) {                                        \
            T sl = s[2 * i], sr = s[2 * i + 1];                                  \
            T cl = c[2 * i], cr = c[2 * i + 1];                                  \
            T sn, e;                                                             \
            two_sum_##SFX(sl, sr, &sn, &e);                                      \
            s[i] = sn;                                                           \
            c[i] = (cl + cr) + e;                                                \
        }                                                                        \
        if (m & 1) { s[h] = s[m - 1]; c[h] = c[m - 1]; }                         \
        m = h + (m & 1);                                                         \
    }                                                                            \
    return s[0] + c[0];                                                          \
}                                                                                \
                                                                                 \
/* Kahan's loop in index order ("Kahan's Summation Formula"). */                 \
static T kahan_seq_##SFX(const T* a, int64_t n) {                                \
    T s = 0, c = 0;                                                              \
    for (int64_t i = 0; i < n; ++i) {                                            \
        T y = a[i] - c;                                                          \
        T t = s + y;                                                             \
        c = (t - s) - y;                                                         \
        s = t;                                                                   \
    }                                                                            \
    return s;                                                                    \
}                                                                                \
                                                                                 \
static T max_nan_##SFX(T v) {                                                    \
    if (v != v) return v;                                                        \
    return v > (T)0 ? v : (T)0;                                                  \
}                                                                                \
                                                                                 \
static T rescale_##SFX(T v, int64_t n, int ddof) {                               \
    if (ddof == 0) return v;                                                     \
    T f = (T)n / (T)(n - ddof);                                                  \
    return v * f;                                                                \
}                                                                                \
                                                                                 \
/* The formula of reference (section 1: means as the tree sum times        */ \
/* RN(1/n), d = x - mean, two-term); variant 4 takes the TwoSum tree for    */ \
/* d^2 (comp), variant 1 the plain one.                                     */ \
static void ref_slice_##SFX(const T* x, int64_t n, int ddof, int comp, T* var,  \
                            T* mean) {                                           \
    T* d = (T*)malloc(sizeof(T) * (size_t)n);                                    \
    T* t = (T*)malloc(sizeof(T) * (size_t)n);                                    \
    T* c = (T*)malloc(sizeof(T) * (size_t)n);                                    \
    T inv = (T)1 / (T)n;                                                         \
    memcpy(t, x, sizeof(T) * (size_t)n);                                         \
    T m = tree_plain_##SFX(t, n) * inv;                                          \
    for (int64_t i = 0; i < n; ++i) d[i] = x[i] - m;                             \
    for (int64_t i = 0; i < n; ++i) { t[i] = d[i] * d[i]; c[i] = 0; }            \
    T s2 = comp ? tree_twosum_##SFX(t, c, n) : tree_plain_##SFX(t, n);            \
    memcpy(t, d, sizeof(T) * (size_t)n);                                         \
    T md = tree_plain_##SFX(t, n) * inv;                                         \
    T v = (s2 * inv) - (md * md);                                                \
    *var = rescale_##SFX(max_nan_##SFX(v), n, ddof);                             \
    if (mean) *mean = m;                                                         \
    free(d); free(t); free(c);                                                   \
}                                                                                \
                                                                                 \
/* One slice of the kernel or of one of its section 4 variants (the step    */ \
/* changes are listed at orc_var_variant_f32 in oracle.h).                  */ \
static void variant_slice_##SFX(const T* x, int64_t n, int ddof, int variant,  \
                                T* var, T* mean) {                               \
    if (n <= 0) { *var = 0; if (mean) *mean = 0; return; }                       \
    if (variant == 1 || variant == 4) {                                          \
        ref_slice_##SFX(x, n, ddof, variant == 4, var, mean);                    \
        return;                                                                  \
    }                                                                            \
    const int comp = (variant == 2 || variant == 3) ? 0 : (variant == 6 ? 2 : 1); \
    const int twoterm = !(variant == 2 || variant == 5);                         \
    T* d = (T*)malloc(sizeof(T) * (size_t)n);                                    \
    T* t = (T*)malloc(sizeof(T) * (size_t)n);                                    \
    T* sq = (T*)malloc(sizeof(T) * (size_t)n);                                   \
    T* c = (T*)malloc(sizeof(T) * (size_t)n);                                    \
    T nf = (T)n;                                                                 \
    T x0 = x[0], m = 0;                                                          \
    for (int64_t i = 0; i < n; ++i) d[i] = x[i] - x0;            /* step 1 */    \
    memcpy(t, d, sizeof(T) * (size_t)n);                                         \
    m = tree_plain_##SFX(t, n) / nf;                              /* step 2 */    \
    for (int64_t i = 0; i < n; ++i) d[i] = d[i] - m;                             \
    for (int64_t i = 0; i < n; ++i) { sq[i] = d[i] * d[i]; c[i] = 0; }           \
    T s2;                                                         /* step 3 */    \
    if (comp == 1) s2 = tree_twosum_##SFX(sq, c, n);                             \
    else if (comp == 0) s2 = tree_plain_##SFX(sq, n);                            \
    else s2 = kahan_seq_##SFX(sq, n);                                            \
    memcpy(t, d, sizeof(T) * (size_t)n);                                         \
    T s1 = tree_plain_##SFX(t, n);                                               \
    T tm = s1 / nf;                                               /* step 4 */    \
    T v = twoterm ? (s2 / nf) - (tm * tm) : (s2 / nf);                           \
    *var = rescale_##SFX(max_nan_##SFX(v), n, ddof);                             \
    if (mean) *mean = x0 + m;                                                    \
    free(d); free(t); free(sq); free(c);                                         \
}

DEFINE_VAR_PIECES(float, f)
DEFINE_VAR_PIECES(double, d)

/* The error-free transformation itself, exported so that it can be checked
   on its own: s = RN(a + b) and s + e = a + b exactly. */
void orc_two_sum_f32(float a, float b, float* s, float* e) { two_sum_f(a, b, s, e); }
void orc_two_sum_f64(double a, double b, double* s, double* e) { two_sum_d(a, b, s, e); }

static float tree_plain(float* a, int64_t n) { return tree_plain_f(a, n); }

static float max_nan(float v) { return max_nan_f(v); }

static float rescale(float v, int64_t n, int ddof) { return rescale_f(v, n, ddof); }

static void kernel_slice(const float* x, int64_t n, int ddof, float* var, float* mean) {
    variant_slice_f(x, n, ddof, 0, var, mean);
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

/* Section 4 ("Which step does what"): the kernel with steps changed. */
void orc_var_variant_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof, int variant,
                         float* var_out, float* mean_out) {
    int64_t ns = axis == 1 ? rows : cols, len = axis == 1 ? cols : rows;
    float* buf = (float*)malloc(sizeof(float) * (size_t)len);
    for (int64_t s = 0; s < ns; ++s) {
        gather(x, rows, cols, axis, s, buf);
        float mn;
        variant_slice_f(buf, len, ddof, variant, &var_out[s], &mn);
        if (mean_out) mean_out[s] = mn;
    }
    free(buf);
}

/* The kernel on float64 input, every step in float64. */
void orc_var_kernel_f64(const double* x, int64_t rows, int64_t cols, int axis, int ddof,
                        double* var_out, double* mean_out) {
    int64_t ns = axis == 1 ? rows : cols, len = axis == 1 ? cols : rows;
    double* buf = (double*)malloc(sizeof(double) * (size_t)len);
    for (int64_t s = 0; s < ns; ++s) {
        for (int64_t i = 0; i < len; ++i) buf[i] = axis == 1 ? x[s * cols + i] : x[i * cols + s];
        double mn;
        variant_slice_d(buf, len, ddof, 0, &var_out[s], &mn);
        if (mean_out) mean_out[s] = mn;
    }
    free(buf);
}

/* Complex64 [rows, cols] (interleaved re, im): per slice var(re) + var(im)
   by the float32 kernel; the mean is (mean(re), mean(im)). */
void orc_var_kernel_c64_2d(const float* z, int64_t rows, int64_t cols, int axis, int ddof,
                           float* var_out, float* mean_out) {
    int64_t ns = axis == 1 ? rows : cols, len = axis == 1 ? cols : rows;
    float* re = (float*)malloc(sizeof(float) * (size_t)len);
    float* im = (float*)malloc(sizeof(float) * (size_t)len);
    for (int64_t s = 0; s < ns; ++s) {
        for (int64_t i = 0; i < len; ++i) {
            int64_t e = axis == 1 ? s * cols + i : i * cols + s;
            re[i] = z[2 * e];
            im[i] = z[2 * e + 1];
        }
        float vr, vi, mr, mi;
        kernel_slice(re, len, ddof, &vr, &mr);
        kernel_slice(im, len, ddof, &vi, &mi);
        var_out[s] = vr + vi;
        if (mean_out) { mean_out[2 * s] = mr; mean_out[2 * s + 1] = mi; }
    }
    free(re);
    free(im);
}
