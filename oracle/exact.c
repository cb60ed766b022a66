/*
 * Oracle: exact sums.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 * The exact sum of the inputs is the reference every binned result is held
 * to ("SyclReproSum", "Template Parameters": the binned error term is
 * an absolute error against it).
 */
#include "oracle.h"
#include "fixacc.h"
#include <string.h>

static int exact_d(const double* x, int64_t n, fixacc* f) {
    fix_init_default(f);
    for (int64_t i = 0; i < n; ++i) {
        double v = x[i];
        if (v != v || v == 1.0 / 0.0 || v == -1.0 / 0.0) return 1;
        fix_add_double(f, v);
    }
    return 0;
}

static int exact_f(const float* x, int64_t n, fixacc* f) {
    fix_init_default(f);
    for (int64_t i = 0; i < n; ++i) {
        float v = x[i];
        if (v != v || v == 1.0f / 0.0f || v == -1.0f / 0.0f) return 1;
        fix_add_float(f, v);
    }
    return 0;
}

int orc_exact_sum_f64(const double* x, int64_t n, double* out) {
    fixacc f;
    if (exact_d(x, n, &f)) return 1;
    *out = fix_to_double(&f);
    return 0;
}

int orc_exact_sum_f32(const float* x, int64_t n, float* out) {
    fixacc f;
    if (exact_f(x, n, &f)) return 1;
    *out = fix_to_float(&f);
    return 0;
}

static int export_limbs(const fixacc* f, uint64_t* limbs, int max_limbs, int* lsb) {
    int n = f->nl < max_limbs ? f->nl : max_limbs;
    memcpy(limbs, f->limb, sizeof(uint64_t) * (size_t)n);
    *lsb = f->lsb;
    return n;
}

int orc_exact_sum_limbs_f64(const double* x, int64_t n, uint64_t* limbs, int max_limbs, int* lsb) {
    fixacc f;
    if (exact_d(x, n, &f)) return 0;
    return export_limbs(&f, limbs, max_limbs, lsb);
}

int orc_exact_sum_limbs_f32(const float* x, int64_t n, uint64_t* limbs, int max_limbs, int* lsb) {
    fixacc f;
    if (exact_f(x, n, &f)) return 0;
    return export_limbs(&f, limbs, max_limbs, lsb);
}
