/*
 * Oracle: comparison summation modes.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 *  - sequential sum: one accumulator, inputs in order ("Reduction order and
 *    compensation solve related but different problems", first paragraph;
 *    the naive loop of "Kahan's Summation Formula");
 *  - pairwise sum: a balanced tree.  Reading taken: adjacent pairs (2i, 2i+1)
 *    at every level, an unpaired last node passed up unchanged;
 *  - Kahan sum: y = x - c; t = s + y; c = (t - s) - y; s = t (the loop of
 *    "Kahan's Summation Formula", same as the variant described on the
 *    reductions page);
 *  - Neumaier sum: the magnitude comparison of the running sum and the term
 *    picks which of the two loses low-order bits; the accumulated correction
 *    is added at the end (reductions page, Neumaier paragraph).  Reading
 *    taken: the correction is held in the input type.
 *
 * Pins: the printed results of "Kahan's Summation Formula" (naive 991.14154,
 * Kahan 1000.00006 for 10^6 additions of 0.001f); exactness on integer data;
 * tree sum of a power-of-two run equals the sum of its two halves' trees.
 * The chunked variants exist to give a deterministic target for the GPU
 * comparison kernels; their chunking is this library's choice (parity
 * unpinned beyond the reductions of which they are made).
 */
#include "oracle.h"
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define DEFINE_SUMS(T, SFX)                                                      \
T orc_sum_naive_##SFX(const T* x, int64_t n) {                                   \
    T s = 0;                                                                     \
    for (int64_t i = 0; i < n; ++i) s = s + x[i];                                \
    return s;                                                                    \
}                                                                                \
                                                                                 \
T orc_sum_pairwise_##SFX(const T* x, int64_t n) {                                \
    if (n <= 0) return (T)0;                                                     \
    T* a = (T*)malloc(sizeof(T) * (size_t)n);                                    \
    memcpy(a, x, sizeof(T) * (size_t)n);                                         \
    int64_t m = n;                                                               \
    while (m > 1) {                                                              \
        int64_t h = m / 2;                                                       \
        for (int64_t i = 0; i < h; ++i) a[i] = a[2 * i] + a[2 * i + 1];          \
        if (m & 1) a[h] = a[m - 1];                                              \
        m = h + (m & 1);                                                         \
    }                                                                            \
    T r = a[0];                                                                  \
    free(a);                                                                     \
    return r;                                                                    \
}                                                                                \
                                                                                 \
T orc_sum_kahan_##SFX(const T* x, int64_t n) {                                   \
    T s = 0, c = 0;                                                              \
    for (int64_t i = 0; i < n; ++i) {                                            \
        T y = x[i] - c;                                                          \
        T t = s + y;                                                             \
        c = (t - s) - y;                                                         \
        s = t;                                                                   \
    }                                                                            \
    return s;                                                                    \
}                                                                                \
                                                                                 \
static T neumaier_run_##SFX(const T* x, int64_t n) {                             \
    T s = 0, c = 0;                                                              \
    for (int64_t i = 0; i < n; ++i) {                                            \
        T t = s + x[i];                                                          \
        if (fabs((double)s) >= fabs((double)x[i])) c = c + ((s - t) + x[i]);     \
        else c = c + ((x[i] - t) + s);                                           \
        s = t;                                                                   \
    }                                                                            \
    return s + c;                                                                \
}                                                                                \
                                                                                 \
T orc_sum_neumaier_##SFX(const T* x, int64_t n) { return neumaier_run_##SFX(x, n); } \
                                                                                 \
T orc_sum_kahan_chunked_##SFX(const T* x, int64_t n, int64_t chunk) {            \
    if (n <= 0) return (T)0;                                                     \
    int64_t nc = (n + chunk - 1) / chunk;                                        \
    T* p = (T*)malloc(sizeof(T) * (size_t)nc);                                   \
    for (int64_t c = 0; c < nc; ++c) {                                           \
        int64_t b = c * chunk, e = b + chunk < n ? b + chunk : n;                \
        p[c] = orc_sum_kahan_##SFX(x + b, e - b);                                \
    }                                                                            \
    T r = orc_sum_pairwise_##SFX(p, nc);                                         \
    free(p);                                                                     \
    return r;                                                                    \
}                                                                                \
                                                                                 \
T orc_sum_neumaier_chunked_##SFX(const T* x, int64_t n, int64_t chunk) {         \
    if (n <= 0) return (T)0;                                                     \
    int64_t nc = (n + chunk - 1) / chunk;                                        \
    T* p = (T*)malloc(sizeof(T) * (size_t)nc);                                   \
    for (int64_t c = 0; c < nc; ++c) {                                           \
        int64_t b = c * chunk, e = b + chunk < n ? b + chunk : n;                \
        p[c] = neumaier_run_##SFX(x + b, e - b);                                 \
    }                                                                            \
    T r = orc_sum_pairwise_##SFX(p, nc);                                         \
    free(p);                                                                     \
    return r;                                                                    \
}

DEFINE_SUMS(double, f64)
DEFINE_SUMS(float, f32)
