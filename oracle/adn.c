/*
 * Oracle: Ahrens-Demmel-Nguyen (ADN) binned summation, restated from the
 * "SyclReproSum".  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Geometry ("How It Works", "Template Parameters", "Accumulator capacity"):
 *   bin width W = 40 (double) / 13 (float); at most nb = 52 / 21 bins, which
 *   is also the largest fold count K; values below ~2^-1055 / ~2^-144 are
 *   absorbed.  Reading taken here: bin j (0 = coarsest) has grid unit
 *   g_j = 2^(b0 - W j) with b0 = 986 (double) / 117 (float), so the finest
 *   grid is 2^-1054 / 2^-143 and the absorption threshold is half of it.
 *   A value x belongs to the finest bin j with |x| < 2^(b0 - W j + W - 1).
 *
 * Parity pins (tests/test_oracle.py): the Quick Start example (1e16 pairs and
 * 10000 ones sum to exactly 10000 and the last prefix equals the sum), the
 * capacity constants, canonical NaN bits, the 10^6 x 0.001f example, equality
 * of the two forms below, brute-force permutation invariance, the closed-form
 * identity ADN = RN(exact) on grid-aligned inputs, the absolute error
 * bound of "Template Parameters", and the renormalisation period: runs of
 * several periods of the largest odd last-fold piece, checked against exact
 * rationals, fail with any longer period.
 */
#include "oracle.h"
#include "fixacc.h"
#include <math.h>
#include <string.h>
#include <stdlib.h>

typedef struct {
    int W;      /* bin width in bits */
    int nb;     /* number of bins == largest K */
    int b0;     /* exponent of the coarsest grid unit */
    int prec;   /* significand bits of the type */
} geom;

static const geom GD = {40, 52, 986, 53};
static const geom GF = {13, 21, 117, 24};

static int beta(const geom* g, int j) { return g->b0 - g->W * j; }

/* "Accumulator capacity": (2^(p-1) - 1) carries, one carry step per
   2^(p-W-2) deposits. */
static uint64_t max_count(const geom* g) {
    return (((uint64_t)1 << (g->prec - 1)) - 1) << (g->prec - g->W - 2);
}
uint64_t orc_max_count_f32(void) { return max_count(&GF); }
uint64_t orc_max_count_f64(void) { return max_count(&GD); }
int orc_max_k_f32(void) { return GF.nb; }
int orc_max_k_f64(void) { return GD.nb; }
int orc_bin_width_f32(void) { return GF.W; }
int orc_bin_width_f64(void) { return GD.W; }

/* floor(log2|x|) of a finite non-zero value, subnormals included. */
static int ilog2_abs(double ax) {
    int ex;
    frexp(ax, &ex);          /* ax = f * 2^ex, f in [0.5, 1) */
    return ex - 1;
}

/* Finest bin j with |x| < 2^(beta_j + W - 1). */
static int bin_index(const geom* g, double x) {
    int E = ilog2_abs(fabs(x));
    int j = (g->b0 + g->W - 2 - E) / g->W;   /* numerator is positive */
    if (j > g->nb - 1) j = g->nb - 1;
    if (j < 0) j = 0;
    return j;
}
int orc_bin_index_f64(double x) { return bin_index(&GD, x); }
int orc_bin_index_f32(float x) { return bin_index(&GF, (double)x); }

/* ------------------------------------------------------------------------
 * Special values ("How It Works"): any NaN, or +Inf together with -Inf, gives
 * the canonical quiet NaN; otherwise an Inf propagates.
 */
#define FL_NAN 1
#define FL_PINF 2
#define FL_NINF 4

static double special_f64(int flags) {
    if ((flags & FL_NAN) || ((flags & FL_PINF) && (flags & FL_NINF))) {
        uint64_t b = 0x7ff8000000000000ull;
        double r;
        memcpy(&r, &b, 8);
        return r;
    }
    return (flags & FL_PINF) ? INFINITY : -INFINITY;
}
static float special_f32(int flags) {
    if ((flags & FL_NAN) || ((flags & FL_PINF) && (flags & FL_NINF))) {
        uint32_t b = 0x7fc00000u;
        float r;
        memcpy(&r, &b, 4);
        return r;
    }
    return (flags & FL_PINF) ? INFINITY : -INFINITY;
}

static int classify(double x) {
    if (x != x) return FL_NAN;
    if (x == INFINITY) return FL_PINF;
    if (x == -INFINITY) return FL_NINF;
    return 0;
}

/* ------------------------------------------------------------------------
 * Closed form.  With I = min(index of max|x|, nb - K), each finite x is cut
 * into K pieces on the grids g_I .. g_{I+K-1}:
 *     r_0 = x;  piece_k = round_half_away(r_k / g_{I+k}) * g_{I+k};
 *     r_{k+1} = r_k - piece_k,
 * the last remainder being dropped ("How It Works", deposit of x: top W bits
 * to the coarsest fold, next W bits to the next, the rest to the last fold,
 * with the bin rounding made order-independent).  Fold sums are exact
 * integers; the result is the single correct rounding of their total.
 */

/* One value's K digits (piece_k / g_{I+k}), by exact integer arithmetic on a
   fixed-point copy of the running remainder. */
static void pieces(const geom* g, int I, int K, double x, int64_t* a) {
    for (int k = 0; k < K; ++k) a[k] = 0;
    int blast = beta(g, I + K - 1);
    /* |x| < g_last / 2: every rounding gives 0 and the remainder never moves. */
    if (fabs(x) < ldexp(1.0, blast - 1)) return;
    /* x = s * M * 2^e exactly. */
    int ex;
    double fr = frexp(fabs(x), &ex);             /* |x| = fr * 2^ex */
    uint64_t M = (uint64_t)ldexp(fr, 64 - 11);   /* 53 bits, exact */
    int e = ex - 53;
    while (M && !(M & 1)) { M >>= 1; ++e; }      /* canonical odd M */
    int neg = x < 0;
    int L = e < blast - 1 ? e : blast - 1;       /* unit of the fixed point */
    fixacc r;
    /* Width: bits from 2^L up to the top of bin I plus sign and margin. */
    int need = beta(g, I) + g->W + 2 - L;
    int nl = need / 64 + 2;
    if (nl > FIX_MAXL) nl = FIX_MAXL;
    fix_init(&r, nl, L);
    fix_add_u64(&r, M, e, neg);
    for (int k = 0; k < K; ++k) {
        int s = beta(g, I + k) - L;                 /* grid in units of 2^L, s >= 1 */
        int64_t q = fix_floor_shift(&r, s);         /* floor(r / g) */
        int halfbit = fix_bit(&r, s - 1);
        int below = fix_any_below(&r, s - 1);
        int64_t d = q;
        if (halfbit && below) d = q + 1;            /* remainder above half */
        else if (halfbit && !below)                 /* exact tie: away from zero */
            d = (fix_sign(&r) > 0) ? q + 1 : q;
        a[k] = d;
        if (d) fix_add_i128(&r, -(__int128)d, beta(g, I + k));
    }
}

typedef struct {
    int I;
    int flags;
    __int128 F[ORC_MAXK];
} cstate;

static void closed_state(const geom* g, const double* xd, const float* xf, int64_t n, int K,
                         cstate* st) {
    st->flags = 0;
    st->I = g->nb - K;
    for (int k = 0; k < K; ++k) st->F[k] = 0;
    for (int64_t i = 0; i < n; ++i) {
        double x = xd ? xd[i] : (double)xf[i];
        int c = classify(x);
        if (c) { st->flags |= c; continue; }
        if (x == 0.0) continue;
        int j = bin_index(g, x);
        if (j < st->I) st->I = j;
    }
    int64_t a[ORC_MAXK];
    for (int64_t i = 0; i < n; ++i) {
        double x = xd ? xd[i] : (double)xf[i];
        if (classify(x) || x == 0.0) continue;
        pieces(g, st->I, K, x, a);
        for (int k = 0; k < K; ++k) st->F[k] += a[k];
    }
}

static double state_value(const geom* g, const cstate* st, int K, int is_f32) {
    fixacc f;
    fix_init_default(&f);
    for (int k = 0; k < K; ++k) fix_add_i128(&f, st->F[k], beta(g, st->I + k));
    return is_f32 ? (double)fix_to_float(&f) : fix_to_double(&f);
}

double orc_adn_sum_closed_f64(const double* x, int64_t n, int K) {
    cstate st;
    closed_state(&GD, x, NULL, n, K, &st);
    if (st.flags) return special_f64(st.flags);
    return state_value(&GD, &st, K, 0);
}

float orc_adn_sum_closed_f32(const float* x, int64_t n, int K) {
    cstate st;
    closed_state(&GF, NULL, x, n, K, &st);
    if (st.flags) return special_f32(st.flags);
    return (float)state_value(&GF, &st, K, 1);
}

static void export_state(const cstate* st, int K, int* I, int64_t* F_hi, uint64_t* F_lo, int* flags) {
    *I = st->I;
    *flags = st->flags;
    for (int k = 0; k < K; ++k) {
        unsigned __int128 u = (unsigned __int128)st->F[k];
        F_lo[k] = (uint64_t)u;
        F_hi[k] = (int64_t)(uint64_t)(u >> 64);
    }
}

void orc_adn_state_closed_f64(const double* x, int64_t n, int K, int* I, int64_t* F_hi,
                              uint64_t* F_lo, int* flags) {
    cstate st;
    closed_state(&GD, x, NULL, n, K, &st);
    export_state(&st, K, I, F_hi, F_lo, flags);
}

void orc_adn_state_closed_f32(const float* x, int64_t n, int K, int* I, int64_t* F_hi,
                              uint64_t* F_lo, int* flags) {
    cstate st;
    closed_state(&GF, NULL, x, n, K, &st);
    export_state(&st, K, I, F_hi, F_lo, flags);
}

/* ------------------------------------------------------------------------
 * Floating-point primary form, one value at a time in input order, as the
 * "SyclReproSum" page's "How It Works" describes it:
 *  - each fold keeps a primary P whose ulp is the fold's grid unit, started
 *    at 1.5 * 2^e (ulp(P) = 2^(e - p + 1) = g), and a carry counter C;
 *  - Deposit: with the least significant bit of the remainder forced to 1
 *    (the sticky bit), S = P + sticky(r) rounds r on the fold's grid with
 *    ties away from zero; the remainder becomes r + (P - S), exactly;
 *  - Renormalize: every 2^(p - W - 2) deposits, the two bits below P's
 *    leading bit (q in 1..3) move into the carry, C += q - 2, and P is reset
 *    to [1.5, 1.75) * 2^e;
 *  - a value above the current bins raises the index: folds shift toward the
 *    finest, the finest ones fall off, fresh folds enter on top.
 * Fold value = (P - 1.5 * 2^e) + C * 2^(e-2).  The primary of bin 0 would
 * overflow (1.5 * 2^1038 / 1.5 * 2^140), so that fold alone is held scaled by
 * 2^-64; scaling by a power of two changes no rounding on its grid.
 */
#define SCALE0 64

#define DEFINE_FP_FORM(T, SFX, UT, GEO)                                                   \
typedef struct {                                                                         \
    int K, I, flags;                                                                     \
    T P[ORC_MAXK];                                                                       \
    int64_t C[ORC_MAXK];                                                                 \
    int sc[ORC_MAXK];   /* 2^-sc scaling of fold k's primary */                           \
    int64_t since;                                                                       \
} fpstate_##SFX;                                                                         \
                                                                                         \
static T sticky_##SFX(T r) {                                                             \
    UT b;                                                                                \
    memcpy(&b, &r, sizeof b);                                                            \
    b |= 1;                                                                              \
    memcpy(&r, &b, sizeof b);                                                            \
    return r;                                                                            \
}                                                                                        \
                                                                                         \
/* exponent e of the primary's binade for bin j */                                       \
static int pexp_##SFX(int j, int sc) { return beta(&GEO, j) + GEO.prec - 1 - sc; }       \
                                                                                         \
static void fresh_##SFX(fpstate_##SFX* s, int k) {                                       \
    int j = s->I + k;                                                                    \
    s->sc[k] = (j == 0) ? SCALE0 : 0;                                                    \
    s->P[k] = (T)ldexp(1.5, pexp_##SFX(j, s->sc[k]));                                    \
    s->C[k] = 0;                                                                         \
}                                                                                        \
                                                                                         \
static void fp_init_##SFX(fpstate_##SFX* s, int K) {                                     \
    s->K = K;                                                                            \
    s->I = GEO.nb - K;                                                                   \
    s->flags = 0;                                                                        \
    s->since = 0;                                                                        \
    for (int k = 0; k < K; ++k) fresh_##SFX(s, k);                                       \
}                                                                                        \
                                                                                         \
static void renorm_##SFX(fpstate_##SFX* s) {                                             \
    for (int k = 0; k < s->K; ++k) {                                                     \
        int e = pexp_##SFX(s->I + k, s->sc[k]);                                          \
        T lead = (T)ldexp(1.0, e);                                                       \
        T quarter = (T)ldexp(1.0, e - 2);                                                \
        int q = (int)floor((double)((s->P[k] - lead) / quarter));                        \
        s->C[k] += q - 2;                                                                \
        s->P[k] = s->P[k] - (T)(q - 2) * quarter;                                        \
    }                                                                                    \
}                                                                                        \
                                                                                         \
static void raise_##SFX(fpstate_##SFX* s, int j) {                                       \
    int d = s->I - j;                                                                    \
    for (int k = s->K - 1; k >= 0; --k) {                                                \
        if (k >= d) {                                                                    \
            s->P[k] = s->P[k - d];                                                       \
            s->C[k] = s->C[k - d];                                                       \
            s->sc[k] = s->sc[k - d];                                                     \
        }                                                                                \
    }                                                                                    \
    s->I = j;                                                                            \
    for (int k = 0; k < d && k < s->K; ++k) fresh_##SFX(s, k);                           \
}                                                                                        \
                                                                                         \
static void deposit_##SFX(fpstate_##SFX* s, T x) {                                       \
    int c = classify((double)x);                                                         \
    if (c) { s->flags |= c; return; }                                                    \
    if (x == 0) return;                                                                  \
    int j = bin_index(&GEO, (double)x);                                                  \
    if (j < s->I) raise_##SFX(s, j);                                                     \
    T r = x;                                                                             \
    for (int k = 0; k < s->K; ++k) {                                                     \
        T rs = s->sc[k] ? (T)ldexp((double)r, -s->sc[k]) : r;                            \
        T S = s->P[k] + sticky_##SFX(rs);                                                \
        if (k < s->K - 1) {                                                              \
            T d = s->P[k] - S;                                                           \
            r = r + (s->sc[k] ? (T)ldexp((double)d, s->sc[k]) : d);                      \
        }                                                                                \
        s->P[k] = S;                                                                     \
    }                                                                                    \
    if (++s->since == ((int64_t)1 << (GEO.prec - GEO.W - 2))) {                          \
        renorm_##SFX(s);                                                                 \
        s->since = 0;                                                                    \
    }                                                                                    \
}                                                                                        \
                                                                                         \
/* Fold value in units of the fold's grid: exact integer. */                            \
static __int128 fold_##SFX(const fpstate_##SFX* s, int k) {                              \
    int e = pexp_##SFX(s->I + k, s->sc[k]);                                              \
    T base = (T)ldexp(1.5, e);                                                           \
    double dev = ldexp((double)(s->P[k] - base), GEO.prec - 1 - e);                      \
    return (__int128)(int64_t)dev + (__int128)s->C[k] * ((__int128)1 << (GEO.prec - 3)); \
}                                                                                        \
                                                                                         \
static double fp_value_##SFX(const fpstate_##SFX* s, int is_f32) {                      \
    fixacc f;                                                                            \
    fix_init_default(&f);                                                                \
    for (int k = 0; k < s->K; ++k) fix_add_i128(&f, fold_##SFX(s, k), beta(&GEO, s->I + k)); \
    return is_f32 ? (double)fix_to_float(&f) : fix_to_double(&f);                        \
}

DEFINE_FP_FORM(double, d, uint64_t, GD)
DEFINE_FP_FORM(float, f, uint32_t, GF)

double orc_adn_sum_fp_f64(const double* x, int64_t n, int K) {
    fpstate_d s;
    fp_init_d(&s, K);
    for (int64_t i = 0; i < n; ++i) deposit_d(&s, x[i]);
    if (s.flags) return special_f64(s.flags);
    return fp_value_d(&s, 0);
}

float orc_adn_sum_fp_f32(const float* x, int64_t n, int K) {
    fpstate_f s;
    fp_init_f(&s, K);
    for (int64_t i = 0; i < n; ++i) deposit_f(&s, x[i]);
    if (s.flags) return special_f32(s.flags);
    return (float)fp_value_f(&s, 1);
}

/* ------------------------------------------------------------------------
 * Cumulative sums ("How It Works", cumsum paragraph; "API Reference"):
 * out[i] is the reproducible sum of x[0] .. x[i], so each prefix carries its
 * own index and the last output equals the full sum.
 */
void orc_adn_cumsum_f64(const double* x, double* out, int64_t n, int K) {
    fpstate_d s;
    fp_init_d(&s, K);
    for (int64_t i = 0; i < n; ++i) {
        deposit_d(&s, x[i]);
        out[i] = s.flags ? special_f64(s.flags) : fp_value_d(&s, 0);
    }
}

void orc_adn_cumsum_f32(const float* x, float* out, int64_t n, int K) {
    fpstate_f s;
    fp_init_f(&s, K);
    for (int64_t i = 0; i < n; ++i) {
        deposit_f(&s, x[i]);
        out[i] = s.flags ? special_f32(s.flags) : (float)fp_value_f(&s, 1);
    }
}

void orc_adn_cumsum_at_f64(const double* x, int64_t n, int K, const int64_t* pos, int64_t m,
                           double* out) {
    fpstate_d s;
    fp_init_d(&s, K);
    int64_t p = 0;
    for (int64_t i = 0; i < n && p < m; ++i) {
        deposit_d(&s, x[i]);
        while (p < m && pos[p] == i) {
            out[p] = s.flags ? special_f64(s.flags) : fp_value_d(&s, 0);
            ++p;
        }
    }
}

void orc_adn_cumsum_at_f32(const float* x, int64_t n, int K, const int64_t* pos, int64_t m,
                           float* out) {
    fpstate_f s;
    fp_init_f(&s, K);
    int64_t p = 0;
    for (int64_t i = 0; i < n && p < m; ++i) {
        deposit_f(&s, x[i]);
        while (p < m && pos[p] == i) {
            out[p] = s.flags ? special_f32(s.flags) : (float)fp_value_f(&s, 1);
            ++p;
        }
    }
}

/* ------------------------------------------------------------------------
 * Segmented sums: one ADN sum per slice of a row-major [rows, cols] array.
 */
void orc_segsum_f32(const float* x, int64_t rows, int64_t cols, int axis, int K, float* out) {
    int64_t ns = axis == 1 ? rows : cols, len = axis == 1 ? cols : rows;
    float* buf = (float*)malloc(sizeof(float) * (size_t)(len > 0 ? len : 1));
    for (int64_t s = 0; s < ns; ++s) {
        for (int64_t i = 0; i < len; ++i)
            buf[i] = axis == 1 ? x[s * cols + i] : x[i * cols + s];
        out[s] = orc_adn_sum_closed_f32(buf, len, K);
    }
    free(buf);
}
