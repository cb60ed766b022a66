/*
 * Oracle-internal exact fixed-point arithmetic and correct rounding.
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * The exact sum is the plain definition every binned result is measured
 * against ("SyclReproSum", "How It Works": the binned error term is an
 * absolute error against the exact sum).  Rounding follows IEEE 754
 * round-to-nearest-even, including subnormal results and overflow to Inf.
 */
#include "fixacc.h"
#include <string.h>
#include <math.h>

void fix_init(fixacc* f, int nl, int lsb) {
    memset(f, 0, sizeof(*f));
    f->nl = nl;
    f->lsb = lsb;
}

void fix_init_default(fixacc* f) { fix_init(f, FIX_NL_DEFAULT, FIX_LSB_DEFAULT); }

void fix_add_i128(fixacc* f, __int128 v, int e) {
    if (v == 0) return;
    int off = e - f->lsb;               /* bit offset of v's bit 0 */
    int li = off / 64, sh = off % 64;
    /* Spread the 128-bit two's complement value over three limbs after the
       shift, plus sign extension above. */
    unsigned __int128 u = (unsigned __int128)v;
    uint64_t w0 = (uint64_t)u, w1 = (uint64_t)(u >> 64);
    uint64_t ext = (v < 0) ? ~(uint64_t)0 : 0;
    uint64_t c0, c1, c2;
    if (sh == 0) {
        c0 = w0; c1 = w1; c2 = ext;
    } else {
        c0 = w0 << sh;
        c1 = (w1 << sh) | (w0 >> (64 - sh));
        c2 = (ext << sh) | (w1 >> (64 - sh));
    }
    /* Add c0, c1, c2 at limbs li, li+1, li+2 and ext above as one multi-limb
       addition. */
    unsigned carry = 0;
    for (int j = li; j < f->nl; ++j) {
        uint64_t add = (j == li) ? c0 : (j == li + 1) ? c1 : (j == li + 2) ? c2 : ext;
        uint64_t s = f->limb[j] + add;
        unsigned k1 = s < add;
        uint64_t s2 = s + carry;
        unsigned k2 = s2 < s;
        f->limb[j] = s2;
        carry = k1 | k2;
        /* Above the value's own limbs only sign extension is added: with a
           zero extension and no carry, or an all-ones extension and a carry,
           the remaining limbs are unchanged. */
        if (j > li + 2 && ((ext == 0 && carry == 0) || (ext != 0 && carry == 1))) break;
    }
}

void fix_add_u64(fixacc* f, uint64_t m, int e, int neg) {
    if (m == 0) return;
    __int128 v = (__int128)m;
    fix_add_i128(f, neg ? -v : v, e);
}

void fix_add_double(fixacc* f, double x) {
    if (x == 0.0) return;
    uint64_t b;
    memcpy(&b, &x, 8);
    int neg = (int)(b >> 63);
    int be = (int)((b >> 52) & 0x7FF);
    uint64_t mant = b & ((1ull << 52) - 1);
    uint64_t M;
    int e;
    if (be == 0) { M = mant; e = -1074; }
    else { M = mant | (1ull << 52); e = be - 1075; }
    fix_add_u64(f, M, e, neg);
}

void fix_add_float(fixacc* f, float x) {
    if (x == 0.0f) return;
    uint32_t b;
    memcpy(&b, &x, 4);
    int neg = (int)(b >> 31);
    int be = (int)((b >> 23) & 0xFF);
    uint64_t mant = b & ((1u << 23) - 1);
    uint64_t M;
    int e;
    if (be == 0) { M = mant; e = -149; }
    else { M = mant | (1u << 23); e = be - 150; }
    fix_add_u64(f, M, e, neg);
}

int fix_sign(const fixacc* f) {
    if (f->limb[f->nl - 1] >> 63) return -1;
    for (int i = 0; i < f->nl; ++i)
        if (f->limb[i]) return 1;
    return 0;
}

int fix_bit(const fixacc* f, int pos) {
    if (pos < 0) return 0;
    if (pos >= 64 * f->nl) return (int)(f->limb[f->nl - 1] >> 63);
    return (int)((f->limb[pos / 64] >> (pos % 64)) & 1u);
}

int fix_any_below(const fixacc* f, int s) {
    if (s <= 0) return 0;
    int full = s / 64, rem = s % 64;
    for (int i = 0; i < full && i < f->nl; ++i)
        if (f->limb[i]) return 1;
    if (rem && full < f->nl && (f->limb[full] & ((1ull << rem) - 1))) return 1;
    return 0;
}

int64_t fix_floor_shift(const fixacc* f, int s) {
    /* Arithmetic shift right by s, keeping the low 64 bits of the result
       (the caller guarantees the quotient fits). */
    uint64_t ext = (f->limb[f->nl - 1] >> 63) ? ~(uint64_t)0 : 0;
    int li = s / 64, sh = s % 64;
    uint64_t lo = (li < f->nl) ? f->limb[li] : ext;
    uint64_t hi = (li + 1 < f->nl) ? f->limb[li + 1] : ext;
    uint64_t r = sh ? ((lo >> sh) | (hi << (64 - sh))) : lo;
    return (int64_t)r;
}

static void negate(fixacc* g) {
    unsigned carry = 1;
    for (int i = 0; i < g->nl; ++i) {
        uint64_t v = ~g->limb[i];
        uint64_t s = v + carry;
        carry = (s < v);
        g->limb[i] = s;
    }
}

double fix_round(const fixacc* f, int prec, int qmin, int emax) {
    fixacc g = *f;
    int neg = 0;
    if (fix_sign(&g) < 0) { neg = 1; negate(&g); }
    int top = -1;
    for (int i = g.nl - 1; i >= 0; --i) {
        if (g.limb[i]) { top = 64 * i + 63 - __builtin_clzll(g.limb[i]); break; }
    }
    if (top < 0) return 0.0;               /* exact zero -> +0.0 */
    int E = top + g.lsb;                   /* exponent of the leading bit */
    int q = E - prec + 1;                  /* quantum exponent */
    if (q < qmin) q = qmin;
    int qs = q - g.lsb;                    /* bit index of the quantum */
    uint64_t m = 0;
    for (int b = top; b >= qs; --b)
        m = (m << 1) | (uint64_t)fix_bit(&g, b);
    int half = fix_bit(&g, qs - 1);
    int sticky = fix_any_below(&g, qs - 1);
    if (half && (sticky || (m & 1))) m += 1;
    if (m == (1ull << prec)) { m >>= 1; q += 1; }
    if (m != 0 && (63 - __builtin_clzll(m)) + q >= emax) return neg ? -INFINITY : INFINITY;
    double r = ldexp((double)m, q);
    return neg ? -r : r;
}

double fix_to_double(const fixacc* f) { return fix_round(f, 53, -1074, 1024); }
float fix_to_float(const fixacc* f) { return (float)fix_round(f, 24, -149, 128); }
