/*
 * Oracle-internal: exact two's-complement fixed-point integers
 * ("superaccumulator") and correct rounding to binary32/binary64.
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 */
#ifndef REPRO_ORACLE_FIXACC_H
#define REPRO_ORACLE_FIXACC_H
#include <stdint.h>

/* value = sum_{i < nl} limb[i] * 2^(64 i + lsb), two's complement over nl limbs.
   The default accumulator spans 2^-1088 .. 2^1215, which holds every finite
   binary64 value and any sum of up to 2^63 of them exactly. */
#define FIX_MAXL 40
#define FIX_LSB_DEFAULT (-1088)
#define FIX_NL_DEFAULT 36

typedef struct {
    int nl;
    int lsb;
    uint64_t limb[FIX_MAXL];
} fixacc;

void fix_init(fixacc* f, int nl, int lsb);
void fix_init_default(fixacc* f);
/* f += (neg ? -1 : 1) * m * 2^e, requires e >= f->lsb. */
void fix_add_u64(fixacc* f, uint64_t m, int e, int neg);
/* f += v * 2^e for a signed 128-bit v, requires e >= f->lsb. */
void fix_add_i128(fixacc* f, __int128 v, int e);
void fix_add_double(fixacc* f, double x);   /* finite x only */
void fix_add_float(fixacc* f, float x);     /* finite x only */
int  fix_sign(const fixacc* f);             /* -1, 0, +1 */
int  fix_bit(const fixacc* f, int pos);     /* bit at absolute index pos (0..64 nl) */
/* Round to nearest, ties to even, with `prec` significand bits, smallest
   quantum 2^qmin and overflow at 2^emax; returns the rounded value as a
   double (exactly representable), +0.0 for an exact zero, +-Inf on overflow. */
double fix_round(const fixacc* f, int prec, int qmin, int emax);
double fix_to_double(const fixacc* f);
float  fix_to_float(const fixacc* f);
/* floor(f / 2^s) for an f whose quotient fits in int64 (s counted from bit 0). */
int64_t fix_floor_shift(const fixacc* f, int s);
/* 1 if any bit strictly below absolute bit index s is set. */
int fix_any_below(const fixacc* f, int s);

#endif
