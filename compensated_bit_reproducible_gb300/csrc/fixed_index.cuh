// Binned sums at an index fixed before the deposit: device helpers shared
// by the double sum and the K = 3 cumulative sums.
//
// The binned result is a function of the multiset alone: it is the correct
// rounding of sum_i C_I(x_i), where I is the bin index of max|x| (capped at
// nb - K) and C_I(x) is x after the chained round-half-away decomposition on
// the grids g_I .. g_{I+K-1} with the last remainder dropped
// ("SyclReproSum", "How It Works": one-pass index updates give the same
// folds as depositing at the final index from the start).  The per-fold
// split only matters for raising the index in flight; summed over the folds,
// C_I(x) is x rounded to a multiple of the finest grid g_f = g_{I+K-1}, to
// nearest, with exact ties broken by the chained rule: away from zero unless
// the rounding bit of fold K-2 (g_f 2^(W-1)) is set, in which case toward
// zero.  So when I is known, a deposit is one rounding of |x| at g_f and an
// exact integer addition.
//
// The index is guessed from a fixed sample of the input: a subset's maximum
// lies in the same bin as the true maximum or in a finer one, so a guess is
// either right or some element lies above its bin -- which the kernels
// check, falling back to the general one-pass path.
//
// Double rounding.  With P' = |x| 2^64 / g_f = M 2^u (M the 53-bit
// significand), the rounded value is floor((P' + 2^63 - b) / 2^64), b the
// tie bit above (bit 103 of P').  Adding h - b to M (h = 2^(63-u)) and
// shifting by u gives P'' whose bits at and above 64 are exactly that value.
#pragma once
#include "adn.cuh"

namespace repro {
namespace fx {

constexpr int SAMPLE = 256;   // elements sampled for the index guess
// Word positions of P'' for K folds.  A valid element (inside the guessed
// bin) has shift u <= 50 + W (K - 1) over g_f, so its three words end at
// position (u >> 5) + 2.  K <= 3 keeps 7 positions (0..6); K = 6 needs 10.
// The double sum keeps, per sign and per thread, STR - 1 cell pairs (see
// fx_deposit).
template <int K>
struct FxGeo {
  static constexpr int UMAX = 50 + 40 * (K - 1);
  static constexpr int STR = K <= 3 ? 7 : (UMAX >> 5) + 3;
  static constexpr int NPOS = STR - 2;        // kept positions 2..STR-1
  static constexpr int CELLS = 2 * (STR - 1); // sum cell pairs, both signs
};
constexpr int STRIDE = FxGeo<3>::STR;

__device__ __forceinline__ uint32_t shl_clamp32(uint32_t v, int s) {   // s outside [0, 31] gives 0
  uint32_t r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(s));
  return r;
}
__device__ __forceinline__ uint32_t funnel_l(uint32_t lo, uint32_t hi, uint32_t n) {   // (hi:lo << n%32).hi
  uint32_t r;
  asm("shf.l.wrap.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(lo), "r"(hi), "r"(n));
  return r;
}
// a * b + c kept as multiply-adds: with b a kernel argument equal to 1 the
// compiler cannot turn them into integer-ALU additions (the ALU pipe is the
// one this kernel saturates; the multiply-add pipe has room).
__device__ __forceinline__ uint32_t mad32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ uint64_t madw(uint32_t a, uint32_t b, uint64_t c) {
  uint64_t r;
  asm("mad.wide.u32 %0, %1, %2, %3;" : "=l"(r) : "r"(a), "r"(b), "l"(c));
  return r;
}

struct FxConst {
  uint32_t one, negone, c63, c31, c256, c7, Cp;
};

// One deposit into the sum cells.  Sign s, position c = 0..STR-2 has a
// 64-bit cell A[c + (STR - 1) s] (words c and c + 1 of P'') and a 32-bit
// cell B[c + (STR - 1) s] (word c + 2), both at stride NT.  An element's
// words (w2, w1, w0) at position c enter as one 96-bit add into the pair,
// the carry out of A going into B: two cell updates per element.  Words at
// positions 0 and 1 are fraction bits of the element's own P'' and are
// multiplied by 0 before the add (a carry out of them would reach position
// 2).  B takes at most 2^22 per deposit and is emptied by fx_fold every 992
// deposits.  An element beyond the bin (flagged through umax) lands at
// position STR - 2, in bounds.  k.c7 must be (STR - 1) k.one.
// SUBN: subnormal inputs take their true significand (no hidden bit,
// exponent field read as 1), for grids fine enough to see them; without it
// the hidden bit is forced, which is exact whenever g_f / 2 lies above every
// subnormal.
template <int STR = STRIDE, bool SUBN = false>
__device__ __forceinline__ void fx_deposit(uint32_t hi, uint32_t lo, const FxConst& k, uint64_t* A, uint32_t* B,
                                           uint32_t NT, int& umax) {
  uint32_t eb = mad32(hi, k.one + k.one, 0u) >> 21;          // biased exponent
  uint32_t mh;
  if constexpr (SUBN) {
    const uint32_t nz = min(eb, 1u);                          // 0 for a subnormal or zero
    mh = (hi & 0xFFFFFu) | mad32(nz, 0x100000u * k.one, 0u);
    eb = max(eb, 1u);
  } else {
    mh = (hi & 0xFFFFFu) | 0x100000u;
  }
  int us = (int)mad32(eb, k.one, k.Cp);                       // shift of M
  umax = max(umax, us);
  uint32_t u = (uint32_t)max(us, 0);   // tiny values: their words stay below position 2
  uint32_t c = min(u >> 5, (uint32_t)(STR - 2));
  uint32_t hl = shl_clamp32(1u, (int)mad32(u, k.negone, k.c63));
  uint32_t hh = shl_clamp32(1u, (int)mad32(u, k.negone, k.c31));
  uint32_t b = min(mh & mad32(hl, k.c256, 0u), 1u);          // bit 103 of P': rounding bit of fold K-2
  uint64_t Mp = ((((uint64_t)mh) << 32) | lo) + ((((uint64_t)hh) << 32) | hl) - (uint64_t)b;
  uint32_t lo2 = (uint32_t)Mp, mh2 = (uint32_t)(Mp >> 32);
  uint32_t w0 = funnel_l(0u, lo2, u);
  uint32_t w1 = funnel_l(lo2, mh2, u);
  uint32_t w2 = funnel_l(mh2, 0u, u);
  uint32_t f1 = mad32(c, k.one, 127u) >> 7, f0 = mad32(c, k.one, 126u) >> 7;   // c >= 1, c >= 2
  uint32_t off = mad32(mad32(hi >> 31, k.c7, c), NT, 0u);
  uint64_t* p = A + off;
  uint32_t* pb = B + off;
  uint32_t a0, a1, bb = *pb;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(a0), "=r"(a1) : "l"(*p));
  asm("mad.lo.cc.u32 %0, %3, %4, %0;\n\tmadc.lo.cc.u32 %1, %5, %6, %1;\n\tmadc.lo.u32 %2, %7, %8, %2;"
      : "+r"(a0), "+r"(a1), "+r"(bb)
      : "r"(w0), "r"(f0), "r"(w1), "r"(f1), "r"(w2), "r"(k.one));
  uint64_t an;
  asm("mov.b64 %0, {%1, %2};" : "=l"(an) : "r"(a0), "r"(a1));
  *p = an;
  *pb = bb;
}

// Empties the B cells: B at position c + 2 is word 1 of the pair at c + 1,
// and the carry of that add goes to the next B (lowest first, so each
// carry is moved on in the same pass).  The carry of the top pair stays in
// the top B cell (position STR), which no deposit of a valid element uses.
template <int STR = STRIDE>
__device__ __forceinline__ void fx_fold(uint64_t* A, uint32_t* B, uint32_t NT) {
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    uint32_t carry = 0;
#pragma unroll
    for (int c = 0; c <= STR - 3; ++c) {
      uint64_t* pa = A + (c + 1 + (STR - 1) * s) * NT;
      uint32_t* pb = B + (c + (STR - 1) * s) * NT;
      uint32_t a0, a1;
      asm("mov.b64 {%0, %1}, %2;" : "=r"(a0), "=r"(a1) : "l"(*pa));
      asm("add.cc.u32 %0, %0, %2;\n\taddc.u32 %1, 0, 0;" : "+r"(a1), "=r"(carry) : "r"(*pb + carry));
      uint64_t an;
      asm("mov.b64 %0, {%1, %2};" : "=l"(an) : "r"(a0), "r"(a1));
      *pa = an;
      *pb = 0;
    }
    B[(STR - 2 + (STR - 1) * s) * NT] += carry;
  }
}

// Signed 192-bit integer.
struct I192 {
  uint64_t w0, w1, w2;
};
__device__ __forceinline__ I192 i192_add(I192 a, I192 b) {
  I192 r;
  asm("add.cc.u64 %0, %3, %6;\n\taddc.cc.u64 %1, %4, %7;\n\taddc.u64 %2, %5, %8;"
      : "=l"(r.w0), "=l"(r.w1), "=l"(r.w2)
      : "l"(a.w0), "l"(a.w1), "l"(a.w2), "l"(b.w0), "l"(b.w1), "l"(b.w2));
  return r;
}
__device__ __forceinline__ I192 i192_shfl_xor(I192 v, int m) {
  I192 r;
  r.w0 = __shfl_xor_sync(0xffffffffu, v.w0, m);
  r.w1 = __shfl_xor_sync(0xffffffffu, v.w1, m);
  r.w2 = __shfl_xor_sync(0xffffffffu, v.w2, m);
  return r;
}
// v * 2^(32 j) for a W128 v >= 0 (j = 0..4), as I192 (upper bits beyond 192 dropped: |total| < 2^160)
__device__ __forceinline__ I192 i192_from_shifted(W128 v, int j) {
  uint32_t src[4] = {(uint32_t)v.lo, (uint32_t)(v.lo >> 32), (uint32_t)v.hi, (uint32_t)((uint64_t)v.hi >> 32)};
  uint32_t d[6] = {0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (i + j < 6) d[i + j] = src[i];
  return I192{((uint64_t)d[1] << 32) | d[0], ((uint64_t)d[3] << 32) | d[2], ((uint64_t)d[5] << 32) | d[4]};
}
__device__ __forceinline__ I192 i192_neg(I192 a) {
  I192 r{~a.w0, ~a.w1, ~a.w2};
  return i192_add(r, I192{1, 0, 0});
}

// Signed 320-bit integer: block totals for K = 4..6 (|total| < 2^280 in
// units of g_f: an element's rounded value is below 2^(UMAX - 10) <= 2^240,
// at most 2^36 elements).
struct I320 {
  uint64_t w[5];
};
__device__ __forceinline__ I320 i320_add(I320 a, I320 b) {
  I320 r;
  asm("add.cc.u64 %0, %5, %10;\n\taddc.cc.u64 %1, %6, %11;\n\taddc.cc.u64 %2, %7, %12;\n\t"
      "addc.cc.u64 %3, %8, %13;\n\taddc.u64 %4, %9, %14;"
      : "=l"(r.w[0]), "=l"(r.w[1]), "=l"(r.w[2]), "=l"(r.w[3]), "=l"(r.w[4])
      : "l"(a.w[0]), "l"(a.w[1]), "l"(a.w[2]), "l"(a.w[3]), "l"(a.w[4]), "l"(b.w[0]), "l"(b.w[1]),
        "l"(b.w[2]), "l"(b.w[3]), "l"(b.w[4]));
  return r;
}
__device__ __forceinline__ I320 i320_shfl_xor(I320 v, int m) {
  I320 r;
#pragma unroll
  for (int i = 0; i < 5; ++i) r.w[i] = __shfl_xor_sync(0xffffffffu, v.w[i], m);
  return r;
}
// v * 2^(32 j) for a W128 v >= 0 below 2^96 (a column sum), as I320
__device__ __forceinline__ I320 i320_from_shifted(W128 v, int j) {
  uint32_t src[4] = {(uint32_t)v.lo, (uint32_t)(v.lo >> 32), (uint32_t)v.hi, (uint32_t)((uint64_t)v.hi >> 32)};
  uint32_t d[10] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (i + j < 10) d[i + j] = src[i];
  I320 r;
#pragma unroll
  for (int i = 0; i < 5; ++i) r.w[i] = ((uint64_t)d[2 * i + 1] << 32) | d[2 * i];
  return r;
}
__device__ __forceinline__ I320 i320_neg(I320 a) {
  I320 r;
#pragma unroll
  for (int i = 0; i < 5; ++i) r.w[i] = ~a.w[i];
  return i320_add(r, I320{{1, 0, 0, 0, 0}});
}

// The same operations under one name for either width.
__device__ __forceinline__ I192 tot_add(I192 a, I192 b) { return i192_add(a, b); }
__device__ __forceinline__ I320 tot_add(I320 a, I320 b) { return i320_add(a, b); }
__device__ __forceinline__ I192 tot_neg(I192 a) { return i192_neg(a); }
__device__ __forceinline__ I320 tot_neg(I320 a) { return i320_neg(a); }
__device__ __forceinline__ I192 tot_shfl_xor(I192 v, int m) { return i192_shfl_xor(v, m); }
__device__ __forceinline__ I320 tot_shfl_xor(I320 v, int m) { return i320_shfl_xor(v, m); }
__device__ __forceinline__ void tot_from_shifted(W128 v, int j, I192* r) { *r = i192_from_shifted(v, j); }
__device__ __forceinline__ void tot_from_shifted(W128 v, int j, I320* r) { *r = i320_from_shifted(v, j); }
__device__ __forceinline__ I192 tot_ldcg(const I192* q) { return I192{__ldcg(&q->w0), __ldcg(&q->w1), __ldcg(&q->w2)}; }
__device__ __forceinline__ I320 tot_ldcg(const I320* q) {
  I320 r;
#pragma unroll
  for (int i = 0; i < 5; ++i) r.w[i] = __ldcg(&q->w[i]);
  return r;
}

// Number of 64-bit words of a total, and the words themselves.
template <typename TOT> struct TotW;
template <> struct TotW<I192> { static constexpr int N = 3; };
template <> struct TotW<I320> { static constexpr int N = 5; };
__device__ __forceinline__ uint64_t tot_word(const I192& t, int i) { return i == 0 ? t.w0 : i == 1 ? t.w1 : t.w2; }
__device__ __forceinline__ uint64_t tot_word(const I320& t, int i) { return t.w[i]; }

// The thread's cells (after fx_fold) as one signed total TOT in units of
// g_f.  Per sign the kept columns, relative to position 2, are: 0 (A[1] >> 32
// and A[2]), j = 1..STR-4 (A[j + 2]) and STR - 2 (the top B cell).
template <int STR, typename TOT>
__device__ __forceinline__ TOT fx_thread_total(const uint64_t* A, const uint32_t* B, uint32_t NT) {
  TOT t[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const uint64_t* As = A + (STR - 1) * s * NT;
    TOT v, w;
    tot_from_shifted(W128{As[NT] >> 32, 0}, 0, &v);
#pragma unroll
    for (int j = 0; j <= STR - 4; ++j) {
      tot_from_shifted(W128{As[(j + 2) * NT], 0}, j, &w);
      v = tot_add(v, w);
    }
    tot_from_shifted(W128{B[(STR - 2 + (STR - 1) * s) * NT], 0}, STR - 2, &w);
    t[s] = tot_add(v, w);
  }
  return tot_add(t[0], tot_neg(t[1]));
}

// Bin index of a set whose largest biased exponent field is eb (0: all
// zero or subnormal), capped at NB - K.
template <typename T>
__device__ __forceinline__ int index_of_exponent(int eb, int K) {
  typedef Geom<T> G;
  if (eb == 0) return G::NB - K;
  int j = (G::B0 + G::W - 2 - (eb - G::BIAS)) / G::W;
  j = min(j, G::NB - 1);
  return min(j, G::NB - K);
}

// Index guess from the largest exponent field over SAMPLE evenly spaced
// elements (every block computes the same value).  Returns the bin index;
// *emax_out gets the largest biased exponent seen (all-ones: Inf/NaN).
// s_emax: one shared word.  All threads of the block must call it.
template <typename T>
__device__ __forceinline__ int guess_index(const T* __restrict__ x, int64_t n, int K, unsigned* s_emax,
                                           int* emax_out) {
  typedef Geom<T> G;
  constexpr unsigned EMASK = sizeof(T) == 8 ? 0x7FF00000u : 0x7F800000u;
  constexpr int ESH = sizeof(T) == 8 ? 20 : 23;
  if (threadIdx.x == 0) *s_emax = 0;
  __syncthreads();
  const int64_t S = n < SAMPLE ? n : SAMPLE;
  unsigned em = 0;
  for (int64_t j = threadIdx.x; j < S; j += blockDim.x) {
    int64_t pos = (j * n) / S;
    unsigned hi;
    if constexpr (sizeof(T) == 8) hi = (unsigned)__double2hiint(__ldg(x + pos));
    else hi = __float_as_uint(__ldg(x + pos));
    em = max(em, hi & EMASK);
  }
  em = __reduce_max_sync(0xffffffffu, em);
  if ((threadIdx.x & 31) == 0) atomicMax(s_emax, em);
  __syncthreads();
  const int eb = (int)(*s_emax >> ESH);
  *emax_out = eb;
  return index_of_exponent<T>(eb, K);
}

// Largest biased exponent inside bin I: |x| < 2^(beta_I + W - 1).
template <typename T>
__device__ __forceinline__ int bin_top_exponent(int I) {
  typedef Geom<T> G;
  return I == 0 ? (sizeof(T) == 8 ? 2046 : 254) : G::BIAS + beta<T>(I) + G::W - 2;
}

__device__ __forceinline__ FxConst make_const(int bf, uint32_t one, int stride = STRIDE) {
  FxConst k;
  k.one = one;
  k.negone = 0u - one;
  k.c63 = 63u * one;
  k.c31 = 31u * one;
  k.c256 = 256u * one;
  k.c7 = (uint32_t)stride * one;   // cells per sign
  k.Cp = (uint32_t)(-1011 - bf);
  return k;
}

// Rounded value of a finite double |x| at g_f as a 128-bit integer (< 2^122),
// same arithmetic as fx_deposit but in registers: P'' = M' 2^u over six
// 32-bit words through one-hot multipliers 2^(u - 32 j) (no variable word
// selection), value = words 2..5.
__device__ __forceinline__ void round_f64(uint32_t hi, uint32_t lo, const FxConst& k, uint64_t& r_lo, uint64_t& r_hi) {
  uint32_t eb = mad32(hi, k.one + k.one, 0u) >> 21;
  int us = (int)mad32(eb, k.one, k.Cp);
  uint32_t u = (uint32_t)max(us, 0);
  uint32_t mh = (hi & 0xFFFFFu) | 0x100000u;
  uint32_t hl = shl_clamp32(1u, (int)mad32(u, k.negone, k.c63));
  uint32_t hh = shl_clamp32(1u, (int)mad32(u, k.negone, k.c31));
  uint32_t b = min(mh & mad32(hl, k.c256, 0u), 1u);
  uint64_t Mp = ((((uint64_t)mh) << 32) | lo) + ((((uint64_t)hh) << 32) | hl) - (uint64_t)b;
  uint32_t lo2 = (uint32_t)Mp, mh2 = (uint32_t)(Mp >> 32);
  uint32_t q0 = shl_clamp32(1u, (int)u), q1 = shl_clamp32(1u, (int)u - 32), q2 = shl_clamp32(1u, (int)u - 64),
           q3 = shl_clamp32(1u, (int)u - 96), q4 = shl_clamp32(1u, (int)u - 128);
  uint64_t a0 = madw(lo2, q0, 0), a1 = madw(lo2, q1, 0), a2 = madw(lo2, q2, 0), a3 = madw(lo2, q3, 0),
           a4 = madw(lo2, q4, 0);
  uint64_t s0 = madw(mh2, q0, a0 >> 32), s1 = madw(mh2, q1, a1 >> 32), s2 = madw(mh2, q2, a2 >> 32),
           s3 = madw(mh2, q3, a3 >> 32), s4 = madw(mh2, q4, a4 >> 32);
  uint32_t V0 = (uint32_t)a2 | (uint32_t)s1 | (uint32_t)(s0 >> 32);
  uint32_t V1 = (uint32_t)a3 | (uint32_t)s2 | (uint32_t)(s1 >> 32);
  uint32_t V2 = (uint32_t)a4 | (uint32_t)s3 | (uint32_t)(s2 >> 32);
  uint32_t V3 = (uint32_t)s4 | (uint32_t)(s3 >> 32);
  r_lo = ((uint64_t)V1 << 32) | V0;
  r_hi = ((uint64_t)V3 << 32) | V2;
}


// ------------------------------------------------------------------ float
// Float rounding at g_f in 32-bit pieces.  With s = eb + sh (the shift that
// puts g_f at bit 24 of M 2^s), the rounded value is
//   s <= 24:  (M + 2^(23 - s) - b) >> (24 - s),  b = bit 36 - s of M,
//   s >= 24:  M << (s - 24)  (exact, below 2^38; at s = 24 both give M),
// every shift clamped (out-of-range amounts give 0), so the two parts are
// computed unconditionally and one of them is zero.
struct F32Const {
  int c23, c24, cm24, c56;   // constants minus the biased exponent
};
__device__ __forceinline__ F32Const make_f32_const(int sh) {
  return F32Const{23 - sh, 24 - sh, sh - 24, 56 - sh};
}
__device__ __forceinline__ uint32_t shr_clamp32(uint32_t v, int s) {   // s outside [0, 31] gives 0
  uint32_t r;
  asm("shr.b32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(s));
  return r;
}
// |x| rounded at g_f as (lo, hi) 32-bit words; eb: biased exponent field.
__device__ __forceinline__ void round_f32w(uint32_t bits, const F32Const& k, uint32_t& lo, uint32_t& hi) {
  const int eb = (int)((bits >> 23) & 0xFFu);
  const uint32_t M = (bits & 0x7FFFFFu) | 0x800000u;
  const uint32_t h = shl_clamp32(1u, k.c23 - eb);
  // tie bit 36 - s of M, as a mask derived from h: zero whenever h is (the
  // exact case s >= 24, where M is not rounded)
  const uint32_t b = min(M & (h << 13), 1u);
  const uint32_t small = shr_clamp32(M + h - b, k.c24 - eb);
  lo = small | shl_clamp32(M, eb + k.cm24);
  hi = shr_clamp32(M, k.c56 - eb);
}

// Signed 96-bit integer in 32-bit words (float running totals: < 2^71).
struct I96 {
  uint32_t w0, w1, w2;
};
// a + (sign ? -(hi:lo) : (hi:lo)), sm = 0 or all ones
__device__ __forceinline__ I96 i96_add_signed(I96 a, uint32_t lo, uint32_t hi, uint32_t sm) {
  I96 r;
  asm("add.cc.u32 %0, %3, %6;\n\taddc.cc.u32 %1, %4, %7;\n\taddc.u32 %2, %5, %8;"
      : "=r"(r.w0), "=r"(r.w1), "=r"(r.w2)
      : "r"(a.w0), "r"(a.w1), "r"(a.w2), "r"(lo ^ sm), "r"(hi ^ sm), "r"(sm));
  // + 1 for a negation: added through the lowest word with carry
  asm("add.cc.u32 %0, %0, %3;\n\taddc.cc.u32 %1, %1, 0;\n\taddc.u32 %2, %2, 0;"
      : "+r"(r.w0), "+r"(r.w1), "+r"(r.w2)
      : "r"(sm & 1u));
  return r;
}
// Normal results of a * 2^lsb, rounded on the two's complement (no
// negation): with p the leading bit of a (of ~a for a < 0), the 32 bits from
// p down hold the significand field, the half bit and 7 more; the bits below
// fold into one sticky bit.  q = floor(a / 2^(p - 23)) + up (a carry out of
// the window gives 2^24); the magnitude is q for a >= 0 and 2^24 - q for
// a < 0 (bits above p are ones), in [2^23, 2^24], and 2^24 carries into the
// exponent.  False (nothing written) for a = 0 or -1 and outside the normal
// range.
__device__ __forceinline__ bool i96_to_float_normal(I96 a, int lsb, uint32_t* out) {
  const uint32_t s = (uint32_t)((int32_t)a.w2 >> 31);
  const bool z2 = a.w2 == s;
  uint32_t top = z2 ? a.w1 : a.w2, nxt = z2 ? a.w0 : a.w1;
  const uint32_t rest = z2 ? 0u : a.w0;
  int e = z2 ? 0 : 32;   // bit position of nxt
  if (top == s) {
    top = nxt;
    nxt = 0u;
    e -= 32;
  }
  const uint32_t lz = (uint32_t)__clz((int)(top ^ s));   // 32 only for a = 0 or -1
  const int E = e + 63 - (int)lz + lsb;                   // exponent of bit p
  if (lz == 32u || (unsigned)(E + 126) > 253u) return false;
  const uint32_t v = funnel_l(nxt, top, lz);              // bits p .. p - 31
  const uint32_t below = shl_clamp32(nxt, (int)lz) | rest;
  const uint32_t st = ((v & 0x7Fu) | below) != 0u ? 1u : 0u;
  const uint32_t odd = (v >> 8) & 1u;
  const uint32_t w = (v & ~0x7Fu) | st;
  const uint32_t u = w + 0x7Fu + odd;
  const uint32_t q = (u >> 8) | ((uint32_t)(u < w) << 24);
  const uint32_t m = (q ^ s) + (s & ((1u << 24) + 1u));
  *out = (s & 0x80000000u) + ((uint32_t)(E + 126) << 23) + m;
  return true;
}

// Correct rounding of a * 2^lsb to float for |a| * 2^lsb >= 2^-126 or a = 0
// (the fast path's grids guarantee it); overflow gives +-Inf.
__device__ __forceinline__ float i96_to_float(I96 a, int lsb) {
  uint32_t fast;
  if (i96_to_float_normal(a, lsb, &fast)) return __uint_as_float(fast);
  const uint32_t sm = (uint32_t)((int32_t)a.w2 >> 31);
  uint32_t x0 = a.w0 ^ sm, x1 = a.w1 ^ sm, x2 = a.w2 ^ sm;
  asm("add.cc.u32 %0, %0, %3;\n\taddc.cc.u32 %1, %1, 0;\n\taddc.u32 %2, %2, 0;"
      : "+r"(x0), "+r"(x1), "+r"(x2)
      : "r"(sm & 1u));
  const bool t2 = x2 != 0, t1 = x1 != 0;
  const uint32_t top = t2 ? x2 : (t1 ? x1 : x0);
  const uint32_t nxt = t2 ? x1 : (t1 ? x0 : 0u);
  const uint32_t rest = t2 ? x0 : 0u;
  if (top == 0u) return 0.0f;
  const int tw = t2 ? 2 : (t1 ? 1 : 0);
  const int lz = __clz((int)top);
  const uint32_t v = funnel_l(nxt, top, (uint32_t)lz);      // leading bit at 31
  const uint32_t lost = shl_clamp32(nxt, lz) | rest;         // bits below v
  uint32_t m = v >> 8;
  const uint32_t rb = (v >> 7) & 1u;
  const uint32_t st = (v & 0x7Fu) | lost;
  m += rb & ((st != 0u) | (m & 1u));
  const int E = 32 * tw + 31 - lz + lsb;                      // exponent of the leading bit
  uint32_t r = ((uint32_t)(E + 126) << 23) + m;                // a rounding carry moves into the exponent
  if (E > 127) r = 0x7F800000u;
  return __uint_as_float(r | (sm & 0x80000000u));
}

}  // namespace fx
}  // namespace repro
