// Binned (Ahrens-Demmel-Nguyen) summation: device-side building blocks.
//
// The binned format follows the SyclReproSum ("How It Works",
// "Template Parameters", "Accumulator capacity"): a value is split into K
// pieces on a fixed global grid of exponent bins, bin width W = 13 (float) /
// 40 (double), at most 21 / 52 bins.  Bin j has grid unit g_j = 2^(B0 - W j)
// (B0 = 117 / 986, so the finest grid is 2^-143 / 2^-1054 and values below
// half of it, ~2^-144 / ~2^-1055, are absorbed), and holds |x| < 2^(B0 - W j
// + W - 1).  With I the bin of max|x| (capped at nb - K), piece k of x is
// round-half-away-from-zero of the running remainder on grid g_{I+k}, the
// last remainder dropped.  Fold sums are exact integers (units of their
// grid), so any merge order gives the same state; the result is the single
// correct rounding of their total.
//
// Two deposit forms produce the same fold sums:
//  - float: the SyclReproSum page's floating-point primaries (deposit with a forced
//    least-significant "sticky" bit so the grid rounding is order
//    independent, periodic renormalisation), flushed into int64 lanes;
//  - double (and every rare case): integer digits of the same chained
//    rounding.  GB300 runs FP64 adds at a small fraction of the FP32/INT rate,
//    so no floating-point double arithmetic sits on the hot path.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace repro {

// Two's-complement 128-bit integer as two 64-bit words.  (Fold sums need
// more than 64 bits: |F_k| <= N 2^(W-1).)  Plain 64-bit fields keep the
// values well defined in registers, local and shared memory alike.
struct W128 {
  uint64_t lo;
  int64_t hi;
};
__host__ __device__ __forceinline__ W128 w_from(int64_t v) { return W128{(uint64_t)v, v >> 63}; }
__host__ __device__ __forceinline__ W128 w_add(W128 a, W128 b) {
  uint64_t lo = a.lo + b.lo;
  return W128{lo, (int64_t)((uint64_t)a.hi + (uint64_t)b.hi + (uint64_t)(lo < a.lo))};
}
__host__ __device__ __forceinline__ bool w_is_zero(W128 a) { return a.lo == 0 && a.hi == 0; }

template <typename T> struct Geom;
template <> struct Geom<float> {
  static constexpr int W = 13, NB = 21, B0 = 117, P = 24, QMIN = -149, EMAX = 128, BIAS = 127;
  typedef uint32_t U;
};
template <> struct Geom<double> {
  static constexpr int W = 40, NB = 52, B0 = 986, P = 53, QMIN = -1074, EMAX = 1024, BIAS = 1023;
  typedef uint64_t U;
};

template <typename T> __host__ __device__ constexpr int beta(int j) { return Geom<T>::B0 - Geom<T>::W * j; }

// Special-value flags: any NaN, or +Inf with -Inf, gives the canonical quiet
// NaN; otherwise an Inf propagates ("SyclReproSum", "How It Works").
enum : int { FL_NAN = 1, FL_PINF = 2, FL_NINF = 4 };

// ---------------------------------------------------------------- decoding
// |x| = M * 2^e for a finite x (M < 2^53, zero for x == 0).
__device__ __forceinline__ void decode(double x, uint64_t& M, int& e, bool& neg) {
  uint64_t b = (uint64_t)__double_as_longlong(x);
  neg = (b >> 63) != 0;
  int eb = (int)((b >> 52) & 0x7FF);
  uint64_t mant = b & ((1ull << 52) - 1);
  M = eb ? (mant | (1ull << 52)) : mant;
  e = (eb ? eb : 1) - 1075;
}
__device__ __forceinline__ void decode(float x, uint64_t& M, int& e, bool& neg) {
  uint32_t b = (uint32_t)__float_as_uint(x);
  neg = (b >> 31) != 0;
  int eb = (int)((b >> 23) & 0xFF);
  uint32_t mant = b & ((1u << 23) - 1);
  M = eb ? (mant | (1u << 23)) : mant;
  e = (eb ? eb : 1) - 150;
}

// floor(log2|x|) for finite non-zero x.
template <typename T> __device__ __forceinline__ int ilog2_abs(T x) {
  uint64_t M; int e; bool n;
  decode(x, M, e, n);
  return e + 63 - __clzll((long long)M);
}

// Finest bin j with |x| < 2^(beta_j + W - 1).
template <typename T> __device__ __forceinline__ int bin_index(T x) {
  typedef Geom<T> G;
  int j = (G::B0 + G::W - 2 - ilog2_abs(x)) / G::W;
  return j > G::NB - 1 ? G::NB - 1 : j;
}

// Absolute-value bit threshold: |x| bits >= thr means "x is outside bin I (or
// Inf/NaN)".  For I == 0 every finite value fits, only Inf/NaN exceed it.
template <typename T> __device__ __forceinline__ typename Geom<T>::U index_threshold(int I) {
  typedef Geom<T> G;
  typedef typename G::U U;
  if (I == 0) return sizeof(T) == 4 ? (U)0x7F800000u : (U)0x7FF0000000000000ull;
  int ex = beta<T>(I) + G::W - 1;       // threshold 2^ex, a normal number
  return (U)(ex + G::BIAS) << (G::P - 1);
}

template <typename T> __device__ __forceinline__ typename Geom<T>::U abs_bits(T x);
template <> __device__ __forceinline__ uint32_t abs_bits<float>(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }
template <> __device__ __forceinline__ uint64_t abs_bits<double>(double x) {
  return (uint64_t)__double_as_longlong(x) & 0x7FFFFFFFFFFFFFFFull;
}

template <typename T> __device__ __forceinline__ int special_flag(T x) {
  // caller knows x is Inf or NaN
  if (x != x) return FL_NAN;
  return x > 0 ? FL_PINF : FL_NINF;
}

// ----------------------------------------------------- exact integer digits
// bits [lo, lo + w) of |x| = M * 2^e, w <= 62.
__device__ __forceinline__ int64_t field(uint64_t M, int e, int lo, int w) {
  int s = e - lo;
  uint64_t v;
  if (s >= 0) v = (s >= 64) ? 0 : (M << s);
  else v = (-s >= 64) ? 0 : (M >> -s);
  return (int64_t)(v & ((1ull << w) - 1));
}
// 1 if |x| has a set bit strictly below position lo.
__device__ __forceinline__ bool bits_below(uint64_t M, int e, int lo) {
  int s = lo - e;
  if (s <= 0) return false;
  if (s >= 64) return M != 0;
  return (M & ((1ull << s) - 1)) != 0;
}

// Digits a_k = piece_k / g_{I+k} of the chained round-half-away decomposition
// of x, k = 0..K-1.  Exact for every finite x (ties, subnormals, bin 0).
// Works on |x| (the decomposition is odd in x):  with R = floor(r / (g/4))
// and f = "r has bits below g/4", round-half-away(r / g) is
// (R + 2 - [R < 0 and f == 0]) >> 2; the next remainder in units of its own
// quarter-grid is (R - 4 a) 2^W plus the next W bits of |x|.
template <typename T>
__device__ void chain_digits(T x, int I, int K, int64_t* a) {
  typedef Geom<T> G;
  uint64_t M; int e; bool neg;
  decode(x, M, e, neg);
  int lo = beta<T>(I) - 2;
  int64_t R;
  {
    int s = e - lo;   // |x| < 2^(beta_I + W - 1) so R < 2^(W + 1)
    R = (s >= 0) ? (int64_t)(M << s) : ((-s >= 64) ? 0 : (int64_t)(M >> -s));
  }
  bool f = bits_below(M, e, lo);
  for (int k = 0; k < K; ++k) {
    int64_t d = (R + 2 - ((R < 0 && !f) ? 1 : 0)) >> 2;
    a[k] = neg ? -d : d;
    if (k == K - 1) break;
    int nlo = lo - G::W;
    R = (R - 4 * d) * ((int64_t)1 << G::W) + field(M, e, nlo, G::W);   // |R - 4d| <= 2: no overflow
    f = bits_below(M, e, nlo);
    lo = nlo;
  }
}

// -------------------------------------------------- fast digits (double)
// Same digits as chain_digits for a double, with a fixed K and index.  With
// |X| = |x| / 2^(beta_k - 1) written in binary, digit k before tie handling
// is the signed value of the W bits above the binary point of |x| / 2^beta_k
// (the bit at beta_k + W - 1 is the sign: it is the rounding bit of fold
// k - 1) plus the bit just below, beta_k - 1 (round half up).  One shifted
// copy G of the significand per fold holds both: bits [24, 64) the window,
// bit 23 the rounding bit.  Round-half-away differs from round-half-up only
// at an exact tie whose remainder is negative: for |x| that is fold k >= 1
// when the lowest set bit of |x| is beta_k - 1 and the rounding bit of fold
// k - 1 is set; then digit k drops by one and digit k + 1 gains 2^W.
__device__ __forceinline__ uint64_t shl_clamp(uint64_t v, int s) {
  uint64_t r;
  asm("shl.b64 %0, %1, %2;" : "=l"(r) : "l"(v), "r"(s));   // s >= 64 (as unsigned) gives 0
  return r;
}
__device__ __forceinline__ uint64_t shr_clamp(uint64_t v, int s) {
  uint64_t r;
  asm("shr.b64 %0, %1, %2;" : "=l"(r) : "l"(v), "r"(s));
  return r;
}

template <int K>
struct FastD {
  int tsh[K];   // shift of the significand for fold k: biased exponent + tsh[k]
  int tie[K];   // biased exponent + ctz(significand) == tie[k]: tie at fold k
  __device__ __forceinline__ void set(int I) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      int b = beta<double>(I + k);
      tsh[k] = 24 - b - 1075;        // e - (beta_k - 1) + 23, e = eb - 1075
      tie[k] = b - 1 + 1075;
    }
  }
};

// Digits of a finite double x (no Inf/NaN) at the index set in `c`.
template <int K>
__device__ __forceinline__ void fast_digits_f64(double x, const FastD<K>& c, int64_t* a) {
  uint32_t hi = (uint32_t)__double2hiint(x), lo = (uint32_t)__double2loint(x);
  int eb = (int)((hi >> 20) & 0x7FF);
  int ee = eb ? eb : 1;
  uint32_t mh = (hi & 0xFFFFFu) | (eb ? 0x100000u : 0u);
  uint64_t M = ((uint64_t)mh << 32) | lo;
  uint64_t G[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    int t = ee + c.tsh[k];
    G[k] = shl_clamp(M, t) | shr_clamp(M, -t);
    a[k] = ((int64_t)G[k] >> 24) + (int64_t)((G[k] >> 23) & 1);
  }
  // ties with a negative remainder (folds k >= 1)
  int ctz = lo ? (__ffs((int)lo) - 1) : (32 + __ffs((int)mh) - 1);
  int lam = ee + ctz;
#pragma unroll
  for (int k = 1; k < K; ++k) {
    bool cfix = (lam == c.tie[k]) && ((int64_t)G[k] < 0);
    a[k] -= cfix ? 1 : 0;
    if (k + 1 < K) a[k + 1] += cfix ? ((int64_t)1 << Geom<double>::W) : 0;
  }
  if (hi >> 31) {
#pragma unroll
    for (int k = 0; k < K; ++k) a[k] = -a[k];
  }
}

// ------------------------------------------------------------ 128-bit shuffles
__device__ __forceinline__ W128 shfl_xor_w(W128 v, int m) {
  uint32_t w0 = (uint32_t)v.lo, w1 = (uint32_t)(v.lo >> 32), w2 = (uint32_t)v.hi, w3 = (uint32_t)((uint64_t)v.hi >> 32);
  w0 = __shfl_xor_sync(0xffffffffu, w0, m);
  w1 = __shfl_xor_sync(0xffffffffu, w1, m);
  w2 = __shfl_xor_sync(0xffffffffu, w2, m);
  w3 = __shfl_xor_sync(0xffffffffu, w3, m);
  return W128{((uint64_t)w1 << 32) | w0, (int64_t)(((uint64_t)w3 << 32) | w2)};
}
__device__ __forceinline__ W128 shfl_up_w(W128 v, int d) {
  uint32_t w0 = (uint32_t)v.lo, w1 = (uint32_t)(v.lo >> 32), w2 = (uint32_t)v.hi, w3 = (uint32_t)((uint64_t)v.hi >> 32);
  w0 = __shfl_up_sync(0xffffffffu, w0, d);
  w1 = __shfl_up_sync(0xffffffffu, w1, d);
  w2 = __shfl_up_sync(0xffffffffu, w2, d);
  w3 = __shfl_up_sync(0xffffffffu, w3, d);
  return W128{((uint64_t)w1 << 32) | w0, (int64_t)(((uint64_t)w3 << 32) | w2)};
}

// -------------------------------------------------------- merged binned state
// Fold sums as 128-bit integers: |F_k| <= N 2^(W-1) < 2^103 within capacity.
template <int KMAXS> struct State {
  int I;
  int flags;
  W128 F[KMAXS];
};

// F[idx] for 0 <= idx < K, else zero.  Small compile-time arrays use a static
// select chain (stays in registers); large ones index directly.
template <int N, typename V>
__device__ __forceinline__ V fold_at(const V* F, int K, int idx) {
  if constexpr (N <= 8) {
    V v{};
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (j < K && j == idx) v = F[j];
    return v;
  } else {
    return (idx >= 0 && idx < K) ? F[idx] : V{};
  }
}

// Re-express fold sums held at index Ifrom at the coarser index Ito <= Ifrom:
// fold k moves to k + (Ifrom - Ito), the finest ones drop off, new top folds
// are zero.  Exact: a value inside bin Ifrom has zero pieces on coarser grids.
constexpr int KMAXS_SHIFT = 52;
template <typename V, int KT>
__device__ __forceinline__ void shift_folds(V* F, int K, int delta) {
  if (delta <= 0) return;
  // through a copy: no element is read after it has been written
  V t[KMAXS_SHIFT];
  for (int k = 0; k < K; ++k) t[k] = (k >= delta) ? F[k - delta] : V{};
  for (int k = 0; k < K; ++k) F[k] = t[k];
}

// --------------------------------------------------------------- conversion
// Correct rounding (nearest-even) of sum_k F_k g_{I+k} to T, +0.0 for an exact
// zero, +-Inf on overflow; flags first.  One thread; multi-limb arithmetic
// over the exact span of the folds.
template <typename T> __device__ __forceinline__ T canonical_nan();
template <> __device__ __forceinline__ float canonical_nan<float>() { return __uint_as_float(0x7fc00000u); }
template <> __device__ __forceinline__ double canonical_nan<double>() {
  return __longlong_as_double(0x7ff8000000000000ll);
}

template <typename T> __device__ __forceinline__ T from_flags(int flags) {
  if ((flags & FL_NAN) || ((flags & FL_PINF) && (flags & FL_NINF))) return canonical_nan<T>();
  return (flags & FL_PINF) ? (T)INFINITY : (T)-INFINITY;
}

// Assemble sign * m * 2^q (m < 2^P, m * 2^q representable or overflowing).
template <typename T> __device__ __forceinline__ T assemble(bool neg, uint64_t m, int q) {
  typedef Geom<T> G;
  if (m == 0) return neg ? (T)-0.0 : (T)0.0;
  int lb = 63 - __clzll((long long)m);
  if (lb + q >= G::EMAX) return neg ? (T)-INFINITY : (T)INFINITY;
  uint64_t bitsv;
  if (lb == G::P - 1) {
    uint64_t ef = (uint64_t)(q + G::P - 1 + G::BIAS);
    bitsv = (ef << (G::P - 1)) | (m & ((1ull << (G::P - 1)) - 1));
  } else {
    bitsv = m;  // subnormal: q == QMIN
  }
  if (sizeof(T) == 4) {
    uint32_t b = (uint32_t)bitsv | (neg ? 0x80000000u : 0u);
    return (T)__uint_as_float(b);
  } else {
    uint64_t b = bitsv | (neg ? 0x8000000000000000ull : 0ull);
    return (T)__longlong_as_double((long long)b);
  }
}

// Round a non-negative multi-limb integer mag (little-endian uint32 limbs,
// nl limbs) times 2^lsb to T.
template <typename T>
__device__ T round_limbs(bool neg, const uint32_t* mag, int nl, int lsb) {
  typedef Geom<T> G;
  int top = -1;
  for (int i = nl - 1; i >= 0; --i)
    if (mag[i]) { top = 32 * i + 31 - __clz((int)mag[i]); break; }
  if (top < 0) return (T)0.0;   // exact zero -> +0
  int E = top + lsb;
  int q = E - G::P + 1;
  if (q < G::QMIN) q = G::QMIN;
  int qs = q - lsb;
  uint64_t m = 0;
  bool half = false, sticky = false;
  if (qs <= 0) {
    // every bit is kept: m = mag << -qs (fits: top - qs < P)
    for (int b = top; b >= 0; --b) m = (m << 1) | ((mag[b >> 5] >> (b & 31)) & 1u);
    m <<= -qs;
  } else {
    for (int b = top; b >= qs; --b) m = (m << 1) | ((mag[b >> 5] >> (b & 31)) & 1u);
    int hb = qs - 1;
    half = (mag[hb >> 5] >> (hb & 31)) & 1u;
    for (int i = 0; i < (hb >> 5) && !sticky; ++i) sticky = mag[i] != 0;
    if (!sticky && (hb & 31)) sticky = (mag[hb >> 5] & ((1u << (hb & 31)) - 1u)) != 0;
  }
  if (half && (sticky || (m & 1))) m += 1;
  if (m == (1ull << G::P)) { m >>= 1; q += 1; }
  return assemble<T>(neg, m, q);
}

// Maximum limbs: W (K-1) + 128 + 2 bits.
template <typename T> struct ConvLimbs {
  static constexpr int N = (Geom<T>::W * (Geom<T>::NB - 1) + 134) / 32 + 2;
};

template <typename T, int KMAXS>
__device__ T convert_state(const State<KMAXS>& st, int K) {
  typedef Geom<T> G;
  if (st.flags) return from_flags<T>(st.flags);
  constexpr int NLMAX = ConvLimbs<T>::N;
  int nl = (G::W * (K - 1) + 134) / 32 + 2;
  if (nl > NLMAX) nl = NLMAX;
  uint32_t limb[NLMAX];
  for (int i = 0; i < nl; ++i) limb[i] = 0;
  for (int k = 0; k < K; ++k) {
    W128 v = st.F[k];
    if (w_is_zero(v)) continue;
    int off = G::W * (K - 1 - k);
    int li = off >> 5, sh = off & 31;
    // v << sh as 5 words (160 bits) with sign extension above.
    uint32_t ext = (v.hi < 0) ? 0xFFFFFFFFu : 0u;
    uint32_t w[5];
    uint32_t src[5] = {(uint32_t)v.lo, (uint32_t)(v.lo >> 32), (uint32_t)v.hi, (uint32_t)((uint64_t)v.hi >> 32), ext};
    for (int i = 0; i < 5; ++i)
      w[i] = sh ? ((src[i] << sh) | (i ? (src[i - 1] >> (32 - sh)) : 0u)) : src[i];
    uint32_t carry = 0;
    for (int i = li; i < nl; ++i) {
      uint32_t addv = (i - li < 5) ? w[i - li] : ext;
      uint64_t s = (uint64_t)limb[i] + addv + carry;
      limb[i] = (uint32_t)s;
      carry = (uint32_t)(s >> 32);
    }
  }
  bool neg = (limb[nl - 1] >> 31) != 0;
  if (neg) {
    uint32_t c = 1;
    for (int i = 0; i < nl; ++i) {
      uint64_t s = (uint64_t)(~limb[i]) + c;
      limb[i] = (uint32_t)s;
      c = (uint32_t)(s >> 32);
    }
  }
  return round_limbs<T>(neg, limb, nl, beta<T>(st.I + K - 1));
}

// -------------------------------------------- fast conversion (fixed K)
// Correct rounding of sum_k F_k 2^(beta_{I+k}) with compile-time K, in
// registers: the folds are added into a little-endian two's-complement
// integer of NW 32-bit words (bit 0 = the finest grid unit), whose leading
// 64 bits are then rounded to nearest, ties to even, with a sticky bit.
template <typename T, int K> struct ConvW {
  static constexpr int NW = (Geom<T>::W * (K - 1) + 130) / 32 + 1;
};

// w += v * 2^off (v a sign-extended 128-bit value), static offset.
template <int NW, int OFF>
__device__ __forceinline__ void words_add(uint32_t* w, W128 v) {
  constexpr int li = OFF / 32, sh = OFF % 32;
  uint32_t ext = (v.hi < 0) ? 0xFFFFFFFFu : 0u;
  uint32_t s[5] = {(uint32_t)v.lo, (uint32_t)(v.lo >> 32), (uint32_t)v.hi, (uint32_t)((uint64_t)v.hi >> 32), ext};
  uint32_t carry = 0;
#pragma unroll
  for (int i = li; i < NW; ++i) {
    const int r = i - li;
    uint32_t a;
    if (r < 5) a = sh ? ((s[r] << sh) | (r ? (s[r - 1] >> (32 - sh)) : 0u)) : s[r];
    else a = ext;
    uint64_t t = (uint64_t)w[i] + a + carry;
    w[i] = (uint32_t)t;
    carry = (uint32_t)(t >> 32);
  }
}

template <typename T, int K, int k>
struct FoldAdder {
  template <int NW>
  __device__ __forceinline__ static void run(uint32_t* w, const W128* F) {
    words_add<NW, Geom<T>::W * (K - 1 - k)>(w, F[k]);
    FoldAdder<T, K, k + 1>::template run<NW>(w, F);
  }
};
template <typename T, int K>
struct FoldAdder<T, K, K> {
  template <int NW>
  __device__ __forceinline__ static void run(uint32_t*, const W128*) {}
};

template <typename T, int K>
__device__ __forceinline__ T convert_fast(int I, int flags, const W128* F) {
  typedef Geom<T> G;
  constexpr int NW = ConvW<T, K>::NW;
  if (flags) return from_flags<T>(flags);
  uint32_t w[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) w[i] = 0;
  FoldAdder<T, K, 0>::template run<NW>(w, F);
  bool neg = (w[NW - 1] >> 31) != 0;
  if (neg) {
    uint32_t c = 1;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      uint64_t t = (uint64_t)(~w[i]) + c;
      w[i] = (uint32_t)t;
      c = (uint32_t)(t >> 32);
    }
  }
  // leading word and the 64 bits from the leading bit down (a, b, c words)
  int ti = -1;
#pragma unroll
  for (int i = 0; i < NW; ++i)
    if (w[i]) ti = i;
  if (ti < 0) return (T)0.0;
  uint32_t a = 0, b = 0, c = 0;
  bool below = false;   // any set bit in the words under c
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    if (i == ti) a = w[i];
    if (i == ti - 1) b = w[i];
    if (i == ti - 2) c = w[i];
    if (i < ti - 2 && w[i]) below = true;
  }
  int lz = __clz((int)a);
  // top 64 bits: a:b:c shifted left by lz
  uint64_t hi64 = ((uint64_t)a << 32 | b);
  uint64_t top = lz ? ((hi64 << lz) | ((uint64_t)c >> (32 - lz))) : hi64;
  bool st0 = lz ? ((c << lz) != 0) : (c != 0);
  int topbit = 32 * ti + 31 - lz;            // index of the leading bit
  int lsb = beta<T>(I + K - 1);
  int E = topbit + lsb;
  int q = E - G::P + 1;
  if (q < G::QMIN) q = G::QMIN;
  int drop = q - (topbit - 63 + lsb);          // low bits of `top` below the quantum (>= 64 - P)
  uint64_t m;
  bool half, sticky;
  if (drop >= 64) {
    // value below half the smallest quantum cannot occur for a binned value
    m = 0;
    half = (drop == 64) ? ((top >> 63) != 0) : false;
    sticky = st0 || below || (drop == 64 ? ((top << 1) != 0) : (top != 0));
  } else if (drop > 0) {
    m = top >> drop;
    half = ((top >> (drop - 1)) & 1) != 0;
    sticky = st0 || below || ((drop >= 2) ? ((top << (65 - drop)) != 0) : false);
  } else {
    m = top << (-drop);     // every bit kept (few significant bits)
    half = false;
    sticky = false;
  }
  if (half && (sticky || (m & 1))) m += 1;
  if (m == (1ull << G::P)) { m >>= 1; q += 1; }
  return assemble<T>(neg, m, q);
}

}  // namespace repro
