// Per-thread binned accumulators and exact block / grid merges.
#pragma once
#include "adn.cuh"

namespace repro {

constexpr int KMAX_F = 21;
constexpr int KMAX_D = 52;
template <typename T> struct KMax;
template <> struct KMax<float> { static constexpr int V = KMAX_F; };
template <> struct KMax<double> { static constexpr int V = KMAX_D; };

// Compile-time fold count KT (2..8) or KT == 0 for a run-time K (arrays sized
// for the largest K of the type).
template <typename T, int KT> struct KArr { static constexpr int N = KT ? KT : KMax<T>::V; };

// ----------------------------------------------------------------- lanes
// Integer lanes: fold sums of one thread in units of the fold's grid.
template <typename T, int KT>
struct Lanes {
  static constexpr int N = KArr<T, KT>::N;
  int I;
  int flags;
  int K;
  int64_t L[N];

  __device__ __forceinline__ int nk() const { return KT ? KT : K; }

  __device__ __forceinline__ void init(int Kr) {
    K = Kr;
    I = Geom<T>::NB - nk();
    flags = 0;
#pragma unroll(N <= 8 ? N : 1)
    for (int k = 0; k < N; ++k) L[k] = 0;
  }

  // Move to the coarser index j < I (exact re-expression, see shift_folds).
  __device__ __forceinline__ void raise_lanes(int j) {
    int d = I - j;
    if (KT) {
      // repeated single steps keep register indexing static
      for (int s = 0; s < d && s < N; ++s) {
#pragma unroll
        for (int k = N - 1; k > 0; --k) L[k] = L[k - 1];
        L[0] = 0;
      }
    } else {
      shift_folds<int64_t, KT>(L, nk(), d);
    }
    I = j;
  }

  __device__ __forceinline__ void add_digits(T x) {
    int64_t a[N];
    chain_digits<T>(x, I, nk(), a);
#pragma unroll(N <= 8 ? N : 1)
    for (int k = 0; k < N; ++k)
      if (k < nk()) L[k] += a[k];
  }
};

// --------------------------------------------------- float primary form
// Floating-point primaries ("SyclReproSum", "How It Works": deposit with the sticky
// bit, renormalise), one per fold, each with ulp equal to the fold's grid:
// P starts at 1.5 * 2^e, and a deposit S = P + sticky(r) rounds r on the grid
// with ties away from zero; r + (P - S) is the exact remainder.  Every <= 512
// deposits the primaries are flushed into the integer lanes (the drift of P
// stays within its binade: 512 * 2^(W-1) ulps < 2^(p-2) ulps).  Bin 0 would
// need an overflowing primary, so a thread at index 0 uses integer digits.
template <int KT>
struct AccF : Lanes<float, KT> {
  typedef Lanes<float, KT> B;
  static constexpr int N = B::N;
  float P[N];
  float P0[N];
  uint32_t thr;
  float thrf;
  int cnt;

  __device__ __forceinline__ static float primary0(int j) {
    // 1.5 * 2^(beta_j + 23), j >= 1
    return __uint_as_float(((uint32_t)(beta<float>(j) + 23 + 127) << 23) | 0x400000u);
  }

  __device__ __forceinline__ void set_index_consts() {
    thr = index_threshold<float>(this->I);
    thrf = (this->I == 0) ? 0.0f : __uint_as_float(thr);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      if (k < this->nk()) {
        P0[k] = (this->I >= 1) ? primary0(this->I + k) : 1.0f;
        P[k] = P0[k];
      }
    }
  }

  __device__ __forceinline__ void init(int Kr) {
    B::init(Kr);
    cnt = 0;
    set_index_consts();
  }

  __device__ __forceinline__ void flush() {
    if (this->I >= 1) {
#pragma unroll
      for (int k = 0; k < N; ++k) {
        if (k < this->nk()) {
          // same binade: the bit difference is the deviation in ulps
          this->L[k] += (int64_t)((int32_t)(__float_as_uint(P[k]) - __float_as_uint(P0[k])));
          P[k] = P0[k];
        }
      }
    }
    cnt = 0;
  }

  __device__ __forceinline__ void raise(int j) {
    flush();
    this->raise_lanes(j);
    set_index_consts();
  }

  __device__ __forceinline__ void deposit_fp(float x) {
    float r = x;
#pragma unroll
    for (int k = 0; k < N; ++k) {
      if (k < this->nk()) {
        float q = __uint_as_float(__float_as_uint(r) | 1u);
        float S = __fadd_rn(P[k], q);
        if (k + 1 < this->nk()) r = __fadd_rn(r, __fsub_rn(P[k], S));
        P[k] = S;
      }
    }
  }

  // A chunk where some value may lie above the current bins or be Inf/NaN.
  template <int U>
  __device__ __forceinline__ void slow_chunk(float* v) {
    int jmin = this->I;
#pragma unroll
    for (int i = 0; i < U; ++i) {
      float x = v[i];
      if (!(fabsf(x) < thrf) && !(this->I == 0 && fabsf(x) <= 3.4028235e38f)) {
        if (!(fabsf(x) <= 3.4028235e38f)) {
          this->flags |= special_flag(x);
          v[i] = 0.0f;
        } else {
          int j = bin_index<float>(x);
          jmin = j < jmin ? j : jmin;
        }
      }
    }
    if (jmin < this->I) raise(jmin);
    if (this->I >= 1) {
#pragma unroll
      for (int i = 0; i < U; ++i) deposit_fp(v[i]);
      cnt += U;
      if (cnt >= 512 - U) flush();
    } else {
#pragma unroll
      for (int i = 0; i < U; ++i) this->add_digits(v[i]);
    }
  }

  template <int U>
  __device__ __forceinline__ void chunk(float* v) {
    bool out = false;
#pragma unroll
    for (int i = 0; i < U; ++i) out |= !(fabsf(v[i]) < thrf);
    if (out) {
      slow_chunk<U>(v);
    } else {
#pragma unroll
      for (int i = 0; i < U; ++i) deposit_fp(v[i]);
      cnt += U;
      if (cnt >= 512 - U) flush();
    }
  }

  __device__ __forceinline__ void finish() { flush(); }
};

// ------------------------------------------------------- double lane form
template <int KT>
struct AccD : Lanes<double, KT> {
  typedef Lanes<double, KT> B;
  static constexpr int N = B::N;
  uint64_t thr;
  FastD<KT ? KT : 1> fc;

  __device__ __forceinline__ void init(int Kr) {
    B::init(Kr);
    thr = index_threshold<double>(this->I);
    if (KT) fc.set(this->I);
  }

  __device__ __forceinline__ void raise(int j) {
    this->raise_lanes(j);
    thr = index_threshold<double>(this->I);
    if (KT) fc.set(this->I);
  }

  __device__ __forceinline__ void add_fast(double x) {
    if constexpr (KT != 0) {
      int64_t a[KT];
      fast_digits_f64<KT>(x, fc, a);
#pragma unroll
      for (int k = 0; k < KT; ++k) this->L[k] += a[k];
    } else {
      this->add_digits(x);
    }
  }

  template <int U>
  __device__ __forceinline__ void slow_chunk(double* v) {
    int jmin = this->I;
#pragma unroll
    for (int i = 0; i < U; ++i) {
      uint64_t a = abs_bits<double>(v[i]);
      if (a >= thr) {
        if (a >= 0x7FF0000000000000ull) {
          this->flags |= special_flag(v[i]);
          v[i] = 0.0;
        } else {
          int j = bin_index<double>(v[i]);
          jmin = j < jmin ? j : jmin;
        }
      }
    }
    if (jmin < this->I) raise(jmin);
#pragma unroll
    for (int i = 0; i < U; ++i) add_fast(v[i]);
  }

  template <int U>
  __device__ __forceinline__ void chunk(double* v) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < U; ++i) m = max(m, (uint32_t)__double2hiint(v[i]) & 0x7FFFFFFFu);
    if (m >= (uint32_t)(thr >> 32)) {
      slow_chunk<U>(v);
    } else {
#pragma unroll
      for (int i = 0; i < U; ++i) add_fast(v[i]);
    }
  }

  __device__ __forceinline__ void finish() {}
};

template <typename T, int KT> struct AccOf;
template <int KT> struct AccOf<float, KT> { typedef AccF<KT> type; };
template <int KT> struct AccOf<double, KT> { typedef AccD<KT> type; };

// ------------------------------------------------------------ block merge
// Exact merge of every thread's lanes: block-wide minimum index, each thread
// re-expresses its lanes there, 128-bit sums per fold.  Thread 0 receives the
// block state.  Requires blockDim.x a multiple of 32, at most 1024.
template <int N>
__device__ void block_merge(int I, int flags, const int64_t* L, int K, State<N>* out) {
  __shared__ int sI[32];
  __shared__ int sFl[32];
  __shared__ W128 sF[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int wi = __reduce_min_sync(0xffffffffu, I);
  int wf = (int)__reduce_or_sync(0xffffffffu, (unsigned)flags);
  if (lane == 0) { sI[warp] = wi; sFl[warp] = wf; }
  __syncthreads();
  int Ib = sI[0], fb = 0;
  for (int w = 0; w < nw; ++w) { Ib = min(Ib, sI[w]); fb |= sFl[w]; }
  int d = I - Ib;
  if (threadIdx.x == 0) { out->I = Ib; out->flags = fb; }
  for (int k = 0; k < K; ++k) {
    W128 v = w_from(fold_at<N, int64_t>(L, K, k - d));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = w_add(v, shfl_xor_w(v, m));
    __syncthreads();
    if (lane == 0) sF[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
      W128 s = W128{0, 0};
      for (int w = 0; w < nw; ++w) s = w_add(s, sF[w]);
      out->F[k] = s;
    }
  }
  __syncthreads();
}

// Partial states in global memory: per block a 16-byte header (I, flags) and
// K 128-bit fold sums.
__device__ __forceinline__ size_t partial_stride(int K) { return 16 + 16 * (size_t)K; }

template <int N>
__device__ __forceinline__ void store_partial(unsigned char* base, int idx, int K, const State<N>& s) {
  unsigned char* p = base + (size_t)idx * partial_stride(K);
  int* h = (int*)p;
  h[0] = s.I;
  h[1] = s.flags;
  int64_t* F = (int64_t*)(p + 16);
  for (int k = 0; k < K; ++k) {
    F[2 * k] = (int64_t)s.F[k].lo;
    F[2 * k + 1] = s.F[k].hi;
  }
}

}  // namespace repro
