// Binned cumulative sum (SyclReproSum, "How It Works", cumsum
// paragraph): contiguous tiles are reduced to binned totals, the totals are
// scanned exclusively in binned form, and each tile is replayed from its
// incoming state, converting every prefix.  Only tile totals and tile
// prefixes are stored.  Each output uses the index of its own prefix, so
// every prefix is bit-identical for any launch shape and out[n-1] equals the
// binned sum.
#include "accum.cuh"
#include "launch.h"

namespace repro {

constexpr int CS_BLOCK = 256;
constexpr int CS_ITEMS = 16;
constexpr int CS_TILE = CS_BLOCK * CS_ITEMS;

// Tile staging: coalesced copy of the tile into shared memory, thread t then
// owns elements [t * ITEMS, (t + 1) * ITEMS) of it.
template <typename T>
__device__ __forceinline__ int load_tile(const T* __restrict__ in, int64_t n, int64_t tile, T* sm) {
  int64_t base = tile * CS_TILE;
  int cnt = (int)min((int64_t)CS_TILE, n - base);
  for (int i = threadIdx.x; i < cnt; i += blockDim.x) sm[i + i / CS_ITEMS] = in[base + i];
  __syncthreads();
  return cnt;
}

// ------------------------------------------------------------------
// Compile-time K (2..8): every state lives in registers.
//  A. tile totals: the sum kernel's per-thread accumulators and block merge;
//  B. one block scans the tile totals (per-thread sequential runs, then a
//     warp-shuffle scan of the run totals);
//  C. replay: each thread owns ITEMS contiguous elements; the block scan of
//     the threads' own totals plus the tile prefix gives its incoming state;
//     each element's digits are added to that running state, which is then
//     rounded (convert_fast).
template <int K> struct RS {   // register state: index, flags, 128-bit fold sums
  int I;
  int flags;
  W128 F[K];
};

template <int K>
__device__ __forceinline__ void rs_zero(RS<K>& s, int I0) {
  s.I = I0;
  s.flags = 0;
#pragma unroll
  for (int k = 0; k < K; ++k) s.F[k] = W128{0, 0};
}

template <int K>
__device__ __forceinline__ void rs_shift(RS<K>& s, int d) {
  // re-express at index s.I - d (d >= 0): fold k -> k + d
#pragma unroll
  for (int k = K - 1; k >= 0; --k) {
    W128 v = W128{0, 0};
#pragma unroll
    for (int j = 0; j < K; ++j)
      if (j == k - d) v = s.F[j];
    s.F[k] = v;
  }
}

template <int K>
__device__ __forceinline__ void rs_merge(RS<K>& a, const RS<K>& b) {
  RS<K> t = b;
  if (b.I < a.I) { rs_shift(a, a.I - b.I); a.I = b.I; }
  else if (a.I < b.I) { rs_shift(t, b.I - a.I); }
#pragma unroll
  for (int k = 0; k < K; ++k) a.F[k] = w_add(a.F[k], t.F[k]);
  a.flags |= b.flags;
}

template <int K>
__device__ __forceinline__ RS<K> rs_shfl_up(const RS<K>& s, int d) {
  RS<K> o;
  o.I = __shfl_up_sync(0xffffffffu, s.I, d);
  o.flags = __shfl_up_sync(0xffffffffu, s.flags, d);
#pragma unroll
  for (int k = 0; k < K; ++k) o.F[k] = shfl_up_w(s.F[k], d);
  return o;
}

template <int K>
__device__ __forceinline__ void rs_load(RS<K>& s, const unsigned char* p) {
  s.I = ((const int*)p)[0];
  s.flags = ((const int*)p)[1];
  const int64_t* F = (const int64_t*)(p + 16);
#pragma unroll
  for (int k = 0; k < K; ++k) s.F[k] = W128{(uint64_t)F[2 * k], F[2 * k + 1]};
}

template <int K>
__device__ __forceinline__ void rs_store(const RS<K>& s, unsigned char* p) {
  ((int*)p)[0] = s.I;
  ((int*)p)[1] = s.flags;
  int64_t* F = (int64_t*)(p + 16);
#pragma unroll
  for (int k = 0; k < K; ++k) { F[2 * k] = (int64_t)s.F[k].lo; F[2 * k + 1] = s.F[k].hi; }
}

// Exclusive block scan of register states (identity at index I0).
template <int K>
__device__ __forceinline__ RS<K> rs_block_exclusive(const RS<K>& mine, int I0, RS<K>* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  RS<K> inc = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    RS<K> o = rs_shfl_up(inc, d);
    if (lane >= d) {
      rs_merge(o, inc);
      inc = o;
    }
  }
  RS<K> exc = rs_shfl_up(inc, 1);
  if (lane == 0) rs_zero(exc, I0);
  if (lane == 31) sm[warp] = inc;
  __syncthreads();
  RS<K> base;
  rs_zero(base, I0);
  for (int w = 0; w < warp; ++w) rs_merge(base, sm[w]);
  rs_merge(base, exc);
  __syncthreads();
  return base;
}

// Digits of one finite element at index I (compile-time K).
template <typename T, int K> struct Digits;
template <int K> struct Digits<float, K> {
  float P0[K];
  uint32_t thr;
  float thrf;
  __device__ __forceinline__ void set(int I) {
    thr = index_threshold<float>(I);
    thrf = (I == 0) ? 0.0f : __uint_as_float(thr);
#pragma unroll
    for (int k = 0; k < K; ++k)
      P0[k] = (I >= 1) ? __uint_as_float(((uint32_t)(beta<float>(I + k) + 23 + 127) << 23) | 0x400000u) : 1.0f;
  }
  __device__ __forceinline__ bool fits(float x) const { return fabsf(x) < thrf; }
  // exact digits through fresh primaries (the SyclReproSum sticky-bit deposit)
  __device__ __forceinline__ void get(float x, int I, int64_t* a) const {
    float r = x;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      float q = __uint_as_float(__float_as_uint(r) | 1u);
      float S = __fadd_rn(P0[k], q);
      a[k] = (int32_t)(__float_as_uint(S) - __float_as_uint(P0[k]));
      if (k + 1 < K) r = __fadd_rn(r, __fsub_rn(P0[k], S));
    }
  }
};
template <int K> struct Digits<double, K> {
  FastD<K> fc;
  uint32_t thr_hi;
  __device__ __forceinline__ void set(int I) {
    fc.set(I);
    thr_hi = (uint32_t)(index_threshold<double>(I) >> 32);
  }
  __device__ __forceinline__ bool fits(double x) const {
    return ((uint32_t)__double2hiint(x) & 0x7FFFFFFFu) < thr_hi;
  }
  __device__ __forceinline__ void get(double x, int I, int64_t* a) const { fast_digits_f64<K>(x, fc, a); }
};

// Deposit x into a running register state.
template <typename T, int K>
__device__ __forceinline__ void rs_deposit(RS<K>& s, Digits<T, K>& dg, T x) {
  if (!dg.fits(x)) {
    if (!(abs_bits<T>(x) < (sizeof(T) == 4 ? 0x7F800000ull : 0x7FF0000000000000ull))) {
      s.flags |= special_flag(x);
      return;
    }
    if (x == (T)0) return;
    int j = bin_index<T>(x);
    if (j < s.I) {
      rs_shift(s, s.I - j);
      s.I = j;
      dg.set(j);
    }
    if (sizeof(T) == 4 && s.I == 0) {
      // bin 0: the float primary would overflow; exact integer digits
      int64_t a[K];
      chain_digits<T>(x, s.I, K, a);
#pragma unroll
      for (int k = 0; k < K; ++k) s.F[k] = w_add(s.F[k], w_from(a[k]));
      return;
    }
  }
  int64_t a[K];
  dg.get(x, s.I, a);
#pragma unroll
  for (int k = 0; k < K; ++k) s.F[k] = w_add(s.F[k], w_from(a[k]));
}

// A gate (when not null) makes a kernel a fallback that runs only when the
// fast path before it asked for it: the kernel may start early (programmatic
// stream serialization) and waits for that grid before it reads the gate.
__device__ __forceinline__ bool cs_gated_off(const unsigned* gate) {
  if (!gate) return false;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  return *gate == 0u;
}

template <typename T, int KT>
__global__ void __launch_bounds__(CS_BLOCK) cumsum_fast_reduce(const T* __restrict__ in, int64_t n, int K,
                                                               unsigned char* __restrict__ tstate,
                                                               const unsigned* gate) {
  typedef typename AccOf<T, KT>::type Acc;
  if (cs_gated_off(gate)) return;
  const int64_t nt = (n + CS_TILE - 1) / CS_TILE;
  for (int64_t tile = blockIdx.x; tile < nt; tile += gridDim.x) {
    int64_t base = tile * CS_TILE;
    int64_t cnt = min((int64_t)CS_TILE, n - base);
    Acc acc;
    acc.init(K);
    const T* p = in + base;
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
      T v[1] = {p[i]};
      acc.template chunk<1>(v);
    }
    acc.finish();
    State<KT> st;
    block_merge<KT>(acc.I, acc.flags, acc.L, K, &st);
    if (threadIdx.x == 0) store_partial<KT>(tstate, (int)tile, K, st);
  }
}

// carry: null, or a binned state in the repro_state layout (32-byte header
// {index, flags, K, type}, then K 128-bit folds) that every prefix includes;
// a header that is not a state of this K and type gives the canonical NaN.
template <typename T>
__device__ __forceinline__ int carry_flags(const unsigned char* p, int K) {
  const int* h = (const int*)p;
  return h[1] | ((h[2] != K || h[3] != (sizeof(T) == 8 ? 2 : 1)) ? FL_NAN : 0);
}

template <typename T, int KT>
__device__ __forceinline__ void rs_from_carry(RS<KT>& s, const unsigned char* p) {
  rs_zero(s, Geom<T>::NB - KT);
  s.flags = carry_flags<T>(p, KT);
  if (s.flags & FL_NAN) return;   // no fold is read from a state of another K or type
  s.I = ((const int*)p)[0];
  const int64_t* F = (const int64_t*)(p + 32);
#pragma unroll
  for (int k = 0; k < KT; ++k) s.F[k] = W128{(uint64_t)F[2 * k], F[2 * k + 1]};
}

template <typename T, int KT>
__global__ void __launch_bounds__(1024) cumsum_fast_scan(const unsigned char* __restrict__ tstate, int64_t ntiles,
                                                         unsigned char* __restrict__ tpref, const unsigned* gate,
                                                         const unsigned char* __restrict__ carry) {
  __shared__ RS<KT> sm[32];
  if (cs_gated_off(gate)) return;
  const int I0 = Geom<T>::NB - KT;
  const size_t st = 16 + 16 * (size_t)KT;
  int64_t per = (ntiles + blockDim.x - 1) / blockDim.x;
  int64_t b = (int64_t)threadIdx.x * per, e = min(ntiles, b + per);
  RS<KT> agg, x;
  rs_zero(agg, I0);
  for (int64_t t = b; t < e; ++t) {
    rs_load(x, tstate + (size_t)t * st);
    rs_merge(agg, x);
  }
  RS<KT> run = rs_block_exclusive<KT>(agg, I0, sm);
  if (carry) {
    RS<KT> c;
    rs_from_carry<T, KT>(c, carry);
    rs_merge(run, c);
  }
  for (int64_t t = b; t < e; ++t) {
    rs_store(run, tpref + (size_t)t * st);
    rs_load(x, tstate + (size_t)t * st);
    rs_merge(run, x);
  }
}

// First level of the tile scan: block b scans tiles [256 b, 256 b + 256),
// one per thread, into prefixes within its segment and writes the
// segment's total (states past the last tile are zero, the merge identity).
// cumsum_fast_scan then scans the segment totals, and the replay merges
// both prefixes: binned merges are exact, so the order does not matter.
constexpr int CS_SEG = 256;
template <typename T, int KT>
__global__ void __launch_bounds__(CS_SEG) cumsum_seg_scan(const unsigned char* __restrict__ tstate, int64_t ntiles,
                                                          unsigned char* __restrict__ tpref,
                                                          unsigned char* __restrict__ segtot, const unsigned* gate) {
  __shared__ RS<KT> sm[32];
  if (cs_gated_off(gate)) return;
  const int I0 = Geom<T>::NB - KT;
  const size_t st = 16 + 16 * (size_t)KT;
  const int64_t t = (int64_t)blockIdx.x * CS_SEG + threadIdx.x;
  RS<KT> x;
  rs_zero(x, I0);
  if (t < ntiles) rs_load(x, tstate + (size_t)t * st);
  RS<KT> exc = rs_block_exclusive<KT>(x, I0, sm);
  if (t < ntiles) rs_store(exc, tpref + (size_t)t * st);
  if (threadIdx.x == CS_SEG - 1) {
    rs_merge(exc, x);
    rs_store(exc, segtot + (size_t)blockIdx.x * st);
  }
}

template <typename T, int KT>
__device__ __forceinline__ void cumsum_replay_tile(const T* in, T* out, int64_t n, int64_t tile,
                                                   const unsigned char* __restrict__ tpref,
                                                   const unsigned char* __restrict__ segpref, T* sm, RS<KT>* wsm) {
  const int I0 = Geom<T>::NB - KT;
  int cnt = load_tile<T>(in, n, tile, sm);
  const int b = threadIdx.x * CS_ITEMS;
  const int sb = b + threadIdx.x;    // padded position of this thread's first element
  // this thread's own total, then its incoming state
  RS<KT> mine;
  rs_zero(mine, I0);
  {
    Digits<T, KT> dg;
    dg.set(I0);
#pragma unroll 4
    for (int i = 0; i < CS_ITEMS; ++i)
      if (b + i < cnt) rs_deposit<T, KT>(mine, dg, sm[sb + i]);
  }
  RS<KT> run = rs_block_exclusive<KT>(mine, I0, wsm);
  RS<KT> s, sp;
  rs_load(s, tpref + (size_t)tile * (16 + 16 * (size_t)KT));
  rs_load(sp, segpref + (size_t)(tile / CS_SEG) * (16 + 16 * (size_t)KT));
  rs_merge(s, sp);
  rs_merge(s, run);
  Digits<T, KT> dg;
  dg.set(s.I);
#pragma unroll 4
  for (int i = 0; i < CS_ITEMS; ++i) {
    if (b + i < cnt) {
      rs_deposit<T, KT>(s, dg, sm[sb + i]);
      sm[sb + i] = convert_fast<T, KT>(s.I, s.flags, s.F);
    }
  }
  __syncthreads();
  int64_t base = tile * CS_TILE;
  for (int i = threadIdx.x; i < cnt; i += blockDim.x) out[base + i] = sm[i + i / CS_ITEMS];
  __syncthreads();
}

template <typename T, int KT>
__global__ void __launch_bounds__(CS_BLOCK) cumsum_fast_replay(const T* in, T* out, int64_t n,
                                                               const unsigned char* __restrict__ tpref,
                                                               const unsigned char* __restrict__ segpref,
                                                               const unsigned* gate) {
  __shared__ T sm[CS_TILE + CS_TILE / CS_ITEMS];
  __shared__ RS<KT> wsm[CS_BLOCK / 32];
  if (cs_gated_off(gate)) return;
  const int64_t nt = (n + CS_TILE - 1) / CS_TILE;
  for (int64_t tile = blockIdx.x; tile < nt; tile += gridDim.x)
    cumsum_replay_tile<T, KT>(in, out, n, tile, tpref, segpref, sm, wsm);
}


// ------------------------------------------------------------------
// Run-time K (K > 8): a plain design.  Tile totals come from per-thread int64
// lanes and the exact block merge (as in the sum); the tile scan and the
// replay run on one thread per block with the binned state in shared memory.
template <typename T> struct GState {
  static constexpr int N = KMax<T>::V;
  int I;
  int flags;
  uint64_t lo[N];
  int64_t hi[N];
  int64_t dg[N];
  uint32_t limb[ConvLimbs<T>::N];
};

template <typename T>
__device__ void gs_zero(GState<T>* s, int K) {
  s->I = Geom<T>::NB - K;
  s->flags = 0;
  for (int k = 0; k < K; ++k) { s->lo[k] = 0; s->hi[k] = 0; }
}

template <typename T>
__device__ void gs_add(GState<T>* s, int k, W128 v) {
  W128 r = w_add(W128{s->lo[k], s->hi[k]}, v);
  s->lo[k] = r.lo;
  s->hi[k] = r.hi;
}

// Re-express at the coarser index j < s->I (descending, in place: every
// read index is below the written one).
template <typename T>
__device__ void gs_raise(GState<T>* s, int j, int K) {
  int d = s->I - j;
  for (int k = K - 1; k >= 0; --k) {
    if (k >= d) { s->lo[k] = s->lo[k - d]; s->hi[k] = s->hi[k - d]; }
    else { s->lo[k] = 0; s->hi[k] = 0; }
  }
  s->I = j;
}

// s <- merge(s, state stored at p)
template <typename T>
__device__ void gs_merge_stored(GState<T>* s, const unsigned char* p, int K) {
  int Ib = ((const int*)p)[0];
  if (Ib < s->I) gs_raise(s, Ib, K);
  int d = Ib - s->I;
  s->flags |= ((const int*)p)[1];
  const int64_t* F = (const int64_t*)(p + 16);
  for (int k = d; k < K; ++k) gs_add(s, k, W128{(uint64_t)F[2 * (k - d)], F[2 * (k - d) + 1]});
}

template <typename T>
__device__ void gs_store(const GState<T>* s, unsigned char* p, int K) {
  ((int*)p)[0] = s->I;
  ((int*)p)[1] = s->flags;
  int64_t* F = (int64_t*)(p + 16);
  for (int k = 0; k < K; ++k) { F[2 * k] = (int64_t)s->lo[k]; F[2 * k + 1] = s->hi[k]; }
}

template <typename T>
__device__ void gs_deposit(GState<T>* s, T x, int K) {
  uint64_t a = abs_bits<T>(x);
  if (a >= (sizeof(T) == 4 ? 0x7F800000ull : 0x7FF0000000000000ull)) {
    s->flags |= special_flag(x);
    return;
  }
  if (x == (T)0) return;
  int j = bin_index<T>(x);
  if (j < s->I) gs_raise(s, j, K);
  chain_digits<T>(x, s->I, K, s->dg);
  for (int k = 0; k < K; ++k) gs_add(s, k, w_from(s->dg[k]));
}

// Correct rounding of the state (same arithmetic as convert_state, limbs in
// the shared state).
template <typename T>
__device__ T gs_value(GState<T>* s, int K) {
  typedef Geom<T> G;
  if (s->flags) return from_flags<T>(s->flags);
  constexpr int NLMAX = ConvLimbs<T>::N;
  int nl = (G::W * (K - 1) + 134) / 32 + 2;
  if (nl > NLMAX) nl = NLMAX;
  uint32_t* limb = s->limb;
  for (int i = 0; i < nl; ++i) limb[i] = 0;
  for (int k = 0; k < K; ++k) {
    uint64_t vlo = s->lo[k];
    int64_t vhi = s->hi[k];
    if (vlo == 0 && vhi == 0) continue;
    int off = G::W * (K - 1 - k);
    int li = off >> 5, sh = off & 31;
    uint32_t ext = (vhi < 0) ? 0xFFFFFFFFu : 0u;
    uint32_t src[5] = {(uint32_t)vlo, (uint32_t)(vlo >> 32), (uint32_t)vhi, (uint32_t)((uint64_t)vhi >> 32), ext};
    uint32_t carry = 0;
    for (int i = li; i < nl; ++i) {
      int r = i - li;
      uint32_t addv;
      if (r < 5) addv = sh ? ((src[r] << sh) | (r ? (src[r - 1] >> (32 - sh)) : 0u)) : src[r];
      else addv = ext;
      uint64_t t = (uint64_t)limb[i] + addv + carry;
      limb[i] = (uint32_t)t;
      carry = (uint32_t)(t >> 32);
    }
  }
  bool neg = (limb[nl - 1] >> 31) != 0;
  if (neg) {
    uint32_t c = 1;
    for (int i = 0; i < nl; ++i) {
      uint64_t t = (uint64_t)(~limb[i]) + c;
      limb[i] = (uint32_t)t;
      c = (uint32_t)(t >> 32);
    }
  }
  return round_limbs<T>(neg, limb, nl, beta<T>(s->I + K - 1));
}

template <typename T>
__global__ void __launch_bounds__(CS_BLOCK) cumsum_generic_reduce(const T* __restrict__ in, int64_t n, int K,
                                                                  unsigned char* __restrict__ tstate) {
  typedef typename AccOf<T, 0>::type Acc;
  constexpr int N = Acc::N;
  int64_t base = (int64_t)blockIdx.x * CS_TILE;
  int64_t cnt = min((int64_t)CS_TILE, n - base);
  Acc acc;
  acc.init(K);
  for (int64_t i = threadIdx.x; i < cnt; i += blockDim.x) {
    T v[1] = {in[base + i]};
    acc.template chunk<1>(v);
  }
  acc.finish();
  State<N> st;
  block_merge<N>(acc.I, acc.flags, acc.L, K, &st);
  if (threadIdx.x == 0) store_partial<N>(tstate, blockIdx.x, K, st);
}

template <typename T>
__global__ void cumsum_generic_scan(const unsigned char* __restrict__ tstate, int64_t ntiles, int K,
                                    unsigned char* __restrict__ tpref, const unsigned char* __restrict__ carry) {
  __shared__ GState<T> s;
  if (threadIdx.x != 0) return;
  const size_t st = 16 + 16 * (size_t)K;
  gs_zero(&s, K);
  if (carry) {
    // the carried state, restated in the tile-state layout (header, folds)
    const int fl = carry_flags<T>(carry, K);
    if (fl & FL_NAN) {
      s.flags |= fl;
    } else {
      const int Ic = ((const int*)carry)[0];
      if (Ic < s.I) gs_raise(&s, Ic, K);
      s.flags |= fl;
      const int64_t* F = (const int64_t*)(carry + 32);
      const int d = Ic - s.I;
      for (int k = d; k < K; ++k) gs_add(&s, k, W128{(uint64_t)F[2 * (k - d)], F[2 * (k - d) + 1]});
    }
  }
  for (int64_t t = 0; t < ntiles; ++t) {
    gs_store(&s, tpref + (size_t)t * st, K);
    gs_merge_stored(&s, tstate + (size_t)t * st, K);
  }
}

template <typename T>
__global__ void cumsum_generic_replay(const T* in, T* out, int64_t n, int K, const unsigned char* __restrict__ tpref) {
  __shared__ GState<T> s;
  if (threadIdx.x != 0) return;
  const size_t st = 16 + 16 * (size_t)K;
  int64_t base = (int64_t)blockIdx.x * CS_TILE;
  int64_t cnt = min((int64_t)CS_TILE, n - base);
  gs_zero(&s, K);
  gs_merge_stored(&s, tpref + (size_t)blockIdx.x * st, K);
  for (int64_t i = 0; i < cnt; ++i) {
    gs_deposit(&s, in[base + i], K);
    out[base + i] = gs_value(&s, K);
  }
}

template <typename T>
size_t cumsum_workspace_bytes(int64_t n, int K) {
  if (K == 3) return cumsum_k3_workspace_bytes<T>(n);
  if (sizeof(T) == 8 && K >= 4 && K <= 6) return cumsum_fx_workspace_bytes(n, K);
  int64_t nt = (n + CS_TILE - 1) / CS_TILE;
  int64_t nseg = (nt + CS_SEG - 1) / CS_SEG;
  return 2 * (size_t)(nt + nseg) * (16 + 16 * (size_t)K) + 64;   // tile and segment states and prefixes
}

template <typename Kn, typename... A>
static cudaError_t cs_launch(Kn kernel, int64_t grid, int block, cudaStream_t s, bool pdl, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

static int cs_sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 1;
  }
  if (!cached[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
      cudaGetLastError();
      v = 1;
    }
    cached[dev] = v;
  }
  return cached[dev];
}

// gate: null, or a device word that a fast path before these kernels sets
// to nonzero when they must run (otherwise they return at once; their grids
// are then kept to a few blocks per SM, each walking several tiles).
template <typename T, int KT>
static cudaError_t launch_cumsum_k(const T* in, T* out, int64_t n, int K, unsigned char* ws, cudaStream_t s,
                                   const unsigned* gate = nullptr, const unsigned char* carry = nullptr) {
  int64_t nt = (n + CS_TILE - 1) / CS_TILE;
  int64_t nseg = (nt + CS_SEG - 1) / CS_SEG;
  const size_t st = 16 + 16 * (size_t)K;
  unsigned char* tstate = ws;
  unsigned char* tpref = tstate + (size_t)nt * st;
  unsigned char* segtot = tpref + (size_t)nt * st;
  unsigned char* segpref = segtot + (size_t)nseg * st;
  const bool pdl = gate != nullptr;
  const int64_t grid = pdl ? min(nt, (int64_t)4 * cs_sm_count()) : nt;
  cudaError_t e;
  if ((e = cs_launch(cumsum_fast_reduce<T, KT>, grid, CS_BLOCK, s, pdl, in, n, K, tstate, gate)) != cudaSuccess)
    return e;
  if ((e = cs_launch(cumsum_seg_scan<T, KT>, nseg, CS_SEG, s, pdl, (const unsigned char*)tstate, nt, tpref, segtot,
                     gate)) != cudaSuccess)
    return e;
  if ((e = cs_launch(cumsum_fast_scan<T, KT>, 1, 1024, s, pdl, (const unsigned char*)segtot, nseg, segpref,
                     gate, carry)) != cudaSuccess)
    return e;
  return cs_launch(cumsum_fast_replay<T, KT>, grid, CS_BLOCK, s, pdl, in, out, n, (const unsigned char*)tpref,
                   (const unsigned char*)segpref, gate);
}

template <typename T>
cudaError_t launch_cumsum_general(const T* in, T* out, int64_t n, int K, unsigned char* ws, cudaStream_t s,
                                  const unsigned* gate) {
  switch (K) {
    case 4: return launch_cumsum_k<T, 4>(in, out, n, K, ws, s, gate);
    case 5: return launch_cumsum_k<T, 5>(in, out, n, K, ws, s, gate);
    case 6: return launch_cumsum_k<T, 6>(in, out, n, K, ws, s, gate);
    default: return cudaErrorInvalidValue;
  }
}
template cudaError_t launch_cumsum_general<double>(const double*, double*, int64_t, int, unsigned char*,
                                                   cudaStream_t, const unsigned*);

size_t cumsum_general_bytes(int64_t n, int K) {
  int64_t nt = (n + CS_TILE - 1) / CS_TILE;
  int64_t nseg = (nt + CS_SEG - 1) / CS_SEG;
  return 2 * (size_t)(nt + nseg) * (16 + 16 * (size_t)K) + 64;   // tile and segment states and prefixes
}

template <typename T>
static cudaError_t launch_cumsum_generic(const T* in, T* out, int64_t n, int K, unsigned char* ws, cudaStream_t s,
                                         const unsigned char* carry) {
  int64_t nt = (n + CS_TILE - 1) / CS_TILE;
  unsigned char* tstate = ws;
  unsigned char* tpref = ws + (size_t)nt * (16 + 16 * (size_t)K);
  cumsum_generic_reduce<T><<<(unsigned)nt, CS_BLOCK, 0, s>>>(in, n, K, tstate);
  cumsum_generic_scan<T><<<1, 32, 0, s>>>(tstate, nt, K, tpref, carry);
  cumsum_generic_replay<T><<<(unsigned)nt, 32, 0, s>>>(in, out, n, K, tpref);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_cumsum(const T* in, T* out, int64_t n, int K, unsigned char* ws, unsigned char* zc, cudaStream_t s,
                          const unsigned char* carry) {
  switch (K) {
    case 2: return launch_cumsum_k<T, 2>(in, out, n, K, ws, s, nullptr, carry);
    case 3: return launch_cumsum_k3<T>(in, out, n, ws, zc, s, carry);
    case 4:
    case 5:
    case 6:
      if constexpr (sizeof(T) == 8) {
        if (!carry) return launch_cumsum_fx(in, out, n, K, ws, zc, s);
      }
      if (K == 4) return launch_cumsum_k<T, 4>(in, out, n, K, ws, s, nullptr, carry);
      if (K == 5) return launch_cumsum_k<T, 5>(in, out, n, K, ws, s, nullptr, carry);
      return launch_cumsum_k<T, 6>(in, out, n, K, ws, s, nullptr, carry);
    case 7: return launch_cumsum_k<T, 7>(in, out, n, K, ws, s, nullptr, carry);
    case 8: return launch_cumsum_k<T, 8>(in, out, n, K, ws, s, nullptr, carry);
    default: return launch_cumsum_generic<T>(in, out, n, K, ws, s, carry);
  }
}

// Workspace of a cumulative sum with a carried state (the general kernels).
template <typename T>
size_t cumsum_carry_workspace_bytes(int64_t n, int K) {
  if (K == 3) return cumsum_k3_general_bytes<T>(n);
  if (sizeof(T) == 8 && K >= 4 && K <= 6) return cumsum_general_bytes(n, K);
  return cumsum_workspace_bytes<T>(n, K);
}
template size_t cumsum_carry_workspace_bytes<float>(int64_t, int);
template size_t cumsum_carry_workspace_bytes<double>(int64_t, int);

template size_t cumsum_workspace_bytes<float>(int64_t, int);
template size_t cumsum_workspace_bytes<double>(int64_t, int);
template cudaError_t launch_cumsum<float>(const float*, float*, int64_t, int, unsigned char*, unsigned char*,
                                          cudaStream_t, const unsigned char*);
template cudaError_t launch_cumsum<double>(const double*, double*, int64_t, int, unsigned char*, unsigned char*,
                                           cudaStream_t, const unsigned char*);

}  // namespace repro
