// Binned sum: one read of the input, per-thread binned accumulation, exact
// block merge, and a last-block grid merge + conversion (SyclReproSum,
// "How It Works": deposit, renormalize, merge; the sum reads each input
// element exactly once).  The result bits depend only on the multiset of
// inputs, never on the grid, block size or scheduling.
#include "accum.cuh"
#include "launch.h"

namespace repro {

template <typename T> struct Vec;
template <> struct Vec<float> { typedef float4 type; static constexpr int W = 4; };
template <> struct Vec<double> { typedef double2 type; static constexpr int W = 2; };

template <typename T>
__device__ __forceinline__ void unpack(const typename Vec<T>::type& v, T* out);
template <> __device__ __forceinline__ void unpack<float>(const float4& v, float* o) {
  o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
template <> __device__ __forceinline__ void unpack<double>(const double2& v, double* o) {
  o[0] = v.x; o[1] = v.y;
}

// Streaming loads that bypass L1 allocation (each byte is used once).
__device__ __forceinline__ float4 ldg_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ double2 ldg_stream(const double2* p) { return __ldcs(p); }

// Accumulate x[lo, hi) (any alignment) into acc; thread `t` of `nt`.
// Vector part: U 16-byte vectors per thread per iteration, interleaved so that
// each load instruction of a warp covers contiguous memory.
template <typename T, typename Acc, int U>
__device__ __forceinline__ void accumulate_range(Acc& acc, const T* __restrict__ x, int64_t n, int64_t t,
                                                 int64_t nt) {
  typedef typename Vec<T>::type V;
  constexpr int VW = Vec<T>::W;
  int64_t head = (int64_t)(((16 - ((uintptr_t)x & 15)) & 15) / sizeof(T));
  if (head > n) head = n;
  const V* xv = (const V*)(x + head);
  int64_t nv = (n - head) / VW;
  int64_t i = t;
  const int64_t step = (int64_t)U * nt;
  if (i + (int64_t)(U - 1) * nt < nv) {
    // software pipelined: the next group's loads are in flight while the
    // current group is deposited
    V r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = ldg_stream(xv + i + (int64_t)u * nt);
    for (;;) {
      int64_t inext = i + step;
      bool more = inext + (int64_t)(U - 1) * nt < nv;
      V q[U];
      if (more) {
#pragma unroll
        for (int u = 0; u < U; ++u) q[u] = ldg_stream(xv + inext + (int64_t)u * nt);
      }
      T v[U * VW];
#pragma unroll
      for (int u = 0; u < U; ++u) unpack<T>(r[u], v + u * VW);
      acc.template chunk<U * VW>(v);
      i = inext;
      if (!more) break;
#pragma unroll
      for (int u = 0; u < U; ++u) r[u] = q[u];
    }
  }
  for (; i < nv; i += nt) {
    T v[VW];
    unpack<T>(ldg_stream(xv + i), v);
    acc.template chunk<VW>(v);
  }
  // scalar head and tail elements
  int64_t tail0 = head + nv * VW;
  int64_t ns = head + (n - tail0);
  for (int64_t j = t; j < ns; j += nt) {
    T v[1] = {j < head ? x[j] : x[tail0 + (j - head)]};
    acc.template chunk<1>(v);
  }
}

__device__ __forceinline__ W128 ld_w128_cg(const int64_t* p) {
  longlong2 v = __ldcg((const longlong2*)p);
  return W128{(uint64_t)v.x, (int64_t)v.y};
}

template <int N>
__device__ void merge_partials_cg(const unsigned char* base, int np, int K, State<N>* out);

// Last-block merge of all partial states.  Loads use the L2-coherent path
// since the partials were written by other blocks of this launch.
template <int N>
__device__ void merge_partials_cg(const unsigned char* base, int np, int K, State<N>* out) {
  __shared__ int sI[32];
  __shared__ int sFl[32];
  __shared__ W128 sF[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const size_t st = 16 + 16 * (size_t)K;
  int I = 1 << 30, fl = 0;
  for (int p = threadIdx.x; p < np; p += blockDim.x) {
    const int* h = (const int*)(base + (size_t)p * st);
    I = min(I, __ldcg(h));
    fl |= __ldcg(h + 1);
  }
  int wi = __reduce_min_sync(0xffffffffu, I);
  int wf = (int)__reduce_or_sync(0xffffffffu, (unsigned)fl);
  if (lane == 0) { sI[warp] = wi; sFl[warp] = wf; }
  __syncthreads();
  int Ig = sI[0], fg = 0;
  for (int w = 0; w < nw; ++w) { Ig = min(Ig, sI[w]); fg |= sFl[w]; }
  if (threadIdx.x == 0) { out->I = Ig; out->flags = fg; }
  for (int k = 0; k < K; ++k) {
    W128 v = W128{0, 0};
    for (int p = threadIdx.x; p < np; p += blockDim.x) {
      const unsigned char* q = base + (size_t)p * st;
      int src = k - (__ldcg((const int*)q) - Ig);
      if (src >= 0) v = w_add(v, ld_w128_cg((const int64_t*)(q + 16) + 2 * src));
    }
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

// ------------------------------------------------------------ binned states
// A caller-owned state in device memory (repro_state_* calls): a 32-byte
// header {I, flags, K, kind, count (64-bit), 0} and K fold sums as 128-bit
// integers {lo, hi}.  Merging states aligns them to the coarser index (fold k
// of a state at index Ia moves to k + (Ia - I); the finest ones drop, which
// is exact because a value inside bin Ia has zero pieces on coarser grids)
// and adds the folds: the same operation as the grid merge, so any split of
// the input into deposits and any merge order gives the sum's bits.
constexpr int ST_HDR = 32;
constexpr int FL_STATE_BAD = 8;   // K or element type mismatch: finalizes to NaN

template <typename T> __host__ __device__ constexpr int state_kind() { return sizeof(T) == 4 ? 1 : 2; }

__device__ __forceinline__ W128 state_fold(const unsigned char* sp, int K, int idx) {
  if (idx < 0 || idx >= K) return W128{0, 0};
  const int64_t* f = (const int64_t*)(sp + ST_HDR) + 2 * idx;
  return W128{(uint64_t)f[0], f[1]};
}

// Fold k of a state at index Ifrom expressed at the coarser index I <= Ifrom.
__device__ __forceinline__ W128 fold_shifted(const W128* F, int K, int Ifrom, int I, int k) {
  const int src = k - (Ifrom - I);
  return (src >= 0 && src < K) ? F[src] : W128{0, 0};
}

// dst := dst + (I, flags, F, count); one thread.  A header whose K or kind
// differs from the call's only gets the poison flag: its buffer was sized
// for its own K, so no fold is read or written.
template <typename T>
__device__ void state_add(unsigned char* dst, int K, int I, int flags, const W128* F, uint64_t count) {
  int* h = (int*)dst;
  if (h[2] != K || h[3] != state_kind<T>()) {
    h[1] |= FL_STATE_BAD;
    return;
  }
  W128 old[KMAXS_SHIFT];
  const int Id = h[0];
  const int fl = h[1] | flags;
  for (int k = 0; k < K; ++k) old[k] = state_fold(dst, K, k);
  const int In = min(Id, I);
  int64_t* f = (int64_t*)(dst + ST_HDR);
  for (int k = 0; k < K; ++k) {
    const W128 v = w_add(fold_shifted(old, K, Id, In, k), fold_shifted(F, K, I, In, k));
    f[2 * k] = (int64_t)v.lo;
    f[2 * k + 1] = v.hi;
  }
  h[0] = In;
  h[1] = fl;
  *(unsigned long long*)(dst + 16) += count;
}

template <typename T>
__global__ void state_init_kernel(unsigned char* st, int K) {
  int* h = (int*)st;
  h[0] = Geom<T>::NB - K;   // the empty state's index
  h[1] = 0;
  h[2] = K;
  h[3] = state_kind<T>();
  ((unsigned long long*)st)[2] = 0ull;
  ((unsigned long long*)st)[3] = 0ull;
  int64_t* f = (int64_t*)(st + ST_HDR);
  for (int k = 0; k < 2 * K; ++k) f[k] = 0;
}

template <typename T>
__global__ void state_merge_kernel(unsigned char* dst, const unsigned char* src, int K) {
  W128 F[KMAXS_SHIFT];
  const int* h = (const int*)src;
  if (h[2] != K || h[3] != state_kind<T>()) {   // src sized for another K: no fold is read
    const int* hd = (const int*)dst;
    if (hd[2] == K && hd[3] == state_kind<T>()) ((int*)dst)[1] |= FL_STATE_BAD;
    return;
  }
  for (int k = 0; k < K; ++k) F[k] = state_fold(src, K, k);
  state_add<T>(dst, K, h[0], h[1], F, *(const unsigned long long*)(src + 16));
}

template <typename T>
__global__ void state_finalize_kernel(const unsigned char* st, int K, uint64_t capacity, T* result) {
  const int* h = (const int*)st;
  if (h[2] != K || h[3] != state_kind<T>() || (h[1] & FL_STATE_BAD) ||
      *(const unsigned long long*)(st + 16) > capacity) {
    *result = canonical_nan<T>();
    return;
  }
  State<KMax<T>::V> s;
  s.I = h[0];
  s.flags = h[1];
  for (int k = 0; k < K; ++k) s.F[k] = state_fold(st, K, k);
  *result = convert_state<T, KMax<T>::V>(s, K);
}

// ticket: a counter that is zero at launch, and zero again when the kernel
// ends; parts: one partial state per block.
// With `state`, the merged result is added to that binned state (no
// conversion; `result` unused).
template <typename T, int KT, int U>
__global__ void __launch_bounds__(1024) adn_sum_kernel(const T* __restrict__ x, int64_t n, int K,
                                                       unsigned* ticket, unsigned char* __restrict__ parts,
                                                       T* __restrict__ result, unsigned char* __restrict__ state) {
  typedef typename AccOf<T, KT>::type Acc;
  constexpr int N = Acc::N;
  Acc acc;
  acc.init(K);
  accumulate_range<T, Acc, U>(acc, x, n, (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
                              (int64_t)gridDim.x * blockDim.x);
  acc.finish();
  State<N> st;
  block_merge<N>(acc.I, acc.flags, acc.L, K, &st);
  __shared__ bool last;
  if (threadIdx.x == 0) {
    store_partial<N>(parts, blockIdx.x, K, st);
    __threadfence();
    unsigned t = atomicAdd(ticket, 1u);
    last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  merge_partials_cg<N>(parts, gridDim.x, K, &st);
  if (threadIdx.x == 0) {
    if (state) state_add<T>(state, K, st.I, st.flags, st.F, (uint64_t)n);
    else if constexpr (KT != 0) *result = convert_fast<T, KT>(st.I, st.flags, st.F);
    else *result = convert_state<T, N>(st, K);
    // leave the ticket zero for the next call
    *ticket = 0u;
  }
}

// Small inputs: one block, no workspace and no grid merge (the whole state
// is merged inside the block and converted by thread 0).  The result bits
// are the same as the grid path's.
template <typename T, int KT, int U>
__global__ void __launch_bounds__(1024) adn_sum_single(const T* __restrict__ x, int64_t n, int K,
                                                       T* __restrict__ result, unsigned char* __restrict__ state) {
  typedef typename AccOf<T, KT>::type Acc;
  constexpr int N = Acc::N;
  Acc acc;
  acc.init(K);
  accumulate_range<T, Acc, U>(acc, x, n, threadIdx.x, blockDim.x);
  acc.finish();
  State<N> st;
  block_merge<N>(acc.I, acc.flags, acc.L, K, &st);
  if (threadIdx.x == 0) {
    if (state) state_add<T>(state, K, st.I, st.flags, st.F, (uint64_t)n);
    else if constexpr (KT != 0) *result = convert_fast<T, KT>(st.I, st.flags, st.F);
    else *result = convert_state<T, N>(st, K);
  }
}

// --------------------------------------------------------- segmented sums
// One block per row (grid-stride over rows): rows of a row-major [rows, cols]
// array, any cols.
template <int KT, int U>
__global__ void __launch_bounds__(1024) segsum_rows_kernel(const float* __restrict__ x, int64_t rows,
                                                           int64_t cols, int K, float* __restrict__ out) {
  typedef AccF<KT> Acc;
  constexpr int N = Acc::N;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    Acc acc;
    acc.init(K);
    accumulate_range<float, Acc, U>(acc, x + r * cols, cols, threadIdx.x, blockDim.x);
    acc.finish();
    State<N> st;
    block_merge<N>(acc.I, acc.flags, acc.L, K, &st);
    if (threadIdx.x == 0) {
      if constexpr (KT != 0) out[r] = convert_fast<float, KT>(st.I, st.flags, st.F);
      else out[r] = convert_state<float, N>(st, K);
    }
    __syncthreads();
  }
}

// One warp per row (rows up to SEG_WARP_MAX columns): the lanes accumulate
// strided parts of the row and merge exactly inside the warp (block-wide
// minimum index replaced by the warp's, fold sums reduced by shuffles), so a
// row needs no shared memory or block barrier and many rows are in flight
// per SM (64 registers: 32 warps per SM, so 4096 rows fit one wave).  Same
// bits as the block kernel: the merge is exact.
template <int KT, int U>
__global__ void __launch_bounds__(256, 4) segsum_rows_warp(const float* __restrict__ x, int64_t rows, int64_t cols,
                                                        int K, float* __restrict__ out) {
  typedef AccF<KT> Acc;
  constexpr int N = Acc::N;
  const int lane = threadIdx.x & 31;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t GW = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = gw; r < rows; r += GW) {
    Acc acc;
    acc.init(K);
    accumulate_range<float, Acc, U>(acc, x + r * cols, cols, lane, 32);
    acc.finish();
    const int Iw = __reduce_min_sync(0xffffffffu, acc.I);
    const int fl = (int)__reduce_or_sync(0xffffffffu, (unsigned)acc.flags);
    const int d = acc.I - Iw;
    W128 F[N];
#pragma unroll
    for (int k = 0; k < N; ++k) {
      W128 v = W128{0, 0};
      if (k < K) {
        v = w_from(fold_at<N, int64_t>(acc.L, K, k - d));
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) v = w_add(v, shfl_xor_w(v, m));
      }
      F[k] = v;
    }
    if (lane == 0) {
      if constexpr (KT != 0) {
        out[r] = convert_fast<float, KT>(Iw, fl, F);
      } else {
        State<N> st;
        st.I = Iw;
        st.flags = fl;
        for (int k = 0; k < N; ++k) st.F[k] = F[k];
        out[r] = convert_state<float, N>(st, K);
      }
    }
  }
}

// One thread per column, rows walked in order (coalesced across columns).
template <int KT>
__global__ void __launch_bounds__(256) segsum_cols_kernel(const float* __restrict__ x, int64_t rows,
                                                          int64_t cols, int K, float* __restrict__ out) {
  typedef AccF<KT> Acc;
  constexpr int N = Acc::N;
  int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  Acc acc;
  acc.init(K);
  for (int64_t r = 0; r < rows; ++r) {
    float v[1] = {x[r * cols + c]};
    acc.template chunk<1>(v);
  }
  acc.finish();
  State<N> st;
  st.I = acc.I;
  st.flags = acc.flags;
  for (int k = 0; k < N; ++k) st.F[k] = w_from((k < K) ? acc.L[k] : 0);
  out[c] = convert_state<float, N>(st, K);
}

// ------------------------------------------------------------------ launch
template <typename T, int KT>
static cudaError_t launch_sum_k(const T* x, int64_t n, int K, unsigned* ticket, unsigned char* parts, T* result,
                                int grid, int block, cudaStream_t s, unsigned char* state = nullptr) {
  constexpr int U = 4;
  adn_sum_kernel<T, KT, U><<<grid, block, 0, s>>>(x, n, K, ticket, parts, result, state);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_sum(const T* x, int64_t n, int K, unsigned* ticket, unsigned char* parts, T* result, int grid,
                       int block, cudaStream_t s) {
  switch (K) {
    case 2: return launch_sum_k<T, 2>(x, n, K, ticket, parts, result, grid, block, s);
    case 3: return launch_sum_k<T, 3>(x, n, K, ticket, parts, result, grid, block, s);
    case 4: return launch_sum_k<T, 4>(x, n, K, ticket, parts, result, grid, block, s);
    case 5: return launch_sum_k<T, 5>(x, n, K, ticket, parts, result, grid, block, s);
    case 6: return launch_sum_k<T, 6>(x, n, K, ticket, parts, result, grid, block, s);
    case 7: return launch_sum_k<T, 7>(x, n, K, ticket, parts, result, grid, block, s);
    case 8: return launch_sum_k<T, 8>(x, n, K, ticket, parts, result, grid, block, s);
    default: return launch_sum_k<T, 0>(x, n, K, ticket, parts, result, grid, block, s);
  }
}

template <typename T>
cudaError_t launch_sum_single(const T* x, int64_t n, int K, T* result, int block, cudaStream_t s,
                              unsigned char* state) {
  constexpr int U = 1;
  switch (K) {
    case 2: adn_sum_single<T, 2, U><<<1, block, 0, s>>>(x, n, K, result, state); break;
    case 3: adn_sum_single<T, 3, U><<<1, block, 0, s>>>(x, n, K, result, state); break;
    case 4: adn_sum_single<T, 4, U><<<1, block, 0, s>>>(x, n, K, result, state); break;
    case 5: adn_sum_single<T, 5, U><<<1, block, 0, s>>>(x, n, K, result, state); break;
    case 6: adn_sum_single<T, 6, U><<<1, block, 0, s>>>(x, n, K, result, state); break;
    case 7: adn_sum_single<T, 7, U><<<1, block, 0, s>>>(x, n, K, result, state); break;
    case 8: adn_sum_single<T, 8, U><<<1, block, 0, s>>>(x, n, K, result, state); break;
    default: adn_sum_single<T, 0, U><<<1, block, 0, s>>>(x, n, K, result, state); break;
  }
  return cudaGetLastError();
}

template cudaError_t launch_sum_single<float>(const float*, int64_t, int, float*, int, cudaStream_t,
                                              unsigned char*);
template cudaError_t launch_sum_single<double>(const double*, int64_t, int, double*, int, cudaStream_t,
                                               unsigned char*);

// ------------------------------------------------------------ state calls
template <typename T>
cudaError_t launch_state_deposit(const T* x, int64_t n, int K, unsigned char* ws, unsigned char* state, int grid,
                                 int block, cudaStream_t s) {
  unsigned* tk = (unsigned*)ws;
  unsigned char* pp = ws + 256;
  switch (K) {
    case 2: return launch_sum_k<T, 2>(x, n, K, tk, pp, nullptr, grid, block, s, state);
    case 3: return launch_sum_k<T, 3>(x, n, K, tk, pp, nullptr, grid, block, s, state);
    case 4: return launch_sum_k<T, 4>(x, n, K, tk, pp, nullptr, grid, block, s, state);
    case 5: return launch_sum_k<T, 5>(x, n, K, tk, pp, nullptr, grid, block, s, state);
    case 6: return launch_sum_k<T, 6>(x, n, K, tk, pp, nullptr, grid, block, s, state);
    case 7: return launch_sum_k<T, 7>(x, n, K, tk, pp, nullptr, grid, block, s, state);
    case 8: return launch_sum_k<T, 8>(x, n, K, tk, pp, nullptr, grid, block, s, state);
    default: return launch_sum_k<T, 0>(x, n, K, tk, pp, nullptr, grid, block, s, state);
  }
}

template <typename T>
cudaError_t launch_state_op(int op, unsigned char* dst, const unsigned char* src, int K, uint64_t capacity,
                            T* result, cudaStream_t s) {
  if (op == 0) state_init_kernel<T><<<1, 1, 0, s>>>(dst, K);
  else if (op == 1) state_merge_kernel<T><<<1, 1, 0, s>>>(dst, src, K);
  else state_finalize_kernel<T><<<1, 1, 0, s>>>(src, K, capacity, result);
  return cudaGetLastError();
}

template cudaError_t launch_state_deposit<float>(const float*, int64_t, int, unsigned char*, unsigned char*, int, int,
                                                 cudaStream_t);
template cudaError_t launch_state_deposit<double>(const double*, int64_t, int, unsigned char*, unsigned char*, int,
                                                  int, cudaStream_t);
template cudaError_t launch_state_op<float>(int, unsigned char*, const unsigned char*, int, uint64_t, float*,
                                            cudaStream_t);
template cudaError_t launch_state_op<double>(int, unsigned char*, const unsigned char*, int, uint64_t, double*,
                                             cudaStream_t);

template cudaError_t launch_sum<float>(const float*, int64_t, int, unsigned*, unsigned char*, float*, int, int,
                                       cudaStream_t);
template cudaError_t launch_sum<double>(const double*, int64_t, int, unsigned*, unsigned char*, double*, int, int,
                                        cudaStream_t);

// Resident blocks per SM of the sum kernel for this K and block size (one
// wave of blocks covers the GPU; more would leave a partial second wave).
template <typename T, int KT>
static int occ_k(int block) {
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, adn_sum_kernel<T, KT, 4>, block, 0) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return nb > 0 ? nb : 1;
}

template <typename T>
int sum_blocks_per_sm(int K, int block) {
  switch (K) {
    case 2: return occ_k<T, 2>(block);
    case 3: return occ_k<T, 3>(block);
    case 4: return occ_k<T, 4>(block);
    case 5: return occ_k<T, 5>(block);
    case 6: return occ_k<T, 6>(block);
    case 7: return occ_k<T, 7>(block);
    case 8: return occ_k<T, 8>(block);
    default: return occ_k<T, 0>(block);
  }
}
template int sum_blocks_per_sm<float>(int, int);
template int sum_blocks_per_sm<double>(int, int);

size_t sum_workspace_bytes(int K, int grid) { return 256 + (size_t)grid * (16 + 16 * (size_t)K) + 64; }

// Rows up to this many columns use one warp per row.
constexpr int64_t SEG_WARP_MAX = 1 << 16;

cudaError_t launch_segsum(const float* x, int64_t rows, int64_t cols, int axis, int K, float* out, int grid,
                          int block, cudaStream_t s) {
  if (axis == 1 && cols <= SEG_WARP_MAX && (K == 2 || K == 3)) {
    // one warp per row, eight rows per block
    const int64_t g = (rows + 7) / 8;
    const unsigned wg = (unsigned)(g < 65535 * 16 ? g : 65535 * 16);
    if (K == 3) segsum_rows_warp<3, 2><<<wg, 256, 0, s>>>(x, rows, cols, K, out);
    else segsum_rows_warp<2, 2><<<wg, 256, 0, s>>>(x, rows, cols, K, out);
  } else if (axis == 1) {
    switch (K) {
      case 3: segsum_rows_kernel<3, 4><<<grid, block, 0, s>>>(x, rows, cols, K, out); break;
      case 2: segsum_rows_kernel<2, 4><<<grid, block, 0, s>>>(x, rows, cols, K, out); break;
      default: segsum_rows_kernel<0, 1><<<grid, block, 0, s>>>(x, rows, cols, K, out); break;
    }
  } else {
    int g = (int)((cols + 255) / 256);
    switch (K) {
      case 3: segsum_cols_kernel<3><<<g, 256, 0, s>>>(x, rows, cols, K, out); break;
      default: segsum_cols_kernel<0><<<g, 256, 0, s>>>(x, rows, cols, K, out); break;
    }
  }
  return cudaGetLastError();
}

}  // namespace repro
