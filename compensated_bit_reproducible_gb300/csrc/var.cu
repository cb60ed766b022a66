// Variance ("Variance in float32 with a first-element shift, a local
// centring and a compensated tree sum", section 2), every step in the input
// type (float32; float64 input runs the same steps in float64):
//   1. shift      y_i = x_i - x_0
//   2. centring   m = sum(y) / n,  d_i = y_i - m
//   3. TwoSum tree over d_i^2, errors carried up a second array; s2 = final
//      sum + final carry; s1 = sum(d)
//   4. var = max(s2/n - (s1/n)^2, 0) * n/(n - ddof);  mean = x_0 + m.
// Every tree pairs adjacent nodes (2i, 2i+1) level by level and passes an
// unpaired last node up unchanged.  Thread t owns the subtree of leaves
// [t C, t C + C) (C a power of two), so the tree, and the result bits, do not
// depend on the block size.
//
// Variants (template V; section 4, "Which step does what"):
//   0 the kernel;
//   1 the formula of reference (section 1, tf.nn.moments): no shift, means
//     as sum times RN(1/n), plain trees;
//   2 shift + centring, plain tree, no two-term (var = s2/n);
//   3 shift + centring, plain tree, two-term;
//   4 no shift: the formula of reference with the TwoSum tree for d^2;
//   5 shift + centring, TwoSum tree, no two-term;
//   6 shift + centring, s2 by Kahan's sequential loop over d^2 in index
//     order (one thread per slice), two-term.
// A TwoSum node's sum is the plain rounded add, so the plain-tree variants
// run the same tree and read only its sums.
//
// Complex input (section 2, last paragraph) is the real and the imaginary
// parts through the float32 kernel: the variance is RN(var_re + var_im).
// Rows of up to 4096 elements (axis 1) run both parts in one pass with pair
// nodes; other shapes read each part with an element stride of 2, the
// second pass adding its variance to the first's.
#include <cuda_runtime.h>
#include <cstdint>
#include "f32x2.cuh"
#include "launch.h"

namespace repro {

template <typename T> __device__ __forceinline__ T add_rn(T a, T b);
template <typename T> __device__ __forceinline__ T sub_rn(T a, T b);
template <typename T> __device__ __forceinline__ T mul_rn(T a, T b);
template <typename T> __device__ __forceinline__ T div_rn(T a, T b);
template <> __device__ __forceinline__ float add_rn(float a, float b) { return __fadd_rn(a, b); }
template <> __device__ __forceinline__ float sub_rn(float a, float b) { return __fsub_rn(a, b); }
template <> __device__ __forceinline__ float mul_rn(float a, float b) { return __fmul_rn(a, b); }
template <> __device__ __forceinline__ float div_rn(float a, float b) { return __fdiv_rn(a, b); }
template <> __device__ __forceinline__ double add_rn(double a, double b) { return __dadd_rn(a, b); }
template <> __device__ __forceinline__ double sub_rn(double a, double b) { return __dsub_rn(a, b); }
template <> __device__ __forceinline__ double mul_rn(double a, double b) { return __dmul_rn(a, b); }
template <> __device__ __forceinline__ double div_rn(double a, double b) { return __ddiv_rn(a, b); }

template <int V> struct Steps {
  static constexpr bool REF = V == 1 || V == 4;   // the reference formula's means and final step
  static constexpr bool SHIFT = !REF;
  static constexpr int COMP = (V == 1 || V == 2 || V == 3) ? 0 : (V == 6 ? 2 : 1);   // plain, TwoSum, Kahan
  static constexpr bool TWOTERM = !(V == 2 || V == 5);
};

template <typename T>
struct TS {   // TwoSum tree node: sum s, carried error c
  T s, c;
};

template <typename T>
__device__ __forceinline__ TS<T> ts_combine(TS<T> l, TS<T> r) {
  // TwoSum (six operations) and the carry of the two children
  T s = add_rn(l.s, r.s);
  T bb = sub_rn(s, l.s);
  T e = add_rn(sub_rn(l.s, sub_rn(s, bb)), sub_rn(r.s, bb));
  T c = add_rn(add_rn(l.c, r.c), e);
  return TS<T>{s, c};
}

// Node of the pass-2 trees: compensated d^2 tree and plain d tree together.
template <typename T>
struct N2 {
  TS<T> q;
  T d;
};
template <typename T>
__device__ __forceinline__ N2<T> n2_combine(N2<T> l, N2<T> r) {
  return N2<T>{ts_combine(l.q, r.q), add_rn(l.d, r.d)};
}
template <typename T>
__device__ __forceinline__ T f_combine(T l, T r) {
  return add_rn(l, r);
}

// Streaming subtree over a valid prefix of `m` leaves (m <= C, C <= 2^LMAX):
// a binary-counter stack holds complete subtrees; the root of the C-leaf tree
// with the last C - m leaves absent is the right-nested combination of the
// stack from the lowest level up (an absent right sibling passes its left
// sibling through).
template <typename Node, int LMAX>
struct Stack {
  Node s[LMAX + 1];
  int count;
  __device__ __forceinline__ void reset() { count = 0; }
  template <typename F>
  __device__ __forceinline__ void push(Node v, F comb) {
    int lvl = 0;
    int c = count;
#pragma unroll 1
    while (c & 1) {
      v = comb(s[lvl], v);
      c >>= 1;
      ++lvl;
    }
    s[lvl] = v;
    ++count;
  }
  template <typename F>
  __device__ __forceinline__ bool root(Node& out, F comb) const {
    bool have = false;
    Node acc;
#pragma unroll 1
    for (int lvl = 0; lvl <= LMAX; ++lvl) {
      if ((count >> lvl) & 1) {
        acc = have ? comb(s[lvl], acc) : s[lvl];
        have = true;
      }
    }
    out = acc;
    return have;
  }
};

template <typename T> __device__ __forceinline__ T shfl_down_node(T v, int d) {
  return __shfl_down_sync(0xffffffffu, v, d);
}
template <typename T> __device__ __forceinline__ N2<T> shfl_down_node(N2<T> v, int d) {
  return N2<T>{TS<T>{__shfl_down_sync(0xffffffffu, v.q.s, d), __shfl_down_sync(0xffffffffu, v.q.c, d)},
               __shfl_down_sync(0xffffffffu, v.d, d)};
}

template <typename T> __device__ __forceinline__ T shfl_node(T v, int src) {
  return __shfl_sync(0xffffffffu, v, src);
}
template <typename T> __device__ __forceinline__ N2<T> shfl_node(N2<T> v, int src) {
  return N2<T>{TS<T>{__shfl_sync(0xffffffffu, v.q.s, src), __shfl_sync(0xffffffffu, v.q.c, src)},
               __shfl_sync(0xffffffffu, v.d, src)};
}

// Combine the per-thread subtree roots of one slice, in tree order.  Threads
// are numbered by `pos` (0..P-1, P = number of participating threads, a
// multiple of 32 when P > 32, laid out so that pos p and p+1 are adjacent
// lanes for p < 32 within a warp); `have` is false for an empty subtree.
// The result is valid in the thread with pos == 0.
template <typename Node, typename F>
__device__ Node tree_combine_block(Node v, bool have, int P, Node* sm, bool* smv, F comb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // within a warp: levels 1, 2, 4, 8, 16
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    Node o = shfl_down_node(v, d);
    bool oh = __shfl_down_sync(0xffffffffu, have, d);
    if ((lane & (2 * d - 1)) == 0 && lane + d < 32) {
      if (have && oh) v = comb(v, o);
      else if (!have && oh) { v = o; have = true; }
    }
  }
  int nw = P >> 5;
  if (nw <= 1) return v;
  __syncthreads();
  if (lane == 0) { sm[warp] = v; smv[warp] = have; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int step = 1; step < nw; step <<= 1)
      for (int w = 0; w + step < nw; w += 2 * step) {
        if (smv[w] && smv[w + step]) sm[w] = comb(sm[w], sm[w + step]);
        else if (!smv[w] && smv[w + step]) { sm[w] = sm[w + step]; smv[w] = true; }
      }
    v = sm[0];
  }
  __syncthreads();
  return v;
}

// tree_combine_block when every one of the P threads holds a subtree (P a
// power of two); the root is returned in every thread.  At the level that
// pairs nodes d apart, lane L (L a multiple of 2d) combines with lane L + d;
// the other lanes combine too, unconditionally, and their values are never
// read by a lane that carries the tree: lane L + d at level d is a multiple
// of d, so it was a left node, combined correctly, at every lower level.
// One barrier: the warp roots go to shared memory and each warp combines
// them the same way (lanes 0..nw-1 hold roots 0..nw-1).  The caller must
// pass a barrier between the read of `sm` here and its next write
// (alternating two arrays does that).
template <typename Node, typename F>
__device__ __forceinline__ Node tree_combine_block_all(Node v, int P, Node* sm, F comb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) v = comb(v, shfl_down_node(v, d));
  const int nw = P >> 5;
  if (nw > 1) {
    if (lane == 0) sm[warp] = v;
    __syncthreads();
    v = sm[lane < nw ? lane : 0];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      if (d >= nw) break;
      v = comb(v, shfl_down_node(v, d));
    }
  }
  return shfl_node(v, 0);
}

template <typename T>
__device__ __forceinline__ T max_nan0(T v) {
  if (v != v) return v;
  return v > (T)0 ? v : (T)0;
}

// Output of one slice, where every pass-2 quantity is known: variance
// (rescaled, added to *out when `acc`) and mean.
struct VarOut {
  int acc;           // add the variance to the value already in out[s]
  int64_t mstride;   // mean_out[s * mstride]
};

// The slice length n and n - ddof converted to the input type once per
// kernel, outside the slice loops (the divisions stay with the thread that
// needs them: in double they run on the slow FP64 pipe).
template <typename T>
struct Count {
  T nf, nd;
  int ddof;
};
template <typename T>
__device__ __forceinline__ Count<T> make_count(int64_t n, int ddof) {
  return Count<T>{(T)n, (T)(n - ddof), ddof};
}

// Variance and mean of one slice from its pass-2 quantities.
template <typename T, int V>
__device__ __forceinline__ void slice_stats(const N2<T>& tot, T kahan_s2, T x0, T mu, const Count<T>& cnt, T& var,
                                            T& mean) {
  typedef Steps<V> St;
  const T nf = cnt.nf;
  if constexpr (St::REF) {
    T inv = div_rn((T)1, nf);
    T md = mul_rn(tot.d, inv);
    T s2 = St::COMP == 1 ? add_rn(tot.q.s, tot.q.c) : tot.q.s;
    var = max_nan0(sub_rn(mul_rn(s2, inv), mul_rn(md, md)));
    mean = mu;
  } else {
    T s2 = St::COMP == 1 ? add_rn(tot.q.s, tot.q.c) : (St::COMP == 0 ? tot.q.s : kahan_s2);
    T t = div_rn(tot.d, nf);
    T v = St::TWOTERM ? sub_rn(div_rn(s2, nf), mul_rn(t, t)) : div_rn(s2, nf);
    var = max_nan0(v);
    mean = add_rn(x0, mu);
  }
  if (cnt.ddof != 0) var = mul_rn(var, div_rn(nf, cnt.nd));
}

template <typename T, int V>
__device__ __forceinline__ void finish_slice(const N2<T>& tot, T kahan_s2, T x0, T mu, const Count<T>& cnt,
                                             T* out, T* mean_out, int64_t s, VarOut io) {
  T var, mean;
  slice_stats<T, V>(tot, kahan_s2, x0, mu, cnt, var, mean);
  out[s] = io.acc ? add_rn(out[s], var) : var;
  if (mean_out) mean_out[s * io.mstride] = mean;
}

// Kahan's loop over d_i^2 in index order (variant 6), one thread.
template <typename T>
__device__ T kahan_sq(const T* x, int64_t n, int64_t stride, T x0, T mu) {
  T s = (T)0, c = (T)0;
  for (int64_t i = 0; i < n; ++i) {
    T d = sub_rn(sub_rn(x[i * stride], x0), mu);
    T y = sub_rn(mul_rn(d, d), c);
    T t = add_rn(s, y);
    c = sub_rn(sub_rn(t, s), y);
    s = t;
  }
  return s;
}

template <typename T, int V>
__device__ __forceinline__ T leaf1(T xi, T x0) {
  return Steps<V>::SHIFT ? sub_rn(xi, x0) : xi;
}
template <typename T, int V>
__device__ __forceinline__ T leaf_d(T xi, T x0, T mu) {
  typedef Steps<V> St;
  if constexpr (St::SHIFT) return sub_rn(sub_rn(xi, x0), mu);
  else return sub_rn(xi, mu);
}
template <typename T, int V>
__device__ __forceinline__ T mean_of(T sum1, const Count<T>& cnt) {
  return Steps<V>::REF ? mul_rn(sum1, div_rn((T)1, cnt.nf)) : div_rn(sum1, cnt.nf);
}

// Row kernel (axis 1): one block per row, thread t owns leaves [t C, t C + C).
// Element i of row r is x[(r cols + i) es].
template <typename T, int V>
__global__ void __launch_bounds__(1024) var_rows_kernel(const T* __restrict__ x, int64_t rows, int64_t cols,
                                                        int64_t es, int ddof, T* __restrict__ out,
                                                        T* __restrict__ mean_out, VarOut io, int64_t C) {
  typedef Steps<V> St;
  __shared__ T smf[32];
  __shared__ N2<T> sm2[32];
  __shared__ bool smv[32];
  __shared__ T bc[2];
  const int64_t n = cols;
  const Count<T> cnt = make_count<T>(n, ddof);
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* row = x + r * cols * es;
    const T x0 = row[0];
    int64_t b = (int64_t)threadIdx.x * C;
    int64_t m = n - b;
    m = m < 0 ? 0 : (m > C ? C : m);
    T mu = (T)0;
    {
      // pass 1: sum of y (shift) or of x (reference)
      Stack<T, 40> st1;
      st1.reset();
      for (int64_t i = 0; i < m; ++i) st1.push(leaf1<T, V>(row[(b + i) * es], x0), f_combine<T>);
      T v1 = (T)0;
      bool h1 = st1.root(v1, f_combine<T>);
      T sum1 = tree_combine_block<T>(v1, h1, blockDim.x, smf, smv, f_combine<T>);
      if (threadIdx.x == 0) bc[0] = mean_of<T, V>(sum1, cnt);
      __syncthreads();
      mu = bc[0];
    }
    // pass 2: d, the d^2 tree (TwoSum nodes) and the d tree
    Stack<N2<T>, 40> st2;
    st2.reset();
    for (int64_t i = 0; i < m; ++i) {
      T d = leaf_d<T, V>(row[(b + i) * es], x0, mu);
      st2.push(N2<T>{TS<T>{mul_rn(d, d), (T)0}, d}, n2_combine<T>);
    }
    N2<T> v2;
    bool h2 = st2.root(v2, n2_combine<T>);
    N2<T> tot = tree_combine_block<N2<T>>(v2, h2, blockDim.x, sm2, smv, n2_combine<T>);
    if (threadIdx.x == 0) {
      T ks = St::COMP == 2 ? kahan_sq<T>(row, n, es, x0, mu) : (T)0;
      finish_slice<T, V>(tot, ks, x0, mu, cnt, out, mean_out, r, io);
    }
    __syncthreads();
  }
}

// Column kernel (axis 0): a block covers 32 adjacent columns (threadIdx.x)
// and G row groups (threadIdx.y); group g owns rows [g C, g C + C).  Element
// (i, c) is x[(i cols + c) es].
template <typename T, int V>
__global__ void __launch_bounds__(256) var_cols_kernel(const T* __restrict__ x, int64_t rows, int64_t cols,
                                                       int64_t es, int ddof, T* __restrict__ out,
                                                       T* __restrict__ mean_out, VarOut io, int64_t C) {
  typedef Steps<V> St;
  __shared__ T smf[8][32];
  __shared__ N2<T> sm2[8][32];
  __shared__ bool smv[8][32];
  __shared__ T bc[32];
  const int G = blockDim.y;
  const int64_t n = rows;
  const Count<T> cnt = make_count<T>(n, ddof);
  const int64_t c = (int64_t)blockIdx.x * 32 + threadIdx.x;
  const bool col_ok = c < cols;
  const int g = threadIdx.y;
  int64_t b = (int64_t)g * C;
  int64_t m = n - b;
  m = m < 0 ? 0 : (m > C ? C : m);
  if (!col_ok) m = 0;
  const T x0 = col_ok ? x[c * es] : (T)0;
  T mu = (T)0;
  {
    Stack<T, 40> st1;
    st1.reset();
    for (int64_t i = 0; i < m; ++i) st1.push(leaf1<T, V>(x[((b + i) * cols + c) * es], x0), f_combine<T>);
    T v1 = (T)0;
    bool h1 = st1.root(v1, f_combine<T>);
    smf[g][threadIdx.x] = v1;
    smv[g][threadIdx.x] = h1;
    __syncthreads();
    if (g == 0) {
      for (int step = 1; step < G; step <<= 1)
        for (int w = 0; w + step < G; w += 2 * step) {
          if (smv[w][threadIdx.x] && smv[w + step][threadIdx.x])
            smf[w][threadIdx.x] = add_rn(smf[w][threadIdx.x], smf[w + step][threadIdx.x]);
          else if (!smv[w][threadIdx.x] && smv[w + step][threadIdx.x]) {
            smf[w][threadIdx.x] = smf[w + step][threadIdx.x];
            smv[w][threadIdx.x] = true;
          }
        }
      bc[threadIdx.x] = mean_of<T, V>(smf[0][threadIdx.x], cnt);
    }
    __syncthreads();
    mu = bc[threadIdx.x];
  }
  Stack<N2<T>, 40> st2;
  st2.reset();
  for (int64_t i = 0; i < m; ++i) {
    T d = leaf_d<T, V>(x[((b + i) * cols + c) * es], x0, mu);
    st2.push(N2<T>{TS<T>{mul_rn(d, d), (T)0}, d}, n2_combine<T>);
  }
  N2<T> v2;
  bool h2 = st2.root(v2, n2_combine<T>);
  sm2[g][threadIdx.x] = v2;
  smv[g][threadIdx.x] = h2;
  __syncthreads();
  if (g == 0 && col_ok) {
    for (int step = 1; step < G; step <<= 1)
      for (int w = 0; w + step < G; w += 2 * step) {
        if (smv[w][threadIdx.x] && smv[w + step][threadIdx.x])
          sm2[w][threadIdx.x] = n2_combine(sm2[w][threadIdx.x], sm2[w + step][threadIdx.x]);
        else if (!smv[w][threadIdx.x] && smv[w + step][threadIdx.x]) {
          sm2[w][threadIdx.x] = sm2[w + step][threadIdx.x];
          smv[w][threadIdx.x] = true;
        }
      }
    T ks = St::COMP == 2 ? kahan_sq<T>(x + c * es, n, cols * es, x0, mu) : (T)0;
    finish_slice<T, V>(sm2[0][threadIdx.x], ks, x0, mu, cnt, out, mean_out, c, io);
  }
}

// Register version for rows of at most 256 * 16 elements: thread t owns the
// C leaves [t C, t C + C) (C a power of two <= 16) in registers; the subtree
// is the statically unrolled adjacent-pair tree over its valid prefix.
template <typename Node, int C, typename F>
__device__ __forceinline__ bool reg_tree(Node* a, int m, F comb) {
  // a[0..C) with the first m valid; returns whether the root exists (in a[0])
  int cnt = m;
#pragma unroll
  for (int w = C; w > 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w / 2; ++i) {
      if (2 * i + 1 < cnt) a[i] = comb(a[2 * i], a[2 * i + 1]);
      else if (2 * i < cnt) a[i] = a[2 * i];
    }
    cnt = (cnt + 1) >> 1;
  }
  return m > 0;
}

// The same tree when all C leaves are present: no per-node presence tests.
template <typename Node, int C, typename F>
__device__ __forceinline__ void reg_tree_full(Node* a, F comb) {
#pragma unroll
  for (int w = C; w > 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w / 2; ++i) a[i] = comb(a[2 * i], a[2 * i + 1]);
  }
}

__device__ __forceinline__ F2 f2_combine(F2 l, F2 r) { return add2(l, r); }

// Two pass-2 nodes side by side: the operations of ts_combine and
// n2_combine, in the same order, on both lanes.
struct N2x {
  F2 s, c, d;
};
__device__ __forceinline__ N2x n2x_combine(N2x l, N2x r) {
  const F2 s = add2(l.s, r.s);
  const F2 bb = sub2(s, l.s);
  const F2 e = add2(sub2(l.s, sub2(s, bb)), sub2(r.s, bb));
  return N2x{s, add2(add2(l.c, r.c), e), add2(l.d, r.d)};
}

// A thread's full subtree of C float leaves as two half-subtrees in
// lockstep: leaves [0, C/2) in lane x, [C/2, C) in lane y, then one scalar
// combine of the two roots (x left, y right).  That is the adjacent-pair
// tree of the C leaves, with half the floating-point instructions.
template <int V, int C>
__device__ __forceinline__ float root1_packed(const float* v, float x0) {
  constexpr int H = C / 2;
  F2 a[H];
  const F2 X0 = pk2(x0, x0);
#pragma unroll
  for (int j = 0; j < H; ++j) {
    const F2 p = pk2(v[j], v[j + H]);
    a[j] = Steps<V>::SHIFT ? sub2(p, X0) : p;
  }
  reg_tree_full<F2, H>(a, f2_combine);
  float x, y;
  up2(a[0], x, y);
  return add_rn(x, y);
}
template <int V, int C>
__device__ __forceinline__ N2<float> root2_packed(const float* v, float x0, float mu) {
  constexpr int H = C / 2;
  N2x a[H];
  const F2 X0 = pk2(x0, x0), MU = pk2(mu, mu);
#pragma unroll
  for (int j = 0; j < H; ++j) {
    const F2 p = pk2(v[j], v[j + H]);
    const F2 d = Steps<V>::SHIFT ? sub2(sub2(p, X0), MU) : sub2(p, MU);
    float dx, dy;
    up2(d, dx, dy);
    a[j] = N2x{pk2(mul_rn(dx, dx), mul_rn(dy, dy)), 0ull, d};
  }
  reg_tree_full<N2x, H>(a, n2x_combine);
  float sx, sy, cx, cy, dx, dy;
  up2(a[0].s, sx, sy);
  up2(a[0].c, cx, cy);
  up2(a[0].d, dx, dy);
  return n2_combine(N2<float>{TS<float>{sx, cx}, dx}, N2<float>{TS<float>{sy, cy}, dy});
}

// Root of a thread's full subtree in pass 1 / pass 2 (t1, t2: its leaves).
template <typename T, int V, int C>
__device__ __forceinline__ T full_root1(const T* v, T* t1, T x0) {
  if constexpr (sizeof(T) == 4 && C >= 2) {
    return root1_packed<V, C>(v, x0);
  } else {
    reg_tree_full<T, C>(t1, f_combine<T>);
    return t1[0];
  }
}
template <typename T, int V, int C>
__device__ __forceinline__ N2<T> full_root2(const T* v, N2<T>* t2, T x0, T mu) {
  if constexpr (sizeof(T) == 4 && C >= 2) {
    return root2_packed<V, C>(v, x0, mu);
  } else {
    reg_tree_full<N2<T>, C>(t2, n2_combine<T>);
    return t2[0];
  }
}

template <typename T> struct Vec16;
template <> struct Vec16<float> {
  typedef float4 type;
  static constexpr int W = 4;
  __device__ __forceinline__ static void put(const float4& q, float* v) {
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
};
template <> struct Vec16<double> {
  typedef double2 type;
  static constexpr int W = 2;
  __device__ __forceinline__ static void put(const double2& q, double* v) {
    v[0] = q.x; v[1] = q.y;
  }
};

// Resident blocks asked for: five per SM for float (47 registers; the Kahan
// variant's time is one thread's loop per row, so it scales with the blocks
// in flight), three for double (72 registers, no spills).  Without an
// explicit count the compiler gave some instances 79 or 110 registers.
template <typename T, int C, int V>
__global__ void __launch_bounds__(256, sizeof(T) == 4 ? 5 : 3)
    var_rows_reg(const T* __restrict__ x, int64_t rows, int64_t cols, int64_t es, int ddof, T* __restrict__ out,
                 T* __restrict__ mean_out, VarOut io) {
  typedef Steps<V> St;
  typedef Vec16<T> VT;
  __shared__ T smf[32];
  __shared__ N2<T> sm2[32];
  __shared__ bool smv[32];
  __shared__ T bc[1];
  const int n = (int)cols;
  const Count<T> cnt = make_count<T>(n, ddof);
  const int b = threadIdx.x * C;
  int m = n - b;
  m = m < 0 ? 0 : (m > C ? C : m);
  // every thread of the block holds C leaves (the row fills the block).
  // Float only: in the full-row path every warp runs the cross-warp levels,
  // which for double would put eight times the FP64 work of one thread on
  // GB300's slow FP64 pipe.  The Kahan variant, whose time is one thread's
  // sequential loop per row, keeps the general path and its lower register
  // count (more blocks in flight).
  const bool all = sizeof(T) == 4 && St::COMP != 2 && n >= (int)blockDim.x * C;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* row = x + r * cols * es;
    const T x0 = __ldg(row);
    T v[C];
    if (C % VT::W == 0 && es == 1 && m == C && ((((uintptr_t)(row + b)) & 15) == 0)) {
#pragma unroll
      for (int u = 0; u < C / VT::W; ++u) VT::put(__ldcs((const typename VT::type*)(row + b) + u), v + VT::W * u);
    } else {
#pragma unroll
      for (int i = 0; i < C; ++i) v[i] = (i < m) ? row[(b + i) * es] : (T)0;
    }
    T mu = (T)0;
    {
      // pass 1
      T t1[C];
#pragma unroll
      for (int i = 0; i < C; ++i) t1[i] = leaf1<T, V>(v[i], x0);
      if (all) {
        // every thread has the root and forms the same mean
        const T r1 = full_root1<T, V, C>(v, t1, x0);
        mu = mean_of<T, V>(tree_combine_block_all<T>(r1, blockDim.x, smf, f_combine<T>), cnt);
      } else {
        bool h1 = reg_tree<T, C>(t1, m, f_combine<T>);
        T sum1 = tree_combine_block<T>(t1[0], h1, blockDim.x, smf, smv, f_combine<T>);
        if (threadIdx.x == 0) bc[0] = mean_of<T, V>(sum1, cnt);
        __syncthreads();
        mu = bc[0];
      }
    }
    // pass 2
    N2<T> t2[C];
#pragma unroll
    for (int i = 0; i < C; ++i) {
      T d = leaf_d<T, V>(v[i], x0, mu);
      t2[i] = N2<T>{TS<T>{mul_rn(d, d), (T)0}, d};
    }
    N2<T> tot;
    if (all) {
      // one barrier per pass: smf and sm2 alternate, so each is rewritten
      // only after the other pass's barrier
      const N2<T> r2 = full_root2<T, V, C>(v, t2, x0, mu);
      tot = tree_combine_block_all<N2<T>>(r2, blockDim.x, sm2, n2_combine<T>);
    } else {
      bool h2 = reg_tree<N2<T>, C>(t2, m, n2_combine<T>);
      tot = tree_combine_block<N2<T>>(t2[0], h2, blockDim.x, sm2, smv, n2_combine<T>);
    }
    if (threadIdx.x == 0) {
      T ks = St::COMP == 2 ? kahan_sq<T>(row, n, es, x0, mu) : (T)0;
      finish_slice<T, V>(tot, ks, x0, mu, cnt, out, mean_out, r, io);
    }
    if (!all) __syncthreads();
  }
}

template <typename T, int V>
static void launch_rows_reg(int64_t C, const T* x, int64_t rows, int64_t cols, int64_t es, int ddof, T* out,
                            T* mean, VarOut io, unsigned grid, cudaStream_t s) {
  switch (C) {
    case 1: var_rows_reg<T, 1, V><<<grid, 256, 0, s>>>(x, rows, cols, es, ddof, out, mean, io); break;
    case 2: var_rows_reg<T, 2, V><<<grid, 256, 0, s>>>(x, rows, cols, es, ddof, out, mean, io); break;
    case 4: var_rows_reg<T, 4, V><<<grid, 256, 0, s>>>(x, rows, cols, es, ddof, out, mean, io); break;
    case 8: var_rows_reg<T, 8, V><<<grid, 256, 0, s>>>(x, rows, cols, es, ddof, out, mean, io); break;
    default: var_rows_reg<T, 16, V><<<grid, 256, 0, s>>>(x, rows, cols, es, ddof, out, mean, io); break;
  }
}

static int64_t pow2_ceil(int64_t v) {
  int64_t p = 1;
  while (p < v) p <<= 1;
  return p;
}

template <typename T, int V>
static cudaError_t launch_var_v(const T* x, int64_t rows, int64_t cols, int axis, int ddof, int64_t es, T* out,
                                T* mean, VarOut io, cudaStream_t s) {
  if (axis == 1) {
    int block = 256;
    int64_t np = pow2_ceil(cols);
    int64_t C = np / block;
    if (C < 1) C = 1;
    int64_t grid = rows < 65535 * 16 ? rows : 65535 * 16;
    if (C <= 16) launch_rows_reg<T, V>(C, x, rows, cols, es, ddof, out, mean, io, (unsigned)grid, s);
    else var_rows_kernel<T, V><<<(unsigned)grid, block, 0, s>>>(x, rows, cols, es, ddof, out, mean, io, C);
  } else {
    int G = 8;
    int64_t np = pow2_ceil(rows);
    int64_t C = np / G;
    if (C < 1) C = 1;
    dim3 block(32, G);
    unsigned grid = (unsigned)((cols + 31) / 32);
    var_cols_kernel<T, V><<<grid, block, 0, s>>>(x, rows, cols, es, ddof, out, mean, io, C);
  }
  return cudaGetLastError();
}

size_t var_workspace_bytes(int64_t, int64_t, int) { return 0; }

cudaError_t launch_var(const float* x, int64_t rows, int64_t cols, int axis, int ddof, float* out, float* mean,
                       int variant, unsigned char*, cudaStream_t s) {
  const VarOut io{0, 1};
  switch (variant) {
    case 0: return launch_var_v<float, 0>(x, rows, cols, axis, ddof, 1, out, mean, io, s);
    case 1: return launch_var_v<float, 1>(x, rows, cols, axis, ddof, 1, out, mean, io, s);
    case 2: return launch_var_v<float, 2>(x, rows, cols, axis, ddof, 1, out, mean, io, s);
    case 3: return launch_var_v<float, 3>(x, rows, cols, axis, ddof, 1, out, mean, io, s);
    case 4: return launch_var_v<float, 4>(x, rows, cols, axis, ddof, 1, out, mean, io, s);
    case 5: return launch_var_v<float, 5>(x, rows, cols, axis, ddof, 1, out, mean, io, s);
    case 6: return launch_var_v<float, 6>(x, rows, cols, axis, ddof, 1, out, mean, io, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_var_f64(const double* x, int64_t rows, int64_t cols, int axis, int ddof, double* out,
                           double* mean, cudaStream_t s) {
  return launch_var_v<double, 0>(x, rows, cols, axis, ddof, 1, out, mean, VarOut{0, 1}, s);
}

// ------------------------------------------------- complex rows in one pass
// The real and the imaginary parts of a complex64 row run side by side:
// every tree node is a pair combined componentwise, so each part's tree is
// the adjacent-pair tree of the float kernel and gives its bits; the row's
// variance is RN(var_re + var_im) and its mean (mean_re, mean_im), as in two
// strided passes.  Thread t owns complex leaves [t C, t C + C) (C <= 8).
template <typename T>
struct Pair {
  T re, im;
};
template <typename T> __device__ __forceinline__ Pair<T> shfl_down_node(Pair<T> v, int d) {
  return Pair<T>{shfl_down_node(v.re, d), shfl_down_node(v.im, d)};
}
template <typename T> __device__ __forceinline__ Pair<T> shfl_node(Pair<T> v, int src) {
  return Pair<T>{shfl_node(v.re, src), shfl_node(v.im, src)};
}
__device__ __forceinline__ Pair<float> pf_combine(Pair<float> l, Pair<float> r) {
  return Pair<float>{add_rn(l.re, r.re), add_rn(l.im, r.im)};
}
__device__ __forceinline__ Pair<N2<float>> pn2_combine(Pair<N2<float>> l, Pair<N2<float>> r) {
  return Pair<N2<float>>{n2_combine(l.re, r.re), n2_combine(l.im, r.im)};
}

template <int C>
__global__ void __launch_bounds__(512) var_rows_c64(const float* __restrict__ z, int64_t rows, int64_t cols,
                                                    int ddof, float* __restrict__ out,
                                                    float* __restrict__ mean_out) {
  typedef Pair<float> P;
  typedef Pair<N2<float>> Q;
  __shared__ P smf[32];
  __shared__ Q sm2[32];
  __shared__ bool smv[32];
  __shared__ P bc[1];
  const int n = (int)cols;
  const Count<float> cnt = make_count<float>(n, ddof);
  const int b = threadIdx.x * C;
  int m = n - b;
  m = m < 0 ? 0 : (m > C ? C : m);
  const bool all = n >= (int)blockDim.x * C;   // every thread holds C leaves
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const float* row = z + 2 * r * cols;
    const float re0 = __ldg(row), im0 = __ldg(row + 1);
    float vr[C], vi[C];
    if (C % 2 == 0 && m == C && ((((uintptr_t)(row + 2 * b)) & 15) == 0)) {
#pragma unroll
      for (int u = 0; u < C / 2; ++u) {
        const float4 q = __ldcs((const float4*)(row + 2 * b) + u);
        vr[2 * u] = q.x;
        vi[2 * u] = q.y;
        vr[2 * u + 1] = q.z;
        vi[2 * u + 1] = q.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < C; ++i) {
        vr[i] = (i < m) ? row[2 * (b + i)] : 0.f;
        vi[i] = (i < m) ? row[2 * (b + i) + 1] : 0.f;
      }
    }
    P mu;
    {
      // pass 1
      P t1[C];
#pragma unroll
      for (int i = 0; i < C; ++i) t1[i] = P{leaf1<float, 0>(vr[i], re0), leaf1<float, 0>(vi[i], im0)};
      if (all) {
        reg_tree_full<P, C>(t1, pf_combine);
        const P s1 = tree_combine_block_all<P>(t1[0], blockDim.x, smf, pf_combine);
        mu = P{mean_of<float, 0>(s1.re, cnt), mean_of<float, 0>(s1.im, cnt)};
      } else {
        bool h1 = reg_tree<P, C>(t1, m, pf_combine);
        const P s1 = tree_combine_block<P>(t1[0], h1, blockDim.x, smf, smv, pf_combine);
        if (threadIdx.x == 0) bc[0] = P{mean_of<float, 0>(s1.re, cnt), mean_of<float, 0>(s1.im, cnt)};
        __syncthreads();
        mu = bc[0];
      }
    }
    // pass 2
    Q t2[C];
#pragma unroll
    for (int i = 0; i < C; ++i) {
      const float dr = leaf_d<float, 0>(vr[i], re0, mu.re), di = leaf_d<float, 0>(vi[i], im0, mu.im);
      t2[i] = Q{N2<float>{TS<float>{mul_rn(dr, dr), 0.f}, dr}, N2<float>{TS<float>{mul_rn(di, di), 0.f}, di}};
    }
    Q tot;
    if (all) {
      // smf and sm2 alternate: each is rewritten only after the other
      // pass's barrier
      reg_tree_full<Q, C>(t2, pn2_combine);
      tot = tree_combine_block_all<Q>(t2[0], blockDim.x, sm2, pn2_combine);
    } else {
      bool h2 = reg_tree<Q, C>(t2, m, pn2_combine);
      tot = tree_combine_block<Q>(t2[0], h2, blockDim.x, sm2, smv, pn2_combine);
    }
    if (threadIdx.x == 0) {
      float var_re, mean_re, var_im, mean_im;
      slice_stats<float, 0>(tot.re, 0.f, re0, mu.re, cnt, var_re, mean_re);
      slice_stats<float, 0>(tot.im, 0.f, im0, mu.im, cnt, var_im, mean_im);
      out[r] = add_rn(var_re, var_im);
      if (mean_out) {
        mean_out[2 * r] = mean_re;
        mean_out[2 * r + 1] = mean_im;
      }
    }
    if (!all) __syncthreads();
  }
}

cudaError_t launch_var_c64(const float* z, int64_t rows, int64_t cols, int axis, int ddof, float* out,
                           float* mean, cudaStream_t s) {
  if (axis == 1 && cols <= 4096) {
    // one pass: 256 threads and C = 1..8 leaves each, or 512 threads at C = 8
    const int64_t np = pow2_ceil(cols);
    const int block = np <= 2048 ? 256 : 512;
    int64_t C = np / block;
    if (C < 1) C = 1;
    const unsigned grid = (unsigned)(rows < 65535 * 16 ? rows : 65535 * 16);
    switch (C) {
      case 1: var_rows_c64<1><<<grid, block, 0, s>>>(z, rows, cols, ddof, out, mean); break;
      case 2: var_rows_c64<2><<<grid, block, 0, s>>>(z, rows, cols, ddof, out, mean); break;
      case 4: var_rows_c64<4><<<grid, block, 0, s>>>(z, rows, cols, ddof, out, mean); break;
      default: var_rows_c64<8><<<grid, block, 0, s>>>(z, rows, cols, ddof, out, mean); break;
    }
    return cudaGetLastError();
  }
  // two strided passes: real parts (mean to the even floats), then
  // imaginary parts added on
  cudaError_t e = launch_var_v<float, 0>(z, rows, cols, axis, ddof, 2, out, mean, VarOut{0, 2}, s);
  if (e != cudaSuccess) return e;
  return launch_var_v<float, 0>(z + 1, rows, cols, axis, ddof, 2, out, mean ? mean + 1 : nullptr, VarOut{1, 2}, s);
}

}  // namespace repro
