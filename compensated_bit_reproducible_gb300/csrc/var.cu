// Float32 variance ("Variance in float32 with a first-element shift, a local
// centring and a compensated tree sum", section 2), all in float32:
//   1. shift      y_i = x_i - x_0
//   2. centring   m = sum(y) / n,  d_i = y_i - m
//   3. TwoSum tree over d_i^2, errors carried up a second array; s2 = final
//      sum + final carry; s1 = sum(d)
//   4. var = max(s2/n - (s1/n)^2, 0) * n/(n - ddof);  mean = x_0 + m.
// Every tree pairs adjacent nodes (2i, 2i+1) level by level and passes an
// unpaired last node up unchanged.  Thread t owns the subtree of leaves
// [t C, t C + C) (C a power of two), so the tree, and the result bits, do not
// depend on the block size.  Also the formula of reference (section 1,
// tf.nn.moments) on the same trees, for comparison.
#include <cuda_runtime.h>
#include <cstdint>
#include "launch.h"

namespace repro {

struct TS {   // TwoSum tree node: sum s, carried error c
  float s, c;
};

__device__ __forceinline__ TS ts_combine(TS l, TS r) {
  // TwoSum (six operations) and the carry of the two children
  float s = __fadd_rn(l.s, r.s);
  float bb = __fsub_rn(s, l.s);
  float e = __fadd_rn(__fsub_rn(l.s, __fsub_rn(s, bb)), __fsub_rn(r.s, bb));
  float c = __fadd_rn(__fadd_rn(l.c, r.c), e);
  return TS{s, c};
}

// Node of the pass-2 trees: compensated d^2 tree and plain d tree together.
struct N2 {
  TS q;
  float d;
};
__device__ __forceinline__ N2 n2_combine(N2 l, N2 r) { return N2{ts_combine(l.q, r.q), __fadd_rn(l.d, r.d)}; }
__device__ __forceinline__ float f_combine(float l, float r) { return __fadd_rn(l, r); }

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

template <typename Node> __device__ __forceinline__ Node shfl_down_node(Node v, int d);
template <> __device__ __forceinline__ float shfl_down_node<float>(float v, int d) {
  return __shfl_down_sync(0xffffffffu, v, d);
}
template <> __device__ __forceinline__ N2 shfl_down_node<N2>(N2 v, int d) {
  return N2{TS{__shfl_down_sync(0xffffffffu, v.q.s, d), __shfl_down_sync(0xffffffffu, v.q.c, d)},
            __shfl_down_sync(0xffffffffu, v.d, d)};
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
    Node o = shfl_down_node<Node>(v, d);
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

__device__ __forceinline__ float max_nan0(float v) {
  if (v != v) return v;
  return v > 0.0f ? v : 0.0f;
}

// Row kernel (axis 1): one block per row, thread t owns leaves [t C, t C + C).
// MODE 0: the variance kernel; MODE 1: the formula of reference.
template <int MODE>
__global__ void __launch_bounds__(1024) var_rows_kernel(const float* __restrict__ x, int64_t rows, int64_t cols,
                                                        int ddof, float* __restrict__ out, float* __restrict__ mean_out,
                                                        int64_t C) {
  __shared__ float smf[32];
  __shared__ N2 sm2[32];
  __shared__ bool smv[32];
  __shared__ float bc[2];
  const int64_t n = cols;
  const float nf = (float)n;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const float* row = x + r * cols;
    const float x0 = row[0];
    int64_t b = (int64_t)threadIdx.x * C;
    int64_t m = n - b;
    m = m < 0 ? 0 : (m > C ? C : m);
    // pass 1: sum of y (kernel) or of x (reference)
    Stack<float, 40> st1;
    st1.reset();
    for (int64_t i = 0; i < m; ++i) {
      float leaf = (MODE == 0) ? __fsub_rn(row[b + i], x0) : row[b + i];
      st1.push(leaf, f_combine);
    }
    float v1 = 0.0f;
    bool h1 = st1.root(v1, f_combine);
    float sum1 = tree_combine_block<float>(v1, h1, blockDim.x, smf, smv, f_combine);
    if (threadIdx.x == 0)
      bc[0] = (MODE == 0) ? __fdiv_rn(sum1, nf) : __fmul_rn(sum1, __fdiv_rn(1.0f, nf));
    __syncthreads();
    const float mu = bc[0];
    // pass 2: d = y - m (kernel) or x - m (reference); compensated tree of d^2
    // (kernel) or plain tree of d^2 (reference), plain tree of d
    Stack<N2, 40> st2;
    st2.reset();
    for (int64_t i = 0; i < m; ++i) {
      float xi = row[b + i];
      float d = (MODE == 0) ? __fsub_rn(__fsub_rn(xi, x0), mu) : __fsub_rn(xi, mu);
      st2.push(N2{TS{__fmul_rn(d, d), 0.0f}, d}, n2_combine);
    }
    N2 v2;
    bool h2 = st2.root(v2, n2_combine);
    N2 tot = tree_combine_block<N2>(v2, h2, blockDim.x, sm2, smv, n2_combine);
    if (threadIdx.x == 0) {
      float var;
      if (MODE == 0) {
        float s2 = __fadd_rn(tot.q.s, tot.q.c);
        float t = __fdiv_rn(tot.d, nf);
        var = max_nan0(__fsub_rn(__fdiv_rn(s2, nf), __fmul_rn(t, t)));
      } else {
        float inv = __fdiv_rn(1.0f, nf);
        float md = __fmul_rn(tot.d, inv);
        var = max_nan0(__fsub_rn(__fmul_rn(tot.q.s, inv), __fmul_rn(md, md)));
      }
      if (ddof != 0) var = __fmul_rn(var, __fdiv_rn(nf, (float)(n - ddof)));
      out[r] = var;
      if (mean_out) mean_out[r] = (MODE == 0) ? __fadd_rn(x0, mu) : mu;
    }
    __syncthreads();
  }
}

// The reference formula's d^2 tree must be a plain tree: a TwoSum node whose
// carry is ignored has the same sum s as a plain add, so the MODE 1 kernel
// reads tot.q.s only.

// Column kernel (axis 0): a block covers 32 adjacent columns (threadIdx.x)
// and G row groups (threadIdx.y); group g owns rows [g C, g C + C).
template <int MODE>
__global__ void __launch_bounds__(256) var_cols_kernel(const float* __restrict__ x, int64_t rows, int64_t cols,
                                                       int ddof, float* __restrict__ out, float* __restrict__ mean_out,
                                                       int64_t C) {
  __shared__ float smf[8][32];
  __shared__ N2 sm2[8][32];
  __shared__ bool smv[8][32];
  __shared__ float bc[32];
  const int G = blockDim.y;
  const int64_t n = rows;
  const float nf = (float)n;
  const int64_t c = (int64_t)blockIdx.x * 32 + threadIdx.x;
  const bool col_ok = c < cols;
  const int g = threadIdx.y;
  int64_t b = (int64_t)g * C;
  int64_t m = n - b;
  m = m < 0 ? 0 : (m > C ? C : m);
  if (!col_ok) m = 0;
  const float x0 = col_ok ? x[c] : 0.0f;
  Stack<float, 40> st1;
  st1.reset();
  for (int64_t i = 0; i < m; ++i) {
    float xi = x[(b + i) * cols + c];
    st1.push((MODE == 0) ? __fsub_rn(xi, x0) : xi, f_combine);
  }
  float v1 = 0.0f;
  bool h1 = st1.root(v1, f_combine);
  smf[g][threadIdx.x] = v1;
  smv[g][threadIdx.x] = h1;
  __syncthreads();
  if (g == 0) {
    for (int step = 1; step < G; step <<= 1)
      for (int w = 0; w + step < G; w += 2 * step) {
        if (smv[w][threadIdx.x] && smv[w + step][threadIdx.x])
          smf[w][threadIdx.x] = __fadd_rn(smf[w][threadIdx.x], smf[w + step][threadIdx.x]);
        else if (!smv[w][threadIdx.x] && smv[w + step][threadIdx.x]) {
          smf[w][threadIdx.x] = smf[w + step][threadIdx.x];
          smv[w][threadIdx.x] = true;
        }
      }
    float s = smf[0][threadIdx.x];
    bc[threadIdx.x] = (MODE == 0) ? __fdiv_rn(s, nf) : __fmul_rn(s, __fdiv_rn(1.0f, nf));
  }
  __syncthreads();
  const float mu = bc[threadIdx.x];
  Stack<N2, 40> st2;
  st2.reset();
  for (int64_t i = 0; i < m; ++i) {
    float xi = x[(b + i) * cols + c];
    float d = (MODE == 0) ? __fsub_rn(__fsub_rn(xi, x0), mu) : __fsub_rn(xi, mu);
    st2.push(N2{TS{__fmul_rn(d, d), 0.0f}, d}, n2_combine);
  }
  N2 v2;
  bool h2 = st2.root(v2, n2_combine);
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
    N2 tot = sm2[0][threadIdx.x];
    float var;
    if (MODE == 0) {
      float s2 = __fadd_rn(tot.q.s, tot.q.c);
      float t = __fdiv_rn(tot.d, nf);
      var = max_nan0(__fsub_rn(__fdiv_rn(s2, nf), __fmul_rn(t, t)));
    } else {
      float inv = __fdiv_rn(1.0f, nf);
      float md = __fmul_rn(tot.d, inv);
      var = max_nan0(__fsub_rn(__fmul_rn(tot.q.s, inv), __fmul_rn(md, md)));
    }
    if (ddof != 0) var = __fmul_rn(var, __fdiv_rn(nf, (float)(n - ddof)));
    out[c] = var;
    if (mean_out) mean_out[c] = (MODE == 0) ? __fadd_rn(x0, mu) : mu;
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

template <int C, int MODE>
__global__ void __launch_bounds__(256) var_rows_reg(const float* __restrict__ x, int64_t rows, int64_t cols, int ddof,
                                                    float* __restrict__ out, float* __restrict__ mean_out) {
  __shared__ float smf[32];
  __shared__ N2 sm2[32];
  __shared__ bool smv[32];
  __shared__ float bc[1];
  const int n = (int)cols;
  const float nf = (float)n;
  const int b = threadIdx.x * C;
  int m = n - b;
  m = m < 0 ? 0 : (m > C ? C : m);
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const float* row = x + r * cols;
    const float x0 = __ldg(row);
    float v[C];
    if (C % 4 == 0 && m == C && ((((uintptr_t)(row + b)) & 15) == 0)) {
#pragma unroll
      for (int u = 0; u < C / 4; ++u) {
        float4 q = __ldcs((const float4*)(row + b) + u);
        v[4 * u] = q.x; v[4 * u + 1] = q.y; v[4 * u + 2] = q.z; v[4 * u + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < C; ++i) v[i] = (i < m) ? row[b + i] : 0.0f;
    }
    // pass 1
    float t1[C];
#pragma unroll
    for (int i = 0; i < C; ++i) t1[i] = (MODE == 0) ? __fsub_rn(v[i], x0) : v[i];
    bool h1 = reg_tree<float, C>(t1, m, f_combine);
    float sum1 = tree_combine_block<float>(t1[0], h1, blockDim.x, smf, smv, f_combine);
    if (threadIdx.x == 0) bc[0] = (MODE == 0) ? __fdiv_rn(sum1, nf) : __fmul_rn(sum1, __fdiv_rn(1.0f, nf));
    __syncthreads();
    const float mu = bc[0];
    // pass 2
    N2 t2[C];
#pragma unroll
    for (int i = 0; i < C; ++i) {
      float d = (MODE == 0) ? __fsub_rn(__fsub_rn(v[i], x0), mu) : __fsub_rn(v[i], mu);
      t2[i] = N2{TS{__fmul_rn(d, d), 0.0f}, d};
    }
    bool h2 = reg_tree<N2, C>(t2, m, n2_combine);
    N2 tot = tree_combine_block<N2>(t2[0], h2, blockDim.x, sm2, smv, n2_combine);
    if (threadIdx.x == 0) {
      float var;
      if (MODE == 0) {
        float s2 = __fadd_rn(tot.q.s, tot.q.c);
        float t = __fdiv_rn(tot.d, nf);
        var = max_nan0(__fsub_rn(__fdiv_rn(s2, nf), __fmul_rn(t, t)));
      } else {
        float inv = __fdiv_rn(1.0f, nf);
        float md = __fmul_rn(tot.d, inv);
        var = max_nan0(__fsub_rn(__fmul_rn(tot.q.s, inv), __fmul_rn(md, md)));
      }
      if (ddof != 0) var = __fmul_rn(var, __fdiv_rn(nf, (float)(n - ddof)));
      out[r] = var;
      if (mean_out) mean_out[r] = (MODE == 0) ? __fadd_rn(x0, mu) : mu;
    }
    __syncthreads();
  }
}

template <int MODE>
static void launch_rows_reg(int64_t C, const float* x, int64_t rows, int64_t cols, int ddof, float* out, float* mean,
                            unsigned grid, cudaStream_t s) {
  switch (C) {
    case 1: var_rows_reg<1, MODE><<<grid, 256, 0, s>>>(x, rows, cols, ddof, out, mean); break;
    case 2: var_rows_reg<2, MODE><<<grid, 256, 0, s>>>(x, rows, cols, ddof, out, mean); break;
    case 4: var_rows_reg<4, MODE><<<grid, 256, 0, s>>>(x, rows, cols, ddof, out, mean); break;
    case 8: var_rows_reg<8, MODE><<<grid, 256, 0, s>>>(x, rows, cols, ddof, out, mean); break;
    default: var_rows_reg<16, MODE><<<grid, 256, 0, s>>>(x, rows, cols, ddof, out, mean); break;
  }
}

static int64_t pow2_ceil(int64_t v) {
  int64_t p = 1;
  while (p < v) p <<= 1;
  return p;
}

size_t var_workspace_bytes(int64_t, int64_t, int) { return 0; }

cudaError_t launch_var(const float* x, int64_t rows, int64_t cols, int axis, int ddof, float* out, float* mean,
                       int twoterm, unsigned char*, cudaStream_t s) {
  if (axis == 1) {
    int block = 256;
    int64_t np = pow2_ceil(cols);
    int64_t C = np / block;
    if (C < 1) C = 1;
    int64_t grid = rows < 65535 * 16 ? rows : 65535 * 16;
    if (C <= 16) {
      if (twoterm) launch_rows_reg<1>(C, x, rows, cols, ddof, out, mean, (unsigned)grid, s);
      else launch_rows_reg<0>(C, x, rows, cols, ddof, out, mean, (unsigned)grid, s);
      return cudaGetLastError();
    }
    if (twoterm)
      var_rows_kernel<1><<<(unsigned)grid, block, 0, s>>>(x, rows, cols, ddof, out, mean, C);
    else
      var_rows_kernel<0><<<(unsigned)grid, block, 0, s>>>(x, rows, cols, ddof, out, mean, C);
  } else {
    int G = 8;
    int64_t np = pow2_ceil(rows);
    int64_t C = np / G;
    if (C < 1) C = 1;
    dim3 block(32, G);
    unsigned grid = (unsigned)((cols + 31) / 32);
    if (twoterm)
      var_cols_kernel<1><<<grid, block, 0, s>>>(x, rows, cols, ddof, out, mean, C);
    else
      var_cols_kernel<0><<<grid, block, 0, s>>>(x, rows, cols, ddof, out, mean, C);
  }
  return cudaGetLastError();
}

}  // namespace repro
