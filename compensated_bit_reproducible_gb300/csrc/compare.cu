// Comparison summation modes ("Reduction order and compensation solve related
// but different problems"; "Kahan's Summation Formula") and the environment
// probe ("SyclReproSum", "Runtime environment validation").
#include <cuda_runtime.h>
#include <cstdint>
#include "launch.h"

namespace repro {

// ------------------------------------------------------------------ naive
// Plain parallel reduction: per-thread running sums over a grid-stride walk,
// warp and block trees, last block adds the block sums.  The order (and so
// the rounding) depends on the launch shape.
template <typename T>
__global__ void __launch_bounds__(256) naive_kernel(const T* __restrict__ x, int64_t n, T* part, unsigned* ticket,
                                                    T* result) {
  __shared__ T sw[32];
  __shared__ bool last;
  T s = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    s += x[i];
  for (int d = 16; d >= 1; d >>= 1) s += __shfl_down_sync(0xffffffffu, s, d);
  if ((threadIdx.x & 31) == 0) sw[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    T b = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) b += sw[w];
    part[blockIdx.x] = b;
    __threadfence();
    last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    __threadfence();
    T t = 0;
    for (unsigned b = 0; b < gridDim.x; ++b) t += ((volatile T*)part)[b];
    *result = t;
    *ticket = 0;
  }
}

// --------------------------------------------------------------- pairwise
// Adjacent-pair tree over x[0..n) (pass-through of an unpaired last node).
// Level 1: each block reduces 4096 leaves (thread t: 16 leaves), block roots
// written with a presence flag; level 2 (one block) builds the tree over the
// roots with a binary-counter stack per thread.
template <typename T>
__device__ __forceinline__ T tree16(const T* v, int m) {
  // adjacent-pair tree over v[0..m), m <= 16
  T a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = v[i];
  int cnt = m;
#pragma unroll
  for (int w = 16; w > 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w / 2; ++i) {
      if (2 * i + 1 < cnt) a[i] = a[2 * i] + a[2 * i + 1];
      else if (2 * i < cnt) a[i] = a[2 * i];
    }
    cnt = (cnt + 1) / 2;
  }
  return a[0];
}

template <typename T>
__device__ T block_tree(T v, bool have, T* sm, int* smv) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int d = 1; d < 32; d <<= 1) {
    T o = __shfl_down_sync(0xffffffffu, v, d);
    bool oh = __shfl_down_sync(0xffffffffu, (int)have, d);
    if ((lane & (2 * d - 1)) == 0) {
      if (have && oh) v = v + o;
      else if (!have && oh) { v = o; have = true; }
    }
  }
  if (lane == 0) { sm[warp] = v; smv[warp] = have; }
  __syncthreads();
  if (threadIdx.x == 0) {
    int nw = blockDim.x >> 5;
    for (int step = 1; step < nw; step <<= 1)
      for (int w = 0; w + step < nw; w += 2 * step) {
        if (smv[w] && smv[w + step]) sm[w] = sm[w] + sm[w + step];
        else if (!smv[w] && smv[w + step]) { sm[w] = sm[w + step]; smv[w] = 1; }
      }
  }
  __syncthreads();
  return sm[0];
}

template <typename T>
__global__ void __launch_bounds__(256) pairwise_level1(const T* __restrict__ x, int64_t n, T* roots) {
  __shared__ T sm[8];
  __shared__ int smv[8];
  int64_t base = (int64_t)blockIdx.x * 4096 + (int64_t)threadIdx.x * 16;
  int m = (int)max((int64_t)0, min((int64_t)16, n - base));
  T v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = (i < m) ? x[base + i] : (T)0;
  T r = tree16<T>(v, m);
  T b = block_tree<T>(r, m > 0, sm, smv);
  if (threadIdx.x == 0) roots[blockIdx.x] = b;
}

// Tree over vals[0..nv) by one block: thread t owns [t C, t C + C).
template <typename T>
__global__ void __launch_bounds__(256) tree_over(const T* __restrict__ vals, int64_t nv, int64_t C, T* result) {
  __shared__ T sm[8];
  __shared__ int smv[8];
  int64_t b = (int64_t)threadIdx.x * C;
  int64_t m = max((int64_t)0, min(C, nv - b));
  T st[64];
  int64_t count = 0;
  for (int64_t i = 0; i < m; ++i) {
    T v = vals[b + i];
    int lvl = 0;
    int64_t c = count;
    while (c & 1) { v = st[lvl] + v; c >>= 1; ++lvl; }
    st[lvl] = v;
    ++count;
  }
  T acc = 0;
  bool have = false;
  for (int lvl = 0; lvl < 64; ++lvl)
    if ((count >> lvl) & 1) { acc = have ? st[lvl] + acc : st[lvl]; have = true; }
  T r = block_tree<T>(acc, have, sm, smv);
  if (threadIdx.x == 0) *result = (nv > 0) ? r : (T)0;
}

// ---------------------------------------------------- chunked compensated
template <typename T>
__global__ void __launch_bounds__(256) kahan_chunks(const T* __restrict__ x, int64_t n, int64_t chunk, int neumaier,
                                                    T* out) {
  int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t b = c * chunk;
  if (b >= n) return;
  int64_t e = min(n, b + chunk);
  T s = 0, cc = 0;
  if (!neumaier) {
    for (int64_t i = b; i < e; ++i) {
      T y = x[i] - cc;
      T t = s + y;
      cc = (t - s) - y;
      s = t;
    }
    out[c] = s;
  } else {
    for (int64_t i = b; i < e; ++i) {
      T xi = x[i];
      T t = s + xi;
      if (fabs((double)s) >= fabs((double)xi)) cc = cc + ((s - t) + xi);
      else cc = cc + ((xi - t) + s);
      s = t;
    }
    out[c] = s + cc;
  }
}

static int64_t p2ceil(int64_t v) {
  int64_t p = 1;
  while (p < v) p <<= 1;
  return p;
}

template <typename T>
size_t compare_workspace_bytes(int64_t n, int mode) {
  if (mode == 0) return 256 + 2048 * sizeof(T);
  if (mode == 1) return ((n + 4095) / 4096 + 1) * sizeof(T) + 64;
  return ((n + COMPENSATED_CHUNK - 1) / COMPENSATED_CHUNK + 1) * sizeof(T) + 64;
}

template <typename T>
cudaError_t launch_compare(const T* x, int64_t n, int mode, T* result, unsigned char* ws, cudaStream_t s) {
  if (mode == 0) {
    unsigned* ticket = (unsigned*)ws;
    T* part = (T*)(ws + 256);
    int grid = (int)min((int64_t)2048, max((int64_t)1, (n + 4095) / 4096));
    naive_kernel<T><<<grid, 256, 0, s>>>(x, n, part, ticket, result);
  } else {
    int64_t per = (mode == 1) ? 4096 : COMPENSATED_CHUNK;
    int64_t nv = (n + per - 1) / per;
    T* vals = (T*)ws;
    if (nv > 0) {
      if (mode == 1) pairwise_level1<T><<<(unsigned)nv, 256, 0, s>>>(x, n, vals);
      else kahan_chunks<T><<<(unsigned)((nv + 255) / 256), 256, 0, s>>>(x, n, per, mode == 3, vals);
    }
    int64_t C = p2ceil(nv) / 256;
    if (C < 1) C = 1;
    tree_over<T><<<1, 256, 0, s>>>(vals, nv, C, result);
  }
  return cudaGetLastError();
}

template size_t compare_workspace_bytes<float>(int64_t, int);
template size_t compare_workspace_bytes<double>(int64_t, int);
template cudaError_t launch_compare<float>(const float*, int64_t, int, float*, unsigned char*, cudaStream_t);
template cudaError_t launch_compare<double>(const double*, int64_t, int, double*, unsigned char*, cudaStream_t);

// ------------------------------------------------------------ environment
// Each failed check sets one bit of *out.  Operands come from kernel
// arguments so nothing folds at compile time.
__global__ void env_probe_kernel(unsigned* out, float one, float tiny_f, double oned, double tiny_d) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  unsigned bad = 0;
  // IEEE layouts
  if (__float_as_uint(one) != 0x3F800000u) bad |= 1u << 0;
  if ((uint64_t)__double_as_longlong(oned) != 0x3FF0000000000000ull) bad |= 1u << 1;
  // round to nearest, ties to even
  float h = __fmul_rn(one, 5.9604645e-08f);                // 2^-24
  if (__fadd_rn(one, h) != one) bad |= 1u << 2;             // 1 + ulp/2 -> 1 (even)
  float up = __fadd_rn(one, 1.1920929e-07f);                // 1 + 2^-23 (odd)
  if (__fadd_rn(up, h) != __fadd_rn(one, 2.3841858e-07f)) bad |= 1u << 3;   // -> 1 + 2^-22
  double hd = oned * 1.1102230246251565e-16;                 // 2^-53
  if (__dadd_rn(oned, hd) != oned) bad |= 1u << 4;
  // subnormals kept (no flush to zero)
  float sub = __fmul_rn(tiny_f, 0.5f);                      // 2^-127
  if (sub == 0.0f || __fadd_rn(sub, sub) != tiny_f) bad |= 1u << 5;
  double subd = __dmul_rn(tiny_d, 0.5);
  if (subd == 0.0 || __dadd_rn(subd, subd) != tiny_d) bad |= 1u << 6;
  // signed zero
  float nz = __fmul_rn(-one, 0.0f);
  if (__float_as_uint(__fadd_rn(nz, nz)) != 0x80000000u) bad |= 1u << 7;
  // Inf / NaN arithmetic
  float inf = __fdiv_rn(one, 0.0f);
  float nan = __fsub_rn(inf, inf);
  if (!(inf > 3.0e38f) || nan == nan) bad |= 1u << 8;
  *out = bad;
}

cudaError_t launch_env_probe(unsigned* out, cudaStream_t s) {
  env_probe_kernel<<<1, 32, 0, s>>>(out, 1.0f, 1.17549435e-38f, 1.0, 2.2250738585072014e-308);
  return cudaGetLastError();
}

}  // namespace repro
