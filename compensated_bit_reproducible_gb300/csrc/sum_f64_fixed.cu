// Double binned sum (K = 2, 3) at an index fixed before the deposit.
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
// the rounding bit of fold K-2 is set, in which case toward zero.
//
// So when I is known, a deposit is one rounding of |x| at g_f plus an exact
// integer addition.  This kernel guesses I from a sample of the input (a
// subset's maximum can only lie in the same bin as the true maximum or a
// finer one), deposits every element at that index, and checks the guess
// with the running maximum.  If any element lies outside the guessed bin or
// is Inf/NaN, or the index is too fine for the shortcuts below, it sets a
// flag and the general one-pass kernel (launched right after, idle unless
// the flag is set) recomputes the sum.  Both paths give the same bits.
//
// Accumulation.  With P' = |x| * 2^64 / g_f = M * 2^u (M the 53-bit
// significand), the rounded value is floor((P' + 2^63 - b) / 2^64), b the
// tie bit above.  Adding h - b to M (h = 2^(63-u)) and shifting by u gives
// P'' whose bits at and above 64 are exactly that value, so its 32-bit words
// at positions >= 2 can be summed independently, discarding words 0 and 1.
// Each thread keeps one 64-bit cell per word position (and sign) in shared
// memory: M + h - b shifted by u & 31 is three words w0, w1, w2 that land at
// word positions c, c + 1, c + 2 with c = u >> 5 -- an add into three cells
// and no variable-width shifting of a wide accumulator.  The top word w2 is
// below 2^22, so it goes to a 32-bit cell (1024 additions fit) that is
// folded into the 64-bit cells every 992 deposits.
#include "accum.cuh"
#include "launch.h"

namespace repro {

namespace {

constexpr int FX_U = 4;           // 16-byte vectors per thread per step
constexpr int FX_J = 4;           // steps per chunk
constexpr int FX_SAMPLE = 256;    // elements sampled for the index guess
constexpr int FX_STRIDE = 7;      // cells per sign: word positions 0..6
constexpr int FX_CELLS = 14;      // both signs
constexpr int FX_FOLD_CHUNKS = 31;   // 31 chunks x 32 deposits < 1024

// Control words in the zeroed workspace header.
struct FixedCtl {
  unsigned queue;    // next chunk of the dynamic queue
  unsigned ticket;   // finished blocks
  unsigned fail;     // nonzero: the general pass computes the result
};

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

// One deposit.  A: 64-bit cells (stride NT), B: 32-bit cells; sign s word k
// at cell k + 7 s (B: k - 2 + 7 s, only k >= 2 is used).
__device__ __forceinline__ void fx_deposit(uint32_t hi, uint32_t lo, const FxConst& k, uint64_t* A, uint32_t* B,
                                           uint32_t NT, int& umax) {
  uint32_t eb = mad32(hi, k.one + k.one, 0u) >> 21;          // biased exponent
  int us = (int)mad32(eb, k.one, k.Cp);                       // shift of M
  umax = max(umax, us);
  uint32_t u = (uint32_t)max(us, 0);   // tiny values: their words stay below position 2
  uint32_t c = min(u >> 5, 5u);        // beyond the bin (flagged through umax): kept in bounds
  uint32_t mh = (hi & 0xFFFFFu) | 0x100000u;
  uint32_t hl = shl_clamp32(1u, (int)mad32(u, k.negone, k.c63));
  uint32_t hh = shl_clamp32(1u, (int)mad32(u, k.negone, k.c31));
  uint32_t b = min(mh & mad32(hl, k.c256, 0u), 1u);          // bit 103 of P': rounding bit of fold K-2
  uint64_t Mp = ((((uint64_t)mh) << 32) | lo) + ((((uint64_t)hh) << 32) | hl) - (uint64_t)b;
  uint32_t lo2 = (uint32_t)Mp, mh2 = (uint32_t)(Mp >> 32);
  uint32_t w0 = funnel_l(0u, lo2, u);
  uint32_t w1 = funnel_l(lo2, mh2, u);
  uint32_t w2 = funnel_l(mh2, 0u, u);
  uint32_t off = mad32(mad32(hi >> 31, k.c7, c), NT, 0u);
  uint64_t* p = A + off;
  uint32_t* pb = B + off;
  p[0] = madw(w0, k.one, p[0]);
  p[NT] = madw(w1, k.one, p[NT]);
  pb[0] = mad32(w2, k.one, pb[0]);
}

__device__ __forceinline__ void fx_fold(uint64_t* A, uint32_t* B, uint32_t NT) {
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int w = 2; w < FX_STRIDE; ++w) {
      A[(w + FX_STRIDE * s) * NT] += B[(w - 2 + FX_STRIDE * s) * NT];
      B[(w - 2 + FX_STRIDE * s) * NT] = 0;
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

// Block sum of the thread cells into a signed 192-bit total (units of g_f),
// valid in thread 0.  `scratch` (32 x 10 W128) may alias the cells: they are
// read into registers before it is written.
__device__ I192 fx_block_total(const uint64_t* A, uint32_t NT, W128 (*red)[10]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (int)(NT >> 5);
  W128 col[10];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int w = 2; w < FX_STRIDE; ++w) col[s * 5 + (w - 2)] = W128{A[(w + FX_STRIDE * s) * NT], 0};
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 10; ++i) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) col[i] = w_add(col[i], shfl_xor_w(col[i], m));
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < 10; ++i) red[warp][i] = col[i];
  }
  __syncthreads();
  I192 t{0, 0, 0};
  if (threadIdx.x == 0) {
    for (int i = 0; i < 10; ++i) {
      W128 s = W128{0, 0};
      for (int w = 0; w < nw; ++w) s = w_add(s, red[w][i]);
      I192 v = i192_from_shifted(s, i % 5);
      t = i192_add(t, i < 5 ? v : i192_neg(v));
    }
  }
  return t;
}

}  // namespace

// Workspace: ctl (zeroed with the header) and one 24-byte partial per block.
// CNT: the block size as a compile-time constant (128 or 256: registers
// capped for 10 resp. 5 resident blocks per SM, cell offsets folded into the
// addressing), or 0 for any block size up to 1024.
constexpr int fx_max_threads(int cnt) { return cnt ? cnt : 1024; }
constexpr int fx_min_blocks(int cnt) { return cnt ? 1280 / (cnt ? cnt : 1) : 1; }

template <int K, int CNT>
__global__ void __launch_bounds__(fx_max_threads(CNT), fx_min_blocks(CNT))
    sum_f64_fixed_kernel(const double* __restrict__ x, int64_t n, uint32_t one, FixedCtl* ctl,
                         unsigned char* __restrict__ parts, double* __restrict__ result) {
  extern __shared__ __align__(16) unsigned char fx_smem[];
  const uint32_t NT = CNT ? (uint32_t)CNT : blockDim.x;
  uint64_t* A = (uint64_t*)fx_smem + threadIdx.x;
  uint32_t* B = (uint32_t*)(fx_smem + (size_t)FX_CELLS * 8 * NT) + threadIdx.x;
  __shared__ unsigned s_emax;

  // the gated fallback kernel may start launching now; it waits for this
  // grid to complete before it reads the flag
  asm volatile("griddepcontrol.launch_dependents;");
  // 1. Index guess: the largest exponent field over a fixed sample.
  if (threadIdx.x == 0) s_emax = 0;
  __syncthreads();
  {
    const int64_t S = n < FX_SAMPLE ? n : FX_SAMPLE;
    unsigned em = 0;
    for (int64_t j = threadIdx.x; j < S; j += NT) {
      int64_t pos = (j * n) / S;
      em = max(em, (unsigned)__double2hiint(__ldg(x + pos)) & 0x7FF00000u);
    }
    em = __reduce_max_sync(0xffffffffu, em);
    if ((threadIdx.x & 31) == 0) atomicMax(&s_emax, em);
  }
  __syncthreads();
  const int eb_max = (int)(s_emax >> 20);
  typedef Geom<double> G;
  int Ig;
  if (eb_max == 0) Ig = G::NB - K;
  else {
    int j = (G::B0 + G::W - 2 - (eb_max - 1023)) / G::W;
    Ig = min(j, G::NB - 1);
    Ig = min(Ig, G::NB - K);
  }
  const int bf = beta<double>(Ig + K - 1);
  // the shortcuts need g_f/2 above every subnormal and every x with a forced
  // hidden bit below the grid: beta_f >= -1019; Inf/NaN in the sample fail too
  bool usable = (bf >= -1019) && (eb_max < 0x7FF);
  FxConst kc;
  kc.one = one;
  kc.negone = 0u - one;
  kc.c63 = 63u * one;
  kc.c31 = 31u * one;
  kc.c256 = 256u * one;
  kc.c7 = (uint32_t)FX_STRIDE * one;
  kc.Cp = (uint32_t)(-1011 - bf);
  // largest valid shift: |x| < 2^(beta_I + W - 1), i.e. eb <= 1023 + beta_I + 38
  const int eb_thr = (Ig == 0) ? 2046 : 1023 + beta<double>(Ig) + G::W - 2;
  const int u_thr = eb_thr + (int)kc.Cp;

  // 2. Deposits: full chunks from a dynamic queue, then the ragged rest.
#pragma unroll
  for (int w = 0; w < FX_CELLS; ++w) {
    A[w * NT] = 0;
    B[w * NT] = 0;
  }
  int umax = -1;
  int64_t head = (int64_t)(((16 - ((uintptr_t)x & 15)) & 15) / 8);
  if (head > n) head = n;
  const double2* xv = (const double2*)(x + head);
  const int64_t nv = (n - head) / 2;
  const int64_t CV = (int64_t)NT * FX_U * FX_J;
  const int64_t nchunks = usable ? nv / CV : 0;
  int since = 0;
  // chunk numbers come from the queue one chunk ahead, so the atomic's
  // latency overlaps a chunk of deposits
  __shared__ unsigned s_q[2];
  if (threadIdx.x == 0) s_q[0] = nchunks > 0 ? atomicAdd(&ctl->queue, 1u) : 0u;
  __syncthreads();
  for (int slot = 0;; slot ^= 1) {
    const int64_t ch = s_q[slot];
    if (ch >= nchunks) break;   // same value in every thread of the block
    unsigned nxt = 0;
    if (threadIdx.x == 0) nxt = atomicAdd(&ctl->queue, 1u);
    const double2* base = xv + ch * CV + threadIdx.x;
#pragma unroll 1
    for (int j = 0; j < FX_J; ++j) {
      double2 v[FX_U];
#pragma unroll
      for (int q = 0; q < FX_U; ++q) v[q] = __ldcs(base + (int64_t)(j * FX_U + q) * NT);
#pragma unroll
      for (int q = 0; q < FX_U; ++q) {
        fx_deposit((uint32_t)__double2hiint(v[q].x), (uint32_t)__double2loint(v[q].x), kc, A, B, NT, umax);
        fx_deposit((uint32_t)__double2hiint(v[q].y), (uint32_t)__double2loint(v[q].y), kc, A, B, NT, umax);
      }
    }
    if (++since == FX_FOLD_CHUNKS) {
      fx_fold(A, B, NT);
      since = 0;
    }
    if (threadIdx.x == 0) s_q[slot ^ 1] = nxt;
    __syncthreads();
  }
  fx_fold(A, B, NT);
  if (usable) {
    // head element(s) and everything after the last full chunk
    const int64_t tail0 = head + 2 * nchunks * CV;
    const int64_t R = head + (n - tail0);
    const int64_t gt = (int64_t)blockIdx.x * NT + threadIdx.x, G_ = (int64_t)gridDim.x * NT;
    int cnt = 0;
    for (int64_t r = gt; r < R; r += G_) {
      double v = __ldg(x + (r < head ? r : tail0 + (r - head)));
      fx_deposit((uint32_t)__double2hiint(v), (uint32_t)__double2loint(v), kc, A, B, NT, umax);
      if (++cnt == 992) {
        fx_fold(A, B, NT);
        cnt = 0;
      }
    }
    fx_fold(A, B, NT);
  }
  const int fail = __syncthreads_or(!usable || umax > u_thr);

  // 3. Block total, partial, and the last block's merge and conversion.
  I192 t = fx_block_total(A, NT, (W128(*)[10])fx_smem);
  __shared__ bool last;
  if (threadIdx.x == 0) {
    I192* pp = (I192*)parts + blockIdx.x;
    *pp = t;
    if (fail) atomicOr(&ctl->fail, 1u);
    __threadfence();
    unsigned tk = atomicAdd(&ctl->ticket, 1u);
    last = (tk == gridDim.x - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (__ldcg(&ctl->fail)) return;   // the general pass writes the result
  I192 s{0, 0, 0};
  for (int p = threadIdx.x; p < (int)gridDim.x; p += NT) {
    const I192* q = (const I192*)parts + p;
    s = i192_add(s, I192{__ldcg(&q->w0), __ldcg(&q->w1), __ldcg(&q->w2)});
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) s = i192_add(s, i192_shfl_xor(s, m));
  I192* sw = (I192*)fx_smem;   // the cells are no longer needed
  if ((threadIdx.x & 31) == 0) sw[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    I192 tot{0, 0, 0};
    for (int w = 0; w < (int)(NT >> 5); ++w) tot = i192_add(tot, sw[w]);
    // folds of the total (any split with the right weighted sum converts alike)
    W128 F[K];
    const uint64_t m40 = (1ull << 40) - 1;
    F[K - 1] = W128{tot.w0 & m40, 0};
    if (K == 3) {
      F[1] = W128{((tot.w0 >> 40) | (tot.w1 << 24)) & m40, 0};
      // tot >> 80 (arithmetic)
      F[0] = W128{(tot.w1 >> 16) | (tot.w2 << 48), (int64_t)tot.w2 >> 16};
    } else {
      // tot >> 40 (arithmetic)
      F[0] = W128{(tot.w0 >> 40) | (tot.w1 << 24), (int64_t)((tot.w1 >> 40) | (tot.w2 << 24))};
    }
    *result = convert_fast<double, K>(Ig, 0, F);
  }
}

// ------------------------------------------------------------------ host
namespace {
// cells, and at least the epilogue's reduction scratch (32 x 10 W128)
size_t fx_smem_bytes(int block) {
  size_t cells = (size_t)block * FX_CELLS * 12;
  return cells > 5120 ? cells : 5120;
}

template <int K, int CNT>
int fixed_blocks_per_sm(int block) {
  static int cached[64][33] = {};   // per device and block / 32 (one table per K, CNT)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  int* slot = &cached[dev][block >> 5];
  if (*slot) return *slot;
  size_t smem = fx_smem_bytes(block);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(sum_f64_fixed_kernel<K, CNT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
  }
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, sum_f64_fixed_kernel<K, CNT>, block, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  *slot = nb;
  return nb;
}

template <int K>
int blocks_per_sm_k(int block) {
  if (block == 128) return fixed_blocks_per_sm<K, 128>(block);
  if (block == 256) return fixed_blocks_per_sm<K, 256>(block);
  return fixed_blocks_per_sm<K, 0>(block);
}

template <int K>
void launch_k(const double* x, int64_t n, unsigned* ctl, unsigned char* parts, double* result, int grid, int block,
              cudaStream_t s) {
  size_t smem = fx_smem_bytes(block);
  if (block == 128)
    sum_f64_fixed_kernel<K, 128><<<grid, block, smem, s>>>(x, n, 1u, (FixedCtl*)ctl, parts, result);
  else if (block == 256)
    sum_f64_fixed_kernel<K, 256><<<grid, block, smem, s>>>(x, n, 1u, (FixedCtl*)ctl, parts, result);
  else
    sum_f64_fixed_kernel<K, 0><<<grid, block, smem, s>>>(x, n, 1u, (FixedCtl*)ctl, parts, result);
}
}  // namespace

int sum_f64_fixed_grid(int K, int block, int sms) {
  if (K != 2 && K != 3) return 0;
  if (block < 32 || block > 1024 || (block & 31)) return 0;
  int nb = (K == 2) ? blocks_per_sm_k<2>(block) : blocks_per_sm_k<3>(block);
  return nb > 0 ? nb * sms : 0;
}

size_t sum_f64_fixed_workspace_bytes(int grid) { return (size_t)grid * sizeof(I192); }

cudaError_t launch_sum_f64_fixed(const double* x, int64_t n, int K, unsigned* ctl, unsigned char* parts,
                                 double* result, int grid, int block, cudaStream_t s) {
  // make sure the shared-memory attribute is set for this device and block size
  if (sum_f64_fixed_grid(K, block, 1) <= 0) return cudaErrorInvalidConfiguration;
  if (K == 2) launch_k<2>(x, n, ctl, parts, result, grid, block, s);
  else launch_k<3>(x, n, ctl, parts, result, grid, block, s);
  return cudaGetLastError();
}

}  // namespace repro
