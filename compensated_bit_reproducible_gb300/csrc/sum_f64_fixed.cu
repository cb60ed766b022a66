// Double binned sum (K = 2..6) at an index fixed before the deposit (see
// fixed_index.cuh for the reading this rests on).  If any element lies
// outside the guessed bin or is Inf/NaN, or the index is too fine for the
// shortcuts, the kernel sets a flag and the general one-pass kernel
// (launched right after, idle unless the flag is set) computes the sum.
// Both paths give the same bits.
//
// Accumulation.  M + h - b shifted by u & 31 is three 32-bit words w0, w1,
// w2 that land at word positions c, c + 1, c + 2 of P'' (c = u >> 5); words
// below position 2 are dropped.  Each thread keeps, per position and sign,
// a 64-bit cell for words c and c + 1 and a 32-bit cell for word c + 2 in
// shared memory; a deposit is one 96-bit add into that pair (the carry out
// of the 64-bit cell goes into the 32-bit one), with no variable-width shift
// of a wide accumulator.  The 32-bit cells are moved into the 64-bit ones
// every 992 deposits.  K sets only how many positions there are (7 for
// K <= 3, 10 for K = 6) and the width of the block total (192 or 320 bits):
// an element's three words are the same for any K.
#include "accum.cuh"
#include "fixed_index.cuh"
#include "launch.h"

namespace repro {

using namespace fx;

namespace {

constexpr int FX_U = 4;           // 16-byte vectors per thread per step
constexpr int FX_J = 4;           // steps per chunk
constexpr int FX_FOLD_CHUNKS = 31;   // 31 chunks x 32 deposits < 1024

// Control words in the zeroed workspace header.
struct FixedCtl {
  unsigned queue;    // next chunk of the dynamic queue
  unsigned ticket;   // finished blocks
  unsigned fail;     // nonzero: the general pass computes the result
};

}  // namespace

// Workspace: ctl (zeroed with the header) and one 24-byte partial per block.
// CNT: the block size as a compile-time constant (128 or 256: registers
// capped for 10 resp. 5 resident blocks per SM, cell offsets folded into the
// addressing), or 0 for any block size up to 1024.
// K >= 4: the larger cells fit seven 128-thread blocks per SM (three of 256).
constexpr int fx_max_threads(int cnt) { return cnt ? cnt : 1024; }
constexpr int fx_min_blocks(int cnt, int K) { return cnt ? (K <= 3 ? 1280 : 896) / (cnt ? cnt : 1) : 1; }

// Block totals: 192 bits for K <= 3, 320 bits for K = 4..6.
template <int K> struct FxTot { typedef I320 type; };
template <> struct FxTot<2> { typedef I192 type; };
template <> struct FxTot<3> { typedef I192 type; };

// Folds of a total for the conversion (any split with the right weighted sum
// converts alike): 40-bit fields from the bottom, the rest (arithmetic) on top.
template <int K>
__device__ __forceinline__ void fx_folds(const I192& tot, W128* F) {
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
}
template <int K>
__device__ __forceinline__ void fx_folds(const I320& tot, W128* F) {
  const uint64_t m40 = (1ull << 40) - 1;
#pragma unroll
  for (int j = 0; j < K - 1; ++j) {
    const int a = (40 * j) >> 6, b = (40 * j) & 63;
    uint64_t v = tot.w[a] >> b;
    if (b > 24) v |= tot.w[a + 1] << (64 - b);
    F[K - 1 - j] = W128{v & m40, 0};
  }
  // tot >> 40 (K - 1), arithmetic; the shift is 120, 160 or 200 (b != 0)
  constexpr int o = 40 * (K - 1), a = o >> 6, b = o & 63;
  const uint64_t lo = (tot.w[a] >> b) | (tot.w[a + 1] << (64 - b));
  uint64_t hi;
  if constexpr (a + 2 <= 4) hi = (tot.w[a + 1] >> b) | (tot.w[a + 2] << (64 - b));
  else hi = (uint64_t)((int64_t)tot.w[a + 1] >> b);
  F[0] = W128{lo, (int64_t)hi};
}

template <int K, int CNT>
__global__ void __launch_bounds__(fx_max_threads(CNT), fx_min_blocks(CNT, K))
    sum_f64_fixed_kernel(const double* __restrict__ x, int64_t n, uint32_t one, FixedCtl* ctl,
                         unsigned char* __restrict__ parts, double* __restrict__ result) {
  extern __shared__ __align__(16) unsigned char fx_smem[];
  const uint32_t NT = CNT ? (uint32_t)CNT : blockDim.x;
  uint64_t* A = (uint64_t*)fx_smem + threadIdx.x;
  typedef FxGeo<K> Geo;
  typedef typename FxTot<K>::type Tot;
  uint32_t* B = (uint32_t*)(fx_smem + (size_t)Geo::CELLS * 8 * NT) + threadIdx.x;
  __shared__ unsigned s_emax;

  // the gated fallback kernel may start launching now; it waits for this
  // grid to complete before it reads the flag
  asm volatile("griddepcontrol.launch_dependents;");
  // 1. Index guess from a sample.
  int eb_max;
  const int Ig = guess_index<double>(x, n, K, &s_emax, &eb_max);
  const int bf = beta<double>(Ig + K - 1);
  // the shortcuts need g_f/2 above every subnormal and every x with a forced
  // hidden bit below the grid: beta_f >= -1019; Inf/NaN in the sample fail too
  const bool usable = (bf >= -1019) && (eb_max < 0x7FF);
  const FxConst kc = make_const(bf, one, Geo::STR - 1);   // cell pairs per sign
  // largest valid shift: the top of bin Ig
  const int u_thr = bin_top_exponent<double>(Ig) + (int)kc.Cp;

  // 2. Deposits: full chunks from a dynamic queue, then the ragged rest.
#pragma unroll
  for (int w = 0; w < Geo::CELLS; ++w) {
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
        fx_deposit<Geo::STR>((uint32_t)__double2hiint(v[q].x), (uint32_t)__double2loint(v[q].x), kc, A, B, NT,
                             umax);
        fx_deposit<Geo::STR>((uint32_t)__double2hiint(v[q].y), (uint32_t)__double2loint(v[q].y), kc, A, B, NT,
                             umax);
      }
    }
    if (++since == FX_FOLD_CHUNKS) {
      fx_fold<Geo::STR>(A, B, NT);
      since = 0;
    }
    if (threadIdx.x == 0) s_q[slot ^ 1] = nxt;
    __syncthreads();
  }
  fx_fold<Geo::STR>(A, B, NT);
  if (usable) {
    // head element(s) and everything after the last full chunk
    const int64_t tail0 = head + 2 * nchunks * CV;
    const int64_t R = head + (n - tail0);
    const int64_t gt = (int64_t)blockIdx.x * NT + threadIdx.x, G_ = (int64_t)gridDim.x * NT;
    int cnt = 0;
    for (int64_t r = gt; r < R; r += G_) {
      double v = __ldg(x + (r < head ? r : tail0 + (r - head)));
      fx_deposit<Geo::STR>((uint32_t)__double2hiint(v), (uint32_t)__double2loint(v), kc, A, B, NT, umax);
      if (++cnt == 992) {
        fx_fold<Geo::STR>(A, B, NT);
        cnt = 0;
      }
    }
    fx_fold<Geo::STR>(A, B, NT);
  }
  const int fail = __syncthreads_or(!usable || umax > u_thr);

  // 3. Block total, partial, and the last block's merge and conversion.
  Tot t = fx_block_total_t<Geo::STR, Tot>(A, B, NT, (W128(*)[2 * Geo::NPOS])fx_smem);
  __shared__ bool last;
  if (threadIdx.x == 0) {
    Tot* pp = (Tot*)parts + blockIdx.x;
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
  Tot s{};
  for (int p = threadIdx.x; p < (int)gridDim.x; p += NT) s = tot_add(s, tot_ldcg((const Tot*)parts + p));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) s = tot_add(s, tot_shfl_xor(s, m));
  Tot* sw = (Tot*)fx_smem;   // the cells are no longer needed
  if ((threadIdx.x & 31) == 0) sw[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    Tot tot{};
    for (int w = 0; w < (int)(NT >> 5); ++w) tot = tot_add(tot, sw[w]);
    W128 F[K];
    fx_folds<K>(tot, F);
    *result = convert_fast<double, K>(Ig, 0, F);
  }
}

// ------------------------------------------------------------------ host
namespace {
// cells, and at least the epilogue's reduction scratch (32 warps x
// 2 (STR - 2) W128)
template <int K>
size_t fx_smem_bytes(int block) {
  const size_t cells = (size_t)block * FxGeo<K>::CELLS * 12;
  const size_t red = (size_t)32 * 2 * FxGeo<K>::NPOS * sizeof(W128);
  return cells > red ? cells : red;
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
  size_t smem = fx_smem_bytes<K>(block);
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
  size_t smem = fx_smem_bytes<K>(block);
  if (block == 128)
    sum_f64_fixed_kernel<K, 128><<<grid, block, smem, s>>>(x, n, 1u, (FixedCtl*)ctl, parts, result);
  else if (block == 256)
    sum_f64_fixed_kernel<K, 256><<<grid, block, smem, s>>>(x, n, 1u, (FixedCtl*)ctl, parts, result);
  else
    sum_f64_fixed_kernel<K, 0><<<grid, block, smem, s>>>(x, n, 1u, (FixedCtl*)ctl, parts, result);
}
}  // namespace

int sum_f64_fixed_grid(int K, int block, int sms) {
  if (block < 32 || block > 1024 || (block & 31)) return 0;
  int nb = 0;
  switch (K) {
    case 2: nb = blocks_per_sm_k<2>(block); break;
    case 3: nb = blocks_per_sm_k<3>(block); break;
    case 4: nb = blocks_per_sm_k<4>(block); break;
    case 5: nb = blocks_per_sm_k<5>(block); break;
    case 6: nb = blocks_per_sm_k<6>(block); break;
    default: return 0;
  }
  return nb > 0 ? nb * sms : 0;
}

// one partial per block, at the widest total's size
size_t sum_f64_fixed_workspace_bytes(int grid) { return (size_t)grid * sizeof(I320); }

cudaError_t launch_sum_f64_fixed(const double* x, int64_t n, int K, unsigned* ctl, unsigned char* parts,
                                 double* result, int grid, int block, cudaStream_t s) {
  // make sure the shared-memory attribute is set for this device and block size
  if (sum_f64_fixed_grid(K, block, 1) <= 0) return cudaErrorInvalidConfiguration;
  switch (K) {
    case 2: launch_k<2>(x, n, ctl, parts, result, grid, block, s); break;
    case 3: launch_k<3>(x, n, ctl, parts, result, grid, block, s); break;
    case 4: launch_k<4>(x, n, ctl, parts, result, grid, block, s); break;
    case 5: launch_k<5>(x, n, ctl, parts, result, grid, block, s); break;
    default: launch_k<6>(x, n, ctl, parts, result, grid, block, s); break;
  }
  return cudaGetLastError();
}

}  // namespace repro
