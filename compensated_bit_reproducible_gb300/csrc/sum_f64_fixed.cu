// Double binned sum (K = 2..6) at an index fixed before the deposit (see
// fixed_index.cuh for the reading this rests on).  The first pass guesses
// the index from a sample.  If any element lies outside the guessed bin or
// is Inf/NaN, or the index is too fine for its shortcut, it records the
// largest exponent field of the input, and the second pass (launched right
// after, idle otherwise) recomputes the sum at the index of that exponent,
// reading subnormals exactly, or finds which of Inf and NaN occur.  Both
// passes give the binned sum's bits.
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
#include <climits>
#include "accum.cuh"
#include "fixed_index.cuh"
#include "launch.h"

namespace repro {

using namespace fx;

namespace {

constexpr int FX_U = 4;           // 16-byte vectors per thread per step
constexpr int FX_J = 4;           // steps per chunk
constexpr int FX_FOLD_CHUNKS = 992 / (2 * FX_U * FX_J);   // chunks between folds: at most 992 deposits

// Control words, zero at launch and left zero by the two passes (the first
// pass's last block clears what it accumulated and sets run2; the second
// pass's last block clears that).  The block totals are summed by atomics
// as 32-bit digits in 64-bit accumulators (2^32 blocks before one could
// carry out), one accumulator per 128-byte line so that the blocks'
// additions to different digits do not queue on one line.
constexpr int FX_DIGITS = 10;   // 320-bit totals
constexpr int FX_DIG_STRIDE = 16;   // 64-bit words between two accumulators
struct FixedCtl {
  unsigned queue;     // next chunk of the dynamic queue (after the first gridDim.x)
  unsigned ticket;    // finished blocks
  unsigned spare;
  unsigned fail;      // some block of the first pass left the guessed bin
  unsigned emax;      // largest biased exponent field the first pass deposited
  unsigned run2;      // set by the first pass's last block: 1 the second pass deposits, 2 it scans for Inf/NaN
  int I2;             // the second pass's index (from emax)
  unsigned sflags;    // the second pass's Inf/NaN flags (emax all ones)
  unsigned pad[24];
  unsigned long long dig[FX_DIGITS * FX_DIG_STRIDE];
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

template <int K, int CNT, bool SECOND>
__global__ void __launch_bounds__(fx_max_threads(CNT), fx_min_blocks(CNT, K))
    sum_f64_fixed_kernel(const double* __restrict__ x, int64_t n, uint32_t one, FixedCtl* ctl,
                         double* __restrict__ result) {
  extern __shared__ __align__(16) unsigned char fx_smem[];
  const uint32_t NT = CNT ? (uint32_t)CNT : blockDim.x;
  uint64_t* A = (uint64_t*)fx_smem + threadIdx.x;
  typedef FxGeo<K> Geo;
  typedef typename FxTot<K>::type Tot;
  uint32_t* B = (uint32_t*)(fx_smem + (size_t)Geo::CELLS * 8 * NT) + threadIdx.x;
  __shared__ unsigned s_emax;

  __shared__ bool last;
  if constexpr (SECOND) {
    // the second pass: launched as a programmatic dependent of the first, it
    // waits for that grid and runs only if the first one asked for it
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const unsigned mode = __ldcg(&ctl->run2);
    if (mode == 0u) return;
    if (mode == 2u) {
      // the largest exponent field is all ones: the result is Inf or NaN,
      // set by which specials occur (one pass over the input, no deposits)
      __shared__ unsigned s_fl;
      if (threadIdx.x == 0) s_fl = 0u;
      __syncthreads();
      unsigned fl = 0u;
      const int64_t G_ = (int64_t)gridDim.x * NT;
      for (int64_t i = (int64_t)blockIdx.x * NT + threadIdx.x; i < n; i += G_) {
        const double v = __ldcs(x + i);
        if ((((uint32_t)__double2hiint(v)) & 0x7FF00000u) == 0x7FF00000u) fl |= (unsigned)special_flag<double>(v);
      }
      fl = __reduce_or_sync(0xffffffffu, fl);
      if ((threadIdx.x & 31) == 0 && fl) atomicOr(&s_fl, fl);
      __syncthreads();
      if (threadIdx.x == 0) {
        if (s_fl) atomicOr(&ctl->sflags, s_fl);
        __threadfence();
        last = atomicAdd(&ctl->ticket, 1u) == gridDim.x - 1;
      }
      __syncthreads();
      if (!last || threadIdx.x != 0) return;
      __threadfence();
      const int f = (int)__ldcg(&ctl->sflags);
      ctl->sflags = 0u;
      ctl->ticket = 0u;
      ctl->run2 = 0u;
      ctl->emax = 0u;
      *result = from_flags<double>(f);
      return;
    }
  } else {
    // the second pass may start launching now; it waits for this grid to
    // complete before it reads its flag
    asm volatile("griddepcontrol.launch_dependents;");
  }
  // Chunks of CV 16-byte vectors from the first 16-byte boundary on.  Block
  // b takes chunk b first and the rest from a dynamic queue; the first step
  // of chunk b is loaded before the index guess, so its latency overlaps
  // the sample's.
  int64_t head = (int64_t)(((16 - ((uintptr_t)x & 15)) & 15) / 8);
  if (head > n) head = n;
  const double2* xv = (const double2*)(x + head);
  const int64_t nv = (n - head) / 2;
  const int64_t CV = (int64_t)NT * FX_U * FX_J;
  const int64_t nch_all = nv / CV;
  double2 v0[FX_U];
  if ((int64_t)blockIdx.x < nch_all) {
#pragma unroll
    for (int q = 0; q < FX_U; ++q) v0[q] = __ldcs(xv + (int64_t)blockIdx.x * CV + threadIdx.x + (int64_t)q * NT);
  }
  // 1. Index: the first pass guesses it from a sample; the second takes the
  // one the first pass's last block derived from the largest exponent.
  int eb_max = 0;
  const int Ig = SECOND ? __ldcg(&ctl->I2) : guess_index<double>(x, n, K, &s_emax, &eb_max);
  const int bf = beta<double>(Ig + K - 1);
  // The first pass's shortcut (a forced hidden bit) needs g_f/2 above every
  // subnormal: beta_f >= -1019; Inf/NaN in the sample fail it too (it then
  // deposits nothing and only finds the largest exponent).  The second pass
  // reads subnormals exactly and its index holds every element.
  const bool usable = SECOND || ((bf >= -1019) && (eb_max < 0x7FF));
  const FxConst kc = make_const(bf, one, Geo::STR - 1);   // cell pairs per sign
  // largest valid shift: the top of bin Ig
  const int u_thr = bin_top_exponent<double>(Ig) + (int)kc.Cp;

  // 2. Deposits: full chunks, then the ragged rest.
#pragma unroll
  for (int w = 0; w < Geo::CELLS; ++w) {
    A[w * NT] = 0;
    B[w * NT] = 0;
  }
  int umax = INT_MIN / 2;   // largest shift seen
  const int64_t nchunks = usable ? nch_all : 0;
  int since = 0;
  // the next chunk number comes from the queue one chunk ahead, so the
  // atomic's latency overlaps a chunk of deposits
  __shared__ unsigned s_q[2];
  int64_t ch = blockIdx.x;   // same value in every thread of the block
  int j0 = 1;                // the first step of the first chunk is in v0
  if (ch < nchunks) {
#pragma unroll
    for (int q = 0; q < FX_U; ++q) {
      fx_deposit<Geo::STR, SECOND>((uint32_t)__double2hiint(v0[q].x), (uint32_t)__double2loint(v0[q].x), kc, A, B, NT, umax);
      fx_deposit<Geo::STR, SECOND>((uint32_t)__double2hiint(v0[q].y), (uint32_t)__double2loint(v0[q].y), kc, A, B, NT, umax);
    }
  }
  for (int slot = 0; ch < nchunks; slot ^= 1) {
    unsigned nxt = 0;
    if (threadIdx.x == 0) nxt = gridDim.x + atomicAdd(&ctl->queue, 1u);
    const double2* base = xv + ch * CV + threadIdx.x;
#pragma unroll 1
    for (int j = j0; j < FX_J; ++j) {
      double2 v[FX_U];
#pragma unroll
      for (int q = 0; q < FX_U; ++q) v[q] = __ldcs(base + (int64_t)(j * FX_U + q) * NT);
#pragma unroll
      for (int q = 0; q < FX_U; ++q) {
        fx_deposit<Geo::STR, SECOND>((uint32_t)__double2hiint(v[q].x), (uint32_t)__double2loint(v[q].x), kc, A, B, NT,
                             umax);
        fx_deposit<Geo::STR, SECOND>((uint32_t)__double2hiint(v[q].y), (uint32_t)__double2loint(v[q].y), kc, A, B, NT,
                             umax);
      }
    }
    j0 = 0;
    if (++since == FX_FOLD_CHUNKS) {
      fx_fold<Geo::STR>(A, B, NT);
      since = 0;
    }
    if (threadIdx.x == 0) s_q[slot] = nxt;
    __syncthreads();
    ch = s_q[slot];
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
      fx_deposit<Geo::STR, SECOND>((uint32_t)__double2hiint(v), (uint32_t)__double2loint(v), kc, A, B, NT, umax);
      if (++cnt == 992) {
        fx_fold<Geo::STR>(A, B, NT);
        cnt = 0;
      }
    }
    fx_fold<Geo::STR>(A, B, NT);
  }
  if (!usable) {
    // nothing deposited: the largest exponent field, for the second pass
    const int64_t G_ = (int64_t)gridDim.x * NT;
    for (int64_t i = (int64_t)blockIdx.x * NT + threadIdx.x; i < n; i += G_) {
      const uint32_t eb = ((uint32_t)__double2hiint(__ldcs(x + i)) << 1) >> 21;
      umax = max(umax, (int)eb + (int)kc.Cp);
    }
  }
  const int fail = __syncthreads_or(!usable || umax > u_thr);
  // the largest exponent field deposited, for a second pass
  __shared__ int s_umax;
  if (threadIdx.x == 0) s_umax = INT_MIN / 2;
  __syncthreads();
  const int wmax = __reduce_max_sync(0xffffffffu, umax);
  if ((threadIdx.x & 31) == 0) atomicMax(&s_umax, wmax);

  // 3. Block total into the digit accumulators; the last block converts.
  Tot t = fx_thread_total<Geo::STR, Tot>(A, B, NT);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) t = tot_add(t, tot_shfl_xor(t, m));
  __shared__ Tot s_wt[32];
  if ((threadIdx.x & 31) == 0) s_wt[threadIdx.x >> 5] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    Tot bt = s_wt[0];
    for (int w = 1; w < (int)(NT >> 5); ++w) bt = tot_add(bt, s_wt[w]);
    if (!SECOND && s_umax > INT_MIN / 2) atomicMax(&ctl->emax, (unsigned)max(s_umax - (int)kc.Cp, 0));
    if (fail) {
      atomicOr(&ctl->fail, 1u);
    } else {
#pragma unroll
      for (int i = 0; i < 2 * TotW<Tot>::N; ++i) {
        const uint64_t wd = tot_word(bt, i >> 1);
        atomicAdd(&ctl->dig[i * FX_DIG_STRIDE], (unsigned long long)((i & 1) ? wd >> 32 : wd & 0xFFFFFFFFull));
      }
    }
    __threadfence();
    unsigned tk = atomicAdd(&ctl->ticket, 1u);
    last = (tk == gridDim.x - 1);
  }
  __syncthreads();
  if (!last || threadIdx.x != 0) return;
  __threadfence();
  // sum of the digits D_i 2^(32 i), modulo 2^(64 N) (the total fits); the
  // control words are left zero for the next call
  Tot tot{};
#pragma unroll
  for (int i = 0; i < 2 * TotW<Tot>::N; ++i) {
    Tot d;
    tot_from_shifted(W128{__ldcg(&ctl->dig[i * FX_DIG_STRIDE]), 0}, i, &d);
    ctl->dig[i * FX_DIG_STRIDE] = 0ull;
    tot = tot_add(tot, d);
  }
  ctl->queue = 0u;
  ctl->ticket = 0u;
  if constexpr (SECOND) {
    ctl->run2 = 0u;
  } else {
    const unsigned em = __ldcg(&ctl->emax);
    ctl->emax = 0u;
    if (__ldcg(&ctl->fail)) {
      // Some element lies above the guessed bin, or the guess was not
      // usable.  Every element was deposited, so em is the largest exponent
      // field of the input: the second pass recomputes the sum at its index
      // (no element can lie above that bin), or, when em is all ones, finds
      // which of Inf and NaN occur.
      ctl->fail = 0u;
      if (em >= 0x7FFu) {
        ctl->run2 = 2u;
      } else {
        ctl->I2 = index_of_exponent<double>((int)em, K);
        ctl->run2 = 1u;
      }
      return;
    }
  }
  W128 F[K];
  fx_folds<K>(tot, F);
  *result = convert_fast<double, K>(Ig, 0, F);
}

// ------------------------------------------------------------------ host
namespace {
// the cells: per thread a 64-bit and a 32-bit cell per position and sign
template <int K>
size_t fx_smem_bytes(int block) {
  return (size_t)block * FxGeo<K>::CELLS * 12;
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
    if (cudaFuncSetAttribute(sum_f64_fixed_kernel<K, CNT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(sum_f64_fixed_kernel<K, CNT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
  }
  // the grid is sized for the first pass (the second runs on the same grid)
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, sum_f64_fixed_kernel<K, CNT, false>, block, smem) !=
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

template <int K, int CNT>
cudaError_t launch_kc(const double* x, int64_t n, unsigned* ctl, double* result, int grid, int block, int second,
                      cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = fx_smem_bytes<K>(block);
  cfg.stream = s;
  // the second pass overlaps its launch with the first one's tail
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = second ? 1 : 0;
  if (second) return cudaLaunchKernelEx(&cfg, sum_f64_fixed_kernel<K, CNT, true>, x, n, 1u, (FixedCtl*)ctl, result);
  return cudaLaunchKernelEx(&cfg, sum_f64_fixed_kernel<K, CNT, false>, x, n, 1u, (FixedCtl*)ctl, result);
}

template <int K>
cudaError_t launch_k(const double* x, int64_t n, unsigned* ctl, double* result, int grid, int block, int second,
                     cudaStream_t s) {
  if (block == 128) return launch_kc<K, 128>(x, n, ctl, result, grid, block, second, s);
  if (block == 256) return launch_kc<K, 256>(x, n, ctl, result, grid, block, second, s);
  return launch_kc<K, 0>(x, n, ctl, result, grid, block, second, s);
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

// the control words and digit accumulators, zeroed by the caller
size_t sum_f64_fixed_ctl_bytes() { return sizeof(FixedCtl); }

cudaError_t launch_sum_f64_fixed(const double* x, int64_t n, int K, unsigned* ctl, double* result, int grid, int block,
                                 int second, cudaStream_t s) {
  // make sure the shared-memory attribute is set for this device and block size
  if (sum_f64_fixed_grid(K, block, 1) <= 0) return cudaErrorInvalidConfiguration;
  switch (K) {
    case 2: return launch_k<2>(x, n, ctl, result, grid, block, second, s);
    case 3: return launch_k<3>(x, n, ctl, result, grid, block, second, s);
    case 4: return launch_k<4>(x, n, ctl, result, grid, block, second, s);
    case 5: return launch_k<5>(x, n, ctl, result, grid, block, second, s);
    default: return launch_k<6>(x, n, ctl, result, grid, block, second, s);
  }
}

}  // namespace repro
