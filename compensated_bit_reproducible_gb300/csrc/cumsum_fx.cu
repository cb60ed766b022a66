// Binned cumulative sum of doubles with K = 4, 5 or 6 folds at an index fixed
// before the deposit ("SyclReproSum", "How It Works", cumsum paragraph;
// "Template Parameters": each fold adds W = 40 bits).
//
// Same reading as the K = 3 path (fixed_index.cuh): from the first element
// of the final bin L on (position i*), every prefix has index L and its
// value is the correct rounding of g_f sum_{j <= i} R_j, where R_j is x_j
// rounded once at the finest grid g_f = g_{L+K-1}.  With K folds an
// element's rounded value is below 2^(10 + 40 (K - 1)) grid units (2^240 at
// K = 6), so running totals are 320-bit integers.  Three passes:
//   totals: warps stage 512-element chunks; lane l sums the rounded values
//     of its 16 contiguous elements in 64-bit word cells in shared memory
//     (three cell updates per element); an exclusive warp scan gives the
//     lane prefixes (stored) and the chunk total;
//   scan: exclusive scan of the chunk totals (two levels, last-block ticket),
//     which also decides the path;
//   replay: each lane starts from its prefix, adds each element's rounded
//     value and converts after every element.
// The conversion uses a window fixed for the lane: with |R| <= 2^A for the
// lane's elements and its start below 2^(p0 + 1) in magnitude, every prefix
// of the lane stays below 2^pu (pu = max(p0 + 1, A + 4) + 1), so the lane
// keeps its total pre-shifted by c = 318 - pu bits.  The round-to-odd window
// of a prefix is then the top 64 bits of the shifted total with the bits
// below as one sticky bit, whenever it holds at least 55 bits; one
// cvt.rn.f64.s64 rounds it (see cumsum_k3.cu).  Prefixes below that, and
// lanes whose results leave the normal range, take an exact general
// conversion.
//
// Fallbacks, all with the same bits: a value outside the guessed bin (or
// Inf/NaN, or an index too fine for the shortcuts) makes the general
// per-fold kernels compute everything; if the index settles inside the
// first 4096 elements (i* > 0), the per-fold kernels recompute that tile
// (its prefixes before i* have finer indices); if it settles later, the
// general kernels compute everything.
#include "accum.cuh"
#include "fixed_index.cuh"
#include "launch.h"

namespace repro {
namespace {

using fx::I320;

constexpr int CX_BLOCK = 256;
constexpr int CX_WARPS = CX_BLOCK / 32;
constexpr int CX_CHUNK = 512;                      // elements per warp chunk: lane l owns [16 l, 16 l + 16)
constexpr int CX_PAD = CX_CHUNK + CX_CHUNK / 16;   // staged chunk with one pad element per lane
constexpr int CX_TILE = 4096;                      // first tile: recomputed per fold when 0 < i* < 4096
constexpr int64_t CX_MIN_N = 1 << 17;              // below: the general kernels alone

struct CxCtl {                 // in the stream's control page: zero at the call, and fail,
                               // istar and ticket left zero by the scan; the other words
                               // are written before they are read
  unsigned fail;               // guess failed / Inf, NaN / index too fine
  unsigned general;            // set by the scan: the general kernels compute everything
  int L;                       // the guessed index (written by block 0)
  unsigned tile0;              // set by the scan: the first tile is recomputed per fold
  unsigned long long istar;    // max over elements of bin L of (2^63 - 1 - position), first tile only
  unsigned ticket;             // finished blocks of the scan
};

// Word positions of an element's value M' 2^u (c = u >> 5 <= STR - 3 for a
// valid element); positions 2..STR-1 are kept (below lies under the grid).
template <int K>
struct CxGeo {
  static constexpr int STR = fx::FxGeo<K>::STR;
  static constexpr int NPOS = STR - 2;
};

// ------------------------------------------------------------ 320-bit helpers
__device__ __forceinline__ I320 i320_zero() { return I320{{0, 0, 0, 0, 0}}; }
__device__ __forceinline__ I320 i320_shfl_up(const I320& v, int d) {
  I320 r;
#pragma unroll
  for (int i = 0; i < 5; ++i) r.w[i] = __shfl_up_sync(0xffffffffu, v.w[i], d);
  return r;
}
__device__ __forceinline__ I320 i320_shfl(const I320& v, int src) {
  I320 r;
#pragma unroll
  for (int i = 0; i < 5; ++i) r.w[i] = __shfl_sync(0xffffffffu, v.w[i], src);
  return r;
}
// Exclusive warp scan; *total gets the warp sum.
__device__ __forceinline__ I320 i320_warp_exclusive(const I320& v, I320* total) {
  const int lane = threadIdx.x & 31;
  I320 inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const I320 o = i320_shfl_up(inc, d);
    if (lane >= d) inc = fx::i320_add(inc, o);
  }
  *total = i320_shfl(inc, 31);
  return fx::i320_add(inc, fx::i320_neg(v));
}
// v += d 2^(32 j) for a signed 64-bit d, J a compile-time word offset.
template <int J>
__device__ __forceinline__ void i320_add_word(I320& v, int64_t d) {
  const uint64_t x = (uint64_t)(d >> 63);
  I320 a;
#pragma unroll
  for (int i = 0; i < 5; ++i) a.w[i] = i < J / 2 ? 0 : x;
  if constexpr (J % 2 == 0) {
    a.w[J / 2] = (uint64_t)d;
  } else {
    a.w[J / 2] = (uint64_t)d << 32;
    if constexpr (J / 2 + 1 < 5) a.w[J / 2 + 1] = (uint64_t)(d >> 32);
  }
  v = fx::i320_add(v, a);
}
__device__ __forceinline__ I320 i320_ldcg(const I320* q) {
  I320 r;
#pragma unroll
  for (int i = 0; i < 5; ++i) r.w[i] = __ldcg(&q->w[i]);
  return r;
}

// ------------------------------------------------------------------ totals
// One element's value into the thread's cells (stride CX_BLOCK; cell
// (pos - 2) + NPOS s for word position pos and sign s): w0, w1, w2 at
// positions c, c + 1, c + 2, the words below position 2 zeroed by 0/1
// flags (multiply-adds) and sent to a kept position.
template <int STR>
__device__ __forceinline__ void cx_deposit(uint32_t hi, uint32_t lo, const fx::FxConst& k, uint64_t* A) {
  using namespace fx;
  constexpr uint32_t NPOS = STR - 2;
  const uint32_t eb = mad32(hi, k.one + k.one, 0u) >> 21;   // biased exponent
  const int us = (int)mad32(eb, k.one, k.Cp);               // shift of M
  const uint32_t u = (uint32_t)max(us, 0);
  const uint32_t c = min(u >> 5, (uint32_t)(STR - 3));      // beyond the bin (fails the guess): in bounds
  const uint32_t mh = (hi & 0xFFFFFu) | 0x100000u;
  const uint32_t hl = shl_clamp32(1u, (int)mad32(u, k.negone, k.c63));
  const uint32_t hh = shl_clamp32(1u, (int)mad32(u, k.negone, k.c31));
  const uint32_t b = min(mh & mad32(hl, k.c256, 0u), 1u);   // rounding bit of fold K-2
  const uint64_t Mp = ((((uint64_t)mh) << 32) | lo) + ((((uint64_t)hh) << 32) | hl) - (uint64_t)b;
  const uint32_t lo2 = (uint32_t)Mp, mh2 = (uint32_t)(Mp >> 32);
  const uint32_t w0 = funnel_l(0u, lo2, u);
  const uint32_t w1 = funnel_l(lo2, mh2, u);
  const uint32_t w2 = funnel_l(mh2, 0u, u);
  const uint32_t f2 = mad32(c, k.one, 126u) >> 7;   // c >= 2
  const uint32_t f1 = mad32(c, k.one, 127u) >> 7;   // c >= 1
  // cell of position c + 2 (w2); w1 at c + 1 (or, zeroed, at 2); w0 at c
  // (or, zeroed, at 2 or 3).  k.c7 holds NPOS: the cells per sign.
  const uint32_t base = mad32(hi >> 31, k.c7, c);
  uint64_t* p0 = A + mad32(mad32(f2, 0xFFFFFFFEu, base), (uint32_t)CX_BLOCK, 0u);
  uint64_t* p1 = A + mad32(mad32(f1, 0xFFFFFFFFu, base), (uint32_t)CX_BLOCK, 0u);
  uint64_t* p2 = A + mad32(base, (uint32_t)CX_BLOCK, 0u);
  *p0 = madw(mad32(w0, f2, 0u), k.one, *p0);
  *p1 = madw(mad32(w1, f1, 0u), k.one, *p1);
  *p2 = madw(w2, k.one, *p2);
  (void)NPOS;
}

// The value of the thread's cells since the last call, which are cleared:
// per position the two signs' cells subtract (each sums at most 16 words
// between calls) and the differences combine at their 32-bit offsets.
template <int STR>
__device__ __forceinline__ I320 cx_take(uint64_t* A) {
  constexpr int NPOS = STR - 2;
  int64_t d[NPOS];
#pragma unroll
  for (int j = 0; j < NPOS; ++j) {
    const uint64_t pos = A[j * CX_BLOCK], neg = A[(j + NPOS) * CX_BLOCK];
    A[j * CX_BLOCK] = 0;
    A[(j + NPOS) * CX_BLOCK] = 0;
    d[j] = (int64_t)(pos - neg);
  }
  I320 t = i320_zero();
  i320_add_word<0>(t, d[0]);
  i320_add_word<1>(t, d[1]);
  i320_add_word<2>(t, d[2]);
  i320_add_word<3>(t, d[3]);
  i320_add_word<4>(t, d[4]);
  i320_add_word<5>(t, d[5]);
  if constexpr (NPOS > 6) i320_add_word<6>(t, d[6]);
  if constexpr (NPOS > 7) i320_add_word<7>(t, d[7]);
  return t;
}

// Asks L2 for the warp's next chunk (one 128-byte line per lane) while the
// current one is processed.
__device__ __forceinline__ void cx_prefetch_next(const double* in, int64_t n, int64_t ch_next, int lane) {
  const int64_t i = ch_next * CX_CHUNK + (int64_t)lane * 16;
  if (i < n) asm volatile("prefetch.global.L2 [%0];" ::"l"(in + i));
}

// The lane prefix's top word (bits 256..319 of a value below 2^250 in
// magnitude: copies of the sign) carries the lane's largest exponent field
// in its top 16 bits; the replay takes it from there instead of rereading
// the lane.
__device__ __forceinline__ uint64_t cx_pack(uint64_t w, uint32_t eb) {
  return (w & 0x0000FFFFFFFFFFFFull) | ((uint64_t)eb << 48);
}
__device__ __forceinline__ uint64_t cx_word(uint64_t w) { return (uint64_t)((int64_t)(w << 16) >> 16); }

// Coalesced copy of a chunk (cnt elements at g) into the warp's padded buffer.
__device__ __forceinline__ void cx_stage(double* buf, const double* g, int cnt, int lane) {
  if (cnt == CX_CHUNK && ((((uintptr_t)g) & 15) == 0)) {
    const double2* p = (const double2*)g;
#pragma unroll
    for (int k = 0; k < CX_CHUNK / 2 / 32; ++k) {
      const int i = (k * 32 + lane) * 2;
      const double2 v = __ldcs(p + k * 32 + lane);
      buf[i + i / 16] = v.x;
      buf[i + 1 + (i + 1) / 16] = v.y;
    }
  } else {
    for (int i = lane; i < cnt; i += 32) buf[i + i / 16] = g[i];
  }
}

template <int K>
__host__ __device__ constexpr int cx_cell_bytes() {
  return 2 * CxGeo<K>::NPOS * CX_BLOCK * 8;
}

// Pass 1.  Lane prefixes go to five planes of 64-bit words (one word of each
// lane's 320-bit prefix per plane).
template <int K>
__global__ void __launch_bounds__(CX_BLOCK) cx_totals(const double* __restrict__ in, int64_t n, int64_t nch,
                                                      uint32_t one, CxCtl* ctl, uint64_t* __restrict__ lanep,
                                                      I320* __restrict__ ctot) {
  typedef Geom<double> G;
  constexpr int STR = CxGeo<K>::STR;
  __shared__ double sm[CX_WARPS * CX_PAD];
  __shared__ unsigned s_emax;
  extern __shared__ __align__(16) unsigned char cx_smem[];
  int eb_max;
  const int L = fx::guess_index<double>(in, n, K, &s_emax, &eb_max);
  const int bf = beta<double>(L + K - 1);
  const bool usable = bf >= -1019 && eb_max < 0x7FF;
  if (blockIdx.x == 0 && threadIdx.x == 0) ctl->L = L;
  if (!usable) {
    if (threadIdx.x == 0) atomicOr(&ctl->fail, 1u);
    return;
  }
  const int eb_top = fx::bin_top_exponent<double>(L);
  const int eb_bot = G::BIAS + beta<double>(L + 1) + G::W - 1;   // bottom of bin L
  const fx::FxConst kc = fx::make_const(bf, one, CxGeo<K>::NPOS);   // sign stride: NPOS cells
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ebmax = 0;
  int64_t first = INT64_MAX;
  uint64_t* A = (uint64_t*)cx_smem + threadIdx.x;
#pragma unroll
  for (int k = 0; k < 2 * CxGeo<K>::NPOS; ++k) A[k * CX_BLOCK] = 0;
  const int64_t gw = (int64_t)blockIdx.x * CX_WARPS + warp, GW = (int64_t)gridDim.x * CX_WARPS;
  const size_t plane = (size_t)nch * 32;
  for (int64_t ch = gw; ch < nch; ch += GW) {
    const int64_t c0 = ch * CX_CHUNK;
    const int cnt = (int)min((int64_t)CX_CHUNK, n - c0);
    double* buf = sm + warp * CX_PAD;
    cx_prefetch_next(in, n, ch + GW, lane);
    cx_stage(buf, in + c0, cnt, lane);
    __syncwarp();
    const int b = lane * 16, sb = b + lane;
    uint32_t em = 0;
    // each element deposited as it is read (padding elements are zero)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const double x = b + i < cnt ? buf[sb + i] : 0.0;
      const uint32_t hi = (uint32_t)__double2hiint(x);
      em = max(em, hi << 1);
      cx_deposit<STR>(hi, (uint32_t)__double2loint(x), kc, A);
    }
    ebmax = max(ebmax, (int)(em >> 21));
    if (c0 < CX_TILE) {
#pragma unroll 1
      for (int i = 0; i < 16 && b + i < cnt; ++i) {
        if ((int)(((uint32_t)__double2hiint(buf[sb + i]) << 1) >> 21) >= eb_bot) {
          first = min(first, c0 + b + i);
          break;
        }
      }
    }
    const I320 own = cx_take<STR>(A);
    I320 tot;
    const I320 exc = i320_warp_exclusive(own, &tot);
    const size_t li = (size_t)ch * 32 + lane;
#pragma unroll
    for (int i = 0; i < 4; ++i) lanep[i * plane + li] = exc.w[i];
    lanep[4 * plane + li] = cx_pack(exc.w[4], em >> 21);
    __syncwarp();
    if (lane == 0) ctot[ch] = tot;
  }
  const int bad = __syncthreads_or(ebmax > eb_top);
  int64_t f = first;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) f = min(f, (int64_t)__shfl_xor_sync(0xffffffffu, (long long)f, m));
  if (lane == 0 && f != INT64_MAX) atomicMax(&ctl->istar, 0x7FFFFFFFFFFFFFFFull - (unsigned long long)f);
  if (threadIdx.x == 0 && bad) atomicOr(&ctl->fail, 1u);
}

// Pass 2: exclusive scan of the chunk totals.  Block b scans chunks
// [1024 b, 1024 b + 1024) into lpre (four consecutive chunks per thread);
// the last block to finish scans the block totals into bpre and decides the
// path.  Prefix of chunk c: bpre[c >> 10] + lpre[c].
constexpr int CX_SCAN_THREADS = 256;
__global__ void __launch_bounds__(CX_SCAN_THREADS) cx_scan(const I320* __restrict__ ctot, int64_t nch, CxCtl* ctl,
                                                           I320* __restrict__ lpre, I320* __restrict__ btot,
                                                           I320* __restrict__ bpre) {
  constexpr int NW = CX_SCAN_THREADS / 32;
  __shared__ I320 sm[NW];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c0 = (int64_t)blockIdx.x * 1024 + 4 * threadIdx.x;
  I320 v[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = c0 + j < nch ? ctot[c0 + j] : i320_zero();
  // inclusive prefixes of the thread's four chunks
  const I320 p1 = fx::i320_add(v[0], v[1]), p2 = fx::i320_add(p1, v[2]), p3 = fx::i320_add(p2, v[3]);
  I320 wt;
  I320 exc = i320_warp_exclusive(p3, &wt);
  if (lane == 0) sm[warp] = wt;
  __syncthreads();
  I320 base = i320_zero(), all = i320_zero();
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    if (w < warp) base = fx::i320_add(base, sm[w]);
    all = fx::i320_add(all, sm[w]);
  }
  exc = fx::i320_add(base, exc);
  if (c0 < nch) lpre[c0] = exc;
  if (c0 + 1 < nch) lpre[c0 + 1] = fx::i320_add(exc, v[0]);
  if (c0 + 2 < nch) lpre[c0 + 2] = fx::i320_add(exc, p1);
  if (c0 + 3 < nch) lpre[c0 + 3] = fx::i320_add(exc, p2);
  if (threadIdx.x == 0) {
    btot[blockIdx.x] = all;
    __threadfence();
    last = atomicAdd(&ctl->ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int64_t nb = gridDim.x;
  const int64_t per = (nb + CX_SCAN_THREADS - 1) / CX_SCAN_THREADS;
  const int64_t b0 = (int64_t)threadIdx.x * per, b1 = min(nb, b0 + per);
  I320 agg = i320_zero();
  for (int64_t i = b0; i < b1; ++i) agg = fx::i320_add(agg, i320_ldcg(btot + i));
  const I320 exc2 = i320_warp_exclusive(agg, &wt);
  __syncthreads();
  if (lane == 0) sm[warp] = wt;
  __syncthreads();
  I320 run = i320_zero();
  for (int w = 0; w < warp; ++w) run = fx::i320_add(run, sm[w]);
  run = fx::i320_add(run, exc2);
  for (int64_t i = b0; i < b1; ++i) {
    bpre[i] = run;
    run = fx::i320_add(run, i320_ldcg(btot + i));
  }
  if (threadIdx.x == 0) {
    const unsigned long long code = ctl->istar;
    const int64_t istar = code ? (int64_t)(0x7FFFFFFFFFFFFFFFull - code) : INT64_MAX;
    const bool general = ctl->fail != 0u || istar >= (int64_t)CX_TILE;
    ctl->general = general ? 1u : 0u;
    ctl->tile0 = (!general && istar > 0) ? 1u : 0u;
    // every block has taken its ticket and the totals pass has ended: the
    // accumulated words are left zero for the next call on the stream
    ctl->fail = 0u;
    ctl->istar = 0ull;
    ctl->ticket = 0u;
  }
}

// ------------------------------------------------------------------ replay
// Leading bit position of a signed 320-bit v (of ~v for v < 0): -1 for 0, -1.
__device__ __forceinline__ int i320_lead(const uint32_t* x) {
  const uint32_t s = (uint32_t)((int32_t)x[9] >> 31);
  int p = -1;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t a = x[i] ^ s;
    if (a) p = 32 * i + 31 - __clz((int)a);
  }
  return p;
}

// One lane's replay of its 16 elements (those before cnt), results written
// over the staged inputs.
template <int K>
__device__ __forceinline__ void cx_replay_lane(double* buf, int sb, int b, int cnt, const I320& t,
                                               const fx::FxConst& kc, int bf, uint32_t em) {
  uint32_t x[10];
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    x[2 * i] = (uint32_t)t.w[i];
    x[2 * i + 1] = (uint32_t)(t.w[i] >> 32);
  }
  // lane bound: |R| <= 2^A for its elements (em: their largest exponent field)
  const int A = max((int)em, 1) - 1023 + 1 - bf;
  const int p0 = i320_lead(x);                   // |t| <= 2^(p0 + 1)
  const int pu = max(p0 + 1, A + 4) + 1;          // every prefix of the lane is below 2^pu
  int c = 318 - pu;
  // the window's results lie in 2^(pu - 8 + bf) .. 2^(pu + bf): normal, or the exact path throughout
  const bool win = c >= 0 && pu - 8 + bf >= -1022 && pu + bf <= 1023;
  if (!win) c = 0;
  // shift the start by c (per lane): whole words, then a funnel
  {
    const int ws = c >> 5;
    const uint32_t bs = (uint32_t)(c & 31);
    uint32_t y[10];
#pragma unroll
    for (int i = 0; i < 10; ++i) {
      uint32_t v = 0;
#pragma unroll
      for (int j = 0; j <= i; ++j)
        if (j == ws) v = x[i - j];
      y[i] = v;
    }
#pragma unroll
    for (int i = 0; i < 10; ++i) x[i] = fx::funnel_l(i ? y[i - 1] : 0u, y[i], bs);
  }
  const uint32_t eadd = (uint32_t)(256 - c + bf) << 20;
  const uint32_t cc = (uint32_t)c;
#pragma unroll 2
  for (int i = 0; i < 16; ++i) {
    if (b + i < cnt) {
      const double v = buf[sb + i];
      const uint32_t hi = (uint32_t)__double2hiint(v), lo = (uint32_t)__double2loint(v);
      // the element's rounding at g_f, with the fraction bits of M + h - b cleared
      const uint32_t eb = fx::mad32(hi, kc.one + kc.one, 0u) >> 21;
      const uint32_t u = (uint32_t)max((int)fx::mad32(eb, kc.one, kc.Cp), 0);
      const uint32_t mh = (hi & 0xFFFFFu) | 0x100000u;
      const uint32_t hl = fx::shl_clamp32(1u, (int)fx::mad32(u, kc.negone, kc.c63));
      const uint32_t hh = fx::shl_clamp32(1u, (int)fx::mad32(u, kc.negone, kc.c31));
      const uint32_t rb = min(mh & fx::mad32(hl, kc.c256, 0u), 1u);
      const uint64_t Mp = ((((uint64_t)mh) << 32) | lo) + ((((uint64_t)hh) << 32) | hl) - (uint64_t)rb;
      const int f = 64 - (int)u;   // fraction bits of Mp
      const uint32_t lo2 = (uint32_t)Mp & fx::shl_clamp32(0xFFFFFFFFu, max(f, 0));
      const uint32_t mh2 = (uint32_t)(Mp >> 32) & fx::shl_clamp32(0xFFFFFFFFu, max(f - 32, 0));
      // R 2^c = (Mp' 2^(u + c)) >> 64 through one-hot multipliers (words 2..11 of the product)
      const uint32_t up = fx::mad32(u, kc.one, cc);
      uint32_t r[10];
      uint64_t sp = 0;   // s_{j-1}
      uint64_t spp = 0;  // s_{j-2}
#pragma unroll
      for (int j = 0; j < 12; ++j) {
        const uint32_t q = fx::shl_clamp32(1u, (int)up - 32 * j);
        const uint64_t a = fx::madw(lo2, q, 0);
        const uint64_t sj = fx::madw(mh2, q, a >> 32);
        // product word j = a.lo | s_{j-1}.lo | s_{j-2}.hi; R word j - 2
        if (j >= 2) r[j - 2] = (uint32_t)a | (uint32_t)sp | (uint32_t)(spp >> 32);
        spp = sp;
        sp = sj;
      }
      const uint32_t sm = (uint32_t)((int32_t)hi >> 31);
      // x + (r xor sm) + (sm & 1)
      asm("{\n\t.reg .u32 c;\n\t"
          "add.cc.u32 c, %10, 0xFFFFFFFF;\n\t"
          "addc.cc.u32 %0, %0, %11;\n\t"
          "addc.cc.u32 %1, %1, %12;\n\t"
          "addc.cc.u32 %2, %2, %13;\n\t"
          "addc.cc.u32 %3, %3, %14;\n\t"
          "addc.cc.u32 %4, %4, %15;\n\t"
          "addc.cc.u32 %5, %5, %16;\n\t"
          "addc.cc.u32 %6, %6, %17;\n\t"
          "addc.cc.u32 %7, %7, %18;\n\t"
          "addc.cc.u32 %8, %8, %19;\n\t"
          "addc.u32 %9, %9, %20;\n\t}"
          : "+r"(x[0]), "+r"(x[1]), "+r"(x[2]), "+r"(x[3]), "+r"(x[4]), "+r"(x[5]), "+r"(x[6]), "+r"(x[7]),
            "+r"(x[8]), "+r"(x[9])
          : "r"(sm & 1u), "r"(r[0] ^ sm), "r"(r[1] ^ sm), "r"(r[2] ^ sm), "r"(r[3] ^ sm), "r"(r[4] ^ sm),
            "r"(r[5] ^ sm), "r"(r[6] ^ sm), "r"(r[7] ^ sm), "r"(r[8] ^ sm), "r"(r[9] ^ sm));
      double res;
      if (win && ((x[9] ^ (uint32_t)((int32_t)x[9] >> 31)) >> 22) != 0u) {
        // window: words 9:8, the bits below as a sticky bit
        const uint32_t st = min((x[0] | x[1] | x[2]) | (x[3] | x[4] | x[5]) | (x[6] | x[7]), 1u);
        double d;
        asm("cvt.rn.f64.s64 %0, %1;" : "=d"(d) : "l"((long long)((((uint64_t)x[9]) << 32) | (x[8] | st))));
        res = __hiloint2double((int)((uint32_t)__double2hiint(d) + eadd), __double2loint(d));
      } else {
        // exact conversion: magnitude words, then the limb rounding (the rare path)
        uint32_t mag[10];
        const bool neg = (x[9] >> 31) != 0;
        uint32_t cy = neg ? 1u : 0u;
#pragma unroll
        for (int q = 0; q < 10; ++q) {
          const uint64_t tt = (uint64_t)(neg ? ~x[q] : x[q]) + cy;
          mag[q] = (uint32_t)tt;
          cy = (uint32_t)(tt >> 32);
        }
        res = round_limbs<double>(neg, mag, 10, bf - c);
      }
      buf[sb + i] = res;
    }
  }
}

// Pass 3.  Each warp replays whole chunks staged in shared memory; lane l
// starts from chunk prefix + its lane prefix.  When the first tile is
// recomputed per fold, its chunks are skipped here.
template <int K>
__global__ void __launch_bounds__(CX_BLOCK) cx_replay(const double* in, double* out, int64_t n, int64_t nch,
                                                      uint32_t one, const CxCtl* ctl,
                                                      const uint64_t* __restrict__ lanep,
                                                      const I320* __restrict__ lpre, const I320* __restrict__ bpre) {
  __shared__ double sm[CX_WARPS * CX_PAD];
  if (ctl->general) return;
  const int L = ctl->L;
  const int bf = beta<double>(L + K - 1);
  const fx::FxConst kc = fx::make_const(bf, one, CxGeo<K>::STR);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double* buf = sm + warp * CX_PAD;
  const int64_t gw = (int64_t)blockIdx.x * CX_WARPS + warp, GW = (int64_t)gridDim.x * CX_WARPS;
  const int64_t ch_first = ctl->tile0 ? CX_TILE / CX_CHUNK : 0;
  const size_t plane = (size_t)nch * 32;
  int64_t ch = gw;
  while (ch < ch_first) ch += GW;
  for (; ch < nch; ch += GW) {
    const int64_t c0 = ch * CX_CHUNK;
    const int cnt = (int)min((int64_t)CX_CHUNK, n - c0);
    cx_prefetch_next(in, n, ch + GW, lane);
    cx_stage(buf, in + c0, cnt, lane);
    const size_t li = (size_t)ch * 32 + lane;
    I320 t = fx::i320_add(bpre[ch >> 10], lpre[ch]);
    I320 lp;
#pragma unroll
    for (int i = 0; i < 4; ++i) lp.w[i] = lanep[i * plane + li];
    const uint64_t top = lanep[4 * plane + li];
    lp.w[4] = cx_word(top);
    t = fx::i320_add(t, lp);
    __syncwarp();
    cx_replay_lane<K>(buf, lane * 17, lane * 16, cnt, t, kc, bf, (uint32_t)(top >> 48));
    __syncwarp();
    double* g = out + c0;
    if (cnt == CX_CHUNK && ((((uintptr_t)g) & 15) == 0)) {
#pragma unroll
      for (int k = 0; k < CX_CHUNK / 2 / 32; ++k) {
        const int i = (k * 32 + lane) * 2;
        double2 v;
        v.x = buf[i + i / 16];
        v.y = buf[i + 1 + (i + 1) / 16];
        ((double2*)g)[k * 32 + lane] = v;
      }
    } else {
      for (int i = lane; i < cnt; i += 32) g[i] = buf[i + i / 16];
    }
    __syncwarp();
  }
}

int cx_sm_count() {
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

size_t cx_fast_bytes(int64_t n) {
  const int64_t nc = (n + CX_CHUNK - 1) / CX_CHUNK;
  const int64_t nb = (nc + 1023) / 1024;
  // header, lane prefixes (5 planes), chunk totals and prefixes, block totals and prefixes
  return 256 + (size_t)nc * 32 * 40 + 2 * (size_t)nc * sizeof(I320) + 2 * (size_t)nb * sizeof(I320);
}

template <int K>
cudaError_t launch_fx_k(const double* in, double* out, int64_t n, unsigned char* ws, unsigned char* zc,
                        cudaStream_t s) {
  const size_t gb = (cumsum_general_bytes(n, K) + 255) & ~(size_t)255;
  unsigned char* f = ws + gb;
  CxCtl* ctl = (CxCtl*)zc;
  const int64_t nc = (n + CX_CHUNK - 1) / CX_CHUNK;
  const int64_t ncb = (nc + 1023) / 1024;
  uint64_t* lanep = (uint64_t*)(f + 256);
  I320* ctot = (I320*)(lanep + (size_t)nc * 32 * 5);
  I320* lpre = ctot + nc;
  I320* btot = lpre + nc;
  I320* bpre = btot + ncb;
  cudaError_t e;
  static bool attr_set[64] = {};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if ((e = cudaFuncSetAttribute(cx_totals<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, cx_cell_bytes<K>())) !=
        cudaSuccess)
      return e;
    attr_set[dev] = true;
  }
  int bt = 0, br = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bt, cx_totals<K>, CX_BLOCK, cx_cell_bytes<K>()) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&br, cx_replay<K>, CX_BLOCK, 0) != cudaSuccess) {
    cudaGetLastError();
    bt = br = 1;
  }
  const int64_t sms = cx_sm_count();
  const int64_t wb = (nc + CX_WARPS - 1) / CX_WARPS;   // blocks that have a chunk
  const int64_t gt = max((int64_t)1, min(wb, sms * max(bt, 1))), gr = max((int64_t)1, min(wb, sms * max(br, 1)));
  cx_totals<K><<<(unsigned)gt, CX_BLOCK, cx_cell_bytes<K>(), s>>>(in, n, nc, 1u, ctl, lanep, ctot);
  cx_scan<<<(unsigned)ncb, CX_SCAN_THREADS, 0, s>>>(ctot, nc, ctl, lpre, btot, bpre);
  cx_replay<K><<<(unsigned)gr, CX_BLOCK, 0, s>>>(in, out, n, nc, 1u, ctl, lanep, lpre, bpre);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the first tile per fold when the index settles inside it (reads only its
  // own inputs, which the replay above did not overwrite), then everything
  // when the fast path could not be used; both gated and idle otherwise
  if ((e = launch_cumsum_general<double>(in, out, min(n, (int64_t)CX_TILE), K, ws, s, &ctl->tile0)) != cudaSuccess)
    return e;
  return launch_cumsum_general<double>(in, out, n, K, ws, s, &ctl->general);
}

}  // namespace

size_t cumsum_fx_workspace_bytes(int64_t n, int K) {
  const size_t gb = (cumsum_general_bytes(n, K) + 255) & ~(size_t)255;
  return n >= CX_MIN_N ? gb + cx_fast_bytes(n) : cumsum_general_bytes(n, K);
}

cudaError_t launch_cumsum_fx(const double* in, double* out, int64_t n, int K, unsigned char* ws, unsigned char* zc,
                             cudaStream_t s) {
  if (n < CX_MIN_N) return launch_cumsum_general<double>(in, out, n, K, ws, s, nullptr);
  switch (K) {
    case 4: return launch_fx_k<4>(in, out, n, ws, zc, s);
    case 5: return launch_fx_k<5>(in, out, n, ws, zc, s);
    case 6: return launch_fx_k<6>(in, out, n, ws, zc, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace repro
