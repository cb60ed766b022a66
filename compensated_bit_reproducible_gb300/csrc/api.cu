// C-ABI entry points (declared in include/repro.h).  Argument, capacity and
// overlap checks run before any pointer is touched or memory allocated
// ("SyclReproSum", "Accumulator capacity": the length error comes
// before the pointer is inspected).  Temporary memory comes from the
// stream-ordered allocator on the caller's stream.
#include <cuda_runtime.h>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include "../../include/repro.h"
#include "launch.h"

using namespace repro;

namespace {

thread_local int g_last_cuda = 0;

repro_status cuda_fail(cudaError_t e) {
  g_last_cuda = (int)e;
  return REPRO_ERR_CUDA;
}
#define CK(call)                                  \
  do {                                            \
    cudaError_t _e = (call);                      \
    if (_e != cudaSuccess) return cuda_fail(_e);  \
  } while (0)

// "Accumulator capacity": (2^(p-1) - 1) carries, one per 2^(p-W-2) deposits.
constexpr uint64_t MAX_COUNT_F32 = ((1ull << 23) - 1) << 9;
constexpr uint64_t MAX_COUNT_F64 = ((1ull << 52) - 1) << 11;
constexpr int MAXK_F32 = 21, MAXK_F64 = 52;

template <typename T> struct Lim;
template <> struct Lim<float> {
  static constexpr uint64_t COUNT = MAX_COUNT_F32;
  static constexpr int MAXK = MAXK_F32;
};
template <> struct Lim<double> {
  static constexpr uint64_t COUNT = MAX_COUNT_F64;
  static constexpr int MAXK = MAXK_F64;
};

// Workspace comes from a pool of the library's own per device, which keeps
// up to POOL_KEEP bytes mapped across synchronisations (a pool that returns
// everything at each synchronisation makes the next call map its workspace
// afresh, about 0.2 ms).  The process's default pool is left as it is.
constexpr uint64_t POOL_KEEP = 1ull << 30;

cudaError_t ws_alloc(void** p, size_t bytes, cudaStream_t stream) {
  static cudaMemPool_t pools[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaMallocAsync(p, bytes, stream);
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> g(mu);
    if (!pools[dev]) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t np = nullptr;
      if ((e = cudaMemPoolCreate(&np, &props)) != cudaSuccess) return e;
      uint64_t keep = POOL_KEEP;
      if ((e = cudaMemPoolSetAttribute(np, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
        cudaMemPoolDestroy(np);
        return e;
      }
      pools[dev] = np;
    }
    pool = pools[dev];
  }
  return cudaMallocFromPoolAsync(p, bytes, pool, stream);
}

// Control words per device and stream: a page that every kernel using it
// leaves zero when it ends (the sums' tickets, chunk queue, digit
// accumulators and fallback flag).  Calls on one stream run in order, so
// each finds the page zero and none needs a memset; calls on different
// streams use different pages.  Pages live as long as the process (one per
// stream ever used).  A stream that is destroyed while its calls are still
// pending and whose handle is reused at once by a new stream would share
// the page with them.
constexpr size_t CTL_PAGE_BYTES = 4096;
constexpr size_t CTL_SUM_TICKET = 0;      // general sum kernel's ticket
constexpr size_t CTL_SUM_FIXED = 256;     // double fixed-index sum's control words
constexpr size_t CTL_CUMSUM = 2048;       // cumulative sums' control words (256 bytes)

cudaError_t ctl_page(cudaStream_t stream, unsigned char** out) {
  static std::mutex mu;
  static std::map<std::pair<int, cudaStream_t>, unsigned char*> pages;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(mu);
  auto it = pages.find({dev, stream});
  if (it != pages.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  void* p = nullptr;
  if ((e = cudaMalloc(&p, CTL_PAGE_BYTES)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p, 0, CTL_PAGE_BYTES, stream)) != cudaSuccess) {
    cudaFree(p);
    return e;
  }
  pages[{dev, stream}] = (unsigned char*)p;
  *out = (unsigned char*)p;
  return cudaSuccess;
}

// At most this many elements, a sum runs in one block (no workspace, no
// grid merge): below it the grid path's fixed steps cost more than the
// block's longer pass.
constexpr uint64_t SMALL_SUM_MAX = 16384;

// Per host thread, one pinned and mapped slot that the synchronous sum's
// kernel writes its result to (no device allocation and no copy per call).
struct PinnedSlot {
  void* p = nullptr;
  ~PinnedSlot() {
    if (p) cudaFreeHost(p);
  }
};
thread_local PinnedSlot g_slot;

void* result_slot() {
  if (!g_slot.p) {
    if (cudaHostAlloc(&g_slot.p, 64, cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess) {
      cudaGetLastError();
      g_slot.p = nullptr;
    }
  }
  return g_slot.p;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (!cached[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = v > 0 ? v : 152;
  }
  return cached[dev];
}

// ------------------------------------------------------------ environment
std::mutex g_env_mu;
int g_env_state[64] = {0};   // 0 unknown, 1 ok, 2 failed

repro_status validate_env(cudaStream_t stream) {
  if (env_fail_forced()) return REPRO_ERR_ENV;
  int dev = 0;
  CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return REPRO_ERR_ENV;
  {
    std::lock_guard<std::mutex> g(g_env_mu);
    if (g_env_state[dev] == 1) return REPRO_OK;
    if (g_env_state[dev] == 2) return REPRO_ERR_ENV;
  }
  unsigned* d = nullptr;
  CK(ws_alloc((void**)&d, sizeof(unsigned), stream));
  unsigned h = 0xFFFFFFFFu;
  cudaError_t e = launch_env_probe(d, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, d, sizeof(unsigned), cudaMemcpyDeviceToHost, stream);
  cudaError_t e2 = cudaFreeAsync(d, stream);
  if (e == cudaSuccess) e = e2;
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  std::lock_guard<std::mutex> g(g_env_mu);
  g_env_state[dev] = (h == 0) ? 1 : 2;
  return h == 0 ? REPRO_OK : REPRO_ERR_ENV;
}

// ------------------------------------------------------------- pointers
bool is_host_only(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return true;
  }
  return a.type == cudaMemoryTypeUnregistered;
}

template <typename T> bool aligned(const T* p) { return ((uintptr_t)p % sizeof(T)) == 0; }

struct Scratch {
  void* p = nullptr;
  cudaStream_t s = nullptr;
  ~Scratch() {
    if (p) cudaFreeAsync(p, s);
  }
};

// Sizes for which the double sum takes the sampled fixed-index path: below,
// launch latency dominates anyway; above, its 64-bit thread cells could
// overflow (and no device holds that many doubles).
constexpr size_t FIXED_MIN_N = 1u << 16;
constexpr uint64_t FIXED_MAX_N = 1ull << 36;

template <typename T>
repro_status check_sum_args(const T* x, size_t n, int K) {
  if (K < 2 || K > Lim<T>::MAXK) return REPRO_ERR_INVALID_ARG;
  if ((uint64_t)n > Lim<T>::COUNT) return REPRO_ERR_CAPACITY;
  if (n > 0 && (x == nullptr || !aligned(x))) return REPRO_ERR_INVALID_ARG;
  return REPRO_OK;
}

bool launch_ok(const repro_launch* l) {
  if (!l) return true;
  if (l->block != 0 && (l->block < 32 || l->block > 1024 || (l->block % 32) != 0)) return false;
  if (l->grid < 0) return false;
  return true;
}

// Grid for the binned sum: enough blocks to fill the GPU, no more than the
// work needs, and few enough elements per thread that int64 lanes cannot
// overflow (<= 2^23 deposits per thread).
int sum_grid(int64_t n, int block, int elems_per_iter, int blocks_per_sm, const repro_launch* l) {
  if (l && l->grid > 0) {
    int64_t g = l->grid;
    int64_t need = (n + ((int64_t)block << 23) - 1) / ((int64_t)block << 23);
    return (int)(g > need ? g : need);
  }
  int64_t work = (n + (int64_t)block * elems_per_iter - 1) / ((int64_t)block * elems_per_iter);
  int64_t cap = (int64_t)sm_count() * blocks_per_sm;
  int64_t g = work < cap ? work : cap;
  if (g < 1) g = 1;
  return (int)g;
}

template <typename T>
repro_status sum_async_impl(const T* x, size_t n, int K, cudaStream_t stream, T* result_dev,
                            const repro_launch* l) {
  repro_status st = check_sum_args(x, n, K);
  if (st != REPRO_OK) return st;
  if (!result_dev || !aligned(result_dev) || !launch_ok(l)) return REPRO_ERR_INVALID_ARG;
  st = validate_env(stream);
  if (st != REPRO_OK) return st;
  // float: 512 threads per block (two blocks per SM) measured best on the
  // 1e8-element sum; double keeps 256 for the general kernel
  int block = (l && l->block) ? l->block : (sizeof(T) == 4 ? 512 : 256);
  if ((uint64_t)n <= SMALL_SUM_MAX && !(l && l->grid > 0)) {
    // one block, no workspace
    CK(launch_sum_single<T>(x, (int64_t)n, K, result_dev, block, stream));
    return REPRO_OK;
  }
  int grid = sum_grid((int64_t)n, block, 4 * (int)(16 / sizeof(T)), sum_blocks_per_sm<T>(K, block),
                      l);   // 4 vectors per thread per iteration, one wave of blocks
  // double with K = 2..6: the sampled fixed-index kernel runs first and the
  // general kernel only if that one flags its guess
  int fgrid = 0, fblock = 0;
  if constexpr (sizeof(T) == 8) {
    if (K >= 2 && K <= 6 && n >= FIXED_MIN_N && (uint64_t)n <= FIXED_MAX_N) {
      fblock = (l && l->block) ? l->block : 128;
      // zero when the cells do not fit this block size (K = 6 at 1024
      // threads): the general kernel alone runs
      const int fcap = sum_f64_fixed_grid(K, fblock, sm_count());
      fgrid = fcap <= 0 ? 0 : ((l && l->grid > 0) ? l->grid : fcap);
      if (CTL_SUM_FIXED + sum_f64_fixed_ctl_bytes() > CTL_PAGE_BYTES) fgrid = 0;
    }
  }
  // tickets and control words in the stream's page (zero between calls)
  unsigned char* page = nullptr;
  CK(ctl_page(stream, &page));
  if constexpr (sizeof(T) == 8) {
    if (fgrid > 0) {
      // first pass at the sampled index, then the second pass: idle unless
      // the first one missed (an element above the guessed bin, an index too
      // fine for its shortcut, Inf or NaN); then it recomputes the sum at the
      // index of the largest exponent, or finds which specials occur
      unsigned* ctl = (unsigned*)(page + CTL_SUM_FIXED);
      CK(launch_sum_f64_fixed((const double*)x, (int64_t)n, K, ctl, (double*)result_dev, fgrid, fblock, 0, stream));
      CK(launch_sum_f64_fixed((const double*)x, (int64_t)n, K, ctl, (double*)result_dev, fgrid, fblock, 1, stream));
      return REPRO_OK;
    }
  }
  // the general one-pass kernel; its partials in a workspace
  unsigned* ticket = (unsigned*)(page + CTL_SUM_TICKET);
  Scratch ws;
  ws.s = stream;
  CK(ws_alloc(&ws.p, sum_workspace_bytes(K, grid), stream));
  CK(launch_sum<T>(x, (int64_t)n, K, ticket, (unsigned char*)ws.p, result_dev, grid, block, stream));
  return REPRO_OK;
}

template <typename T>
repro_status sum_sync_impl(const T* x, size_t n, int K, cudaStream_t stream, T* result) {
  repro_status st = check_sum_args(x, n, K);
  if (st != REPRO_OK) return st;
  if (!result) return REPRO_ERR_INVALID_ARG;
  if (n == 0) {
    *result = (T)0;
    return REPRO_OK;
  }
  st = validate_env(stream);
  if (st != REPRO_OK) return st;
  // plain host memory is copied to the device first
  Scratch in;
  in.s = stream;
  const T* xd = x;
  if (is_host_only(x)) {
    CK(ws_alloc(&in.p, n * sizeof(T), stream));
    CK(cudaMemcpyAsync(in.p, x, n * sizeof(T), cudaMemcpyHostToDevice, stream));
    xd = (const T*)in.p;
  }
  // the result goes to this thread's pinned slot (mapped, so the kernel
  // writes it directly); without one, to device memory and back
  T* slot = (T*)result_slot();
  if (slot) {
    st = sum_async_impl<T>(xd, n, K, stream, slot, nullptr);
    if (st != REPRO_OK) return st;
    CK(cudaStreamSynchronize(stream));
    *result = *(volatile T*)slot;
    return REPRO_OK;
  }
  Scratch r;
  r.s = stream;
  CK(ws_alloc(&r.p, 16, stream));
  st = sum_async_impl<T>(xd, n, K, stream, (T*)r.p, nullptr);
  if (st != REPRO_OK) return st;
  T h;
  CK(cudaMemcpyAsync(&h, r.p, sizeof(T), cudaMemcpyDeviceToHost, stream));
  CK(cudaStreamSynchronize(stream));
  *result = h;
  return REPRO_OK;
}

template <typename T>
repro_status cumsum_impl(const T* in, T* out, size_t n, int K, cudaStream_t stream, const repro_launch* l) {
  if (K < 2 || K > Lim<T>::MAXK) return REPRO_ERR_INVALID_ARG;
  if ((uint64_t)n > Lim<T>::COUNT) return REPRO_ERR_CAPACITY;
  if (n == 0) return REPRO_OK;
  if (!in || !out || !aligned(in) || !aligned(out) || !launch_ok(l)) return REPRO_ERR_INVALID_ARG;
  uintptr_t a0 = (uintptr_t)in, a1 = a0 + n * sizeof(T), b0 = (uintptr_t)out, b1 = b0 + n * sizeof(T);
  if (in != out && a0 < b1 && b0 < a1) return REPRO_ERR_OVERLAP;
  repro_status st = validate_env(stream);
  if (st != REPRO_OK) return st;
  // plain host memory ("Pointer type handling"): the input is copied to
  // temporary device memory, the output computed there and copied back, and
  // the call waits for it; device, managed and pinned pointers are used as
  // they are
  const bool hin = is_host_only(in), hout = is_host_only(out);
  Scratch tin, tout;
  tin.s = tout.s = stream;
  const T* din = in;
  T* dout = out;
  if (hin) {
    CK(ws_alloc(&tin.p, n * sizeof(T), stream));
    CK(cudaMemcpyAsync(tin.p, in, n * sizeof(T), cudaMemcpyHostToDevice, stream));
    din = (const T*)tin.p;
  }
  if (hout) {
    if (in == out) {
      dout = (T*)tin.p;   // in place on the copy
    } else {
      CK(ws_alloc(&tout.p, n * sizeof(T), stream));
      dout = (T*)tout.p;
    }
  }
  Scratch ws;
  ws.s = stream;
  const size_t wsb = cumsum_workspace_bytes<T>((int64_t)n, K);
  if (wsb) CK(ws_alloc(&ws.p, wsb, stream));   // none for a single tile
  unsigned char* page = nullptr;
  CK(ctl_page(stream, &page));
  CK(launch_cumsum<T>(din, dout, (int64_t)n, K, (unsigned char*)ws.p, page + CTL_CUMSUM, stream));
  if (hout) {
    CK(cudaMemcpyAsync(out, dout, n * sizeof(T), cudaMemcpyDeviceToHost, stream));
    CK(cudaStreamSynchronize(stream));
  }
  return REPRO_OK;
}

// Cumulative sum that starts from a binned state: every prefix includes the
// state's value ("How It Works": states merge exactly, so a chunked or
// sharded input scans as one).  Device-accessible pointers only.
template <typename T>
repro_status cumsum_from_state_impl(const T* in, T* out, size_t n, int K, const void* state, cudaStream_t stream) {
  if (K < 2 || K > Lim<T>::MAXK) return REPRO_ERR_INVALID_ARG;
  if ((uint64_t)n > Lim<T>::COUNT) return REPRO_ERR_CAPACITY;
  if (!state || ((uintptr_t)state & 15u)) return REPRO_ERR_INVALID_ARG;   // states are 16-byte aligned
  if (n == 0) return REPRO_OK;
  if (!in || !out || !aligned(in) || !aligned(out)) return REPRO_ERR_INVALID_ARG;
  uintptr_t a0 = (uintptr_t)in, a1 = a0 + n * sizeof(T), b0 = (uintptr_t)out, b1 = b0 + n * sizeof(T);
  if (in != out && a0 < b1 && b0 < a1) return REPRO_ERR_OVERLAP;
  repro_status st = validate_env(stream);
  if (st != REPRO_OK) return st;
  if (is_host_only(in) || is_host_only(out) || is_host_only(state)) return REPRO_ERR_INVALID_ARG;
  Scratch ws;
  ws.s = stream;
  const size_t wsb = cumsum_carry_workspace_bytes<T>((int64_t)n, K);
  if (wsb) CK(ws_alloc(&ws.p, wsb, stream));
  unsigned char* page = nullptr;
  CK(ctl_page(stream, &page));
  CK(launch_cumsum<T>(in, out, (int64_t)n, K, (unsigned char*)ws.p, page + CTL_CUMSUM, stream,
                      (const unsigned char*)state));
  return REPRO_OK;
}

// Shape checks shared by the variance calls; n must be exact in the element
// type (2^24 for float32, 2^53 for float64).
repro_status var_shape_ok(int64_t rows, int64_t cols, int axis, int ddof, int64_t nmax) {
  if (axis != 0 && axis != 1) return REPRO_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0) return REPRO_ERR_INVALID_ARG;
  int64_t n = axis == 1 ? cols : rows;
  if (ddof < 0 || ddof >= n) return REPRO_ERR_INVALID_ARG;
  if (n > nmax) return REPRO_ERR_INVALID_ARG;
  return REPRO_OK;
}

repro_status var_impl(const float* x, int64_t rows, int64_t cols, int axis, int ddof, float* out, float* mean,
                      int variant, cudaStream_t stream) {
  repro_status st = var_shape_ok(rows, cols, axis, ddof, 1ll << 24);
  if (st != REPRO_OK) return st;
  if (variant < 0 || variant > 6) return REPRO_ERR_INVALID_ARG;
  if (!x || !out || !aligned(x) || !aligned(out) || (mean && !aligned(mean))) return REPRO_ERR_INVALID_ARG;
  st = validate_env(stream);
  if (st != REPRO_OK) return st;
  CK(launch_var(x, rows, cols, axis, ddof, out, mean, variant, nullptr, stream));
  return REPRO_OK;
}

repro_status var_f64_impl(const double* x, int64_t rows, int64_t cols, int axis, int ddof, double* out,
                          double* mean, cudaStream_t stream) {
  repro_status st = var_shape_ok(rows, cols, axis, ddof, 1ll << 53);
  if (st != REPRO_OK) return st;
  if (!x || !out || !aligned(x) || !aligned(out) || (mean && !aligned(mean))) return REPRO_ERR_INVALID_ARG;
  st = validate_env(stream);
  if (st != REPRO_OK) return st;
  CK(launch_var_f64(x, rows, cols, axis, ddof, out, mean, stream));
  return REPRO_OK;
}

repro_status var_c64_impl(const float* z, int64_t rows, int64_t cols, int axis, int ddof, float* out, float* mean,
                          cudaStream_t stream) {
  repro_status st = var_shape_ok(rows, cols, axis, ddof, 1ll << 24);
  if (st != REPRO_OK) return st;
  // complex64: 8-byte pairs
  if (!z || !out || ((uintptr_t)z & 7u) || !aligned(out) || (mean && ((uintptr_t)mean & 7u)))
    return REPRO_ERR_INVALID_ARG;
  st = validate_env(stream);
  if (st != REPRO_OK) return st;
  CK(launch_var_c64(z, rows, cols, axis, ddof, out, mean, stream));
  return REPRO_OK;
}

template <typename T>
repro_status compare_impl(const T* x, size_t n, int mode, T* result, cudaStream_t stream) {
  if ((n > 0 && (!x || !aligned(x))) || !result || !aligned(result)) return REPRO_ERR_INVALID_ARG;
  if (n > (1ull << 40)) return REPRO_ERR_CAPACITY;
  repro_status st = validate_env(stream);
  if (st != REPRO_OK) return st;
  Scratch ws;
  ws.s = stream;
  CK(ws_alloc(&ws.p, compare_workspace_bytes<T>((int64_t)n, mode), stream));
  if (mode == 0) CK(cudaMemsetAsync(ws.p, 0, 256, stream));
  CK(launch_compare<T>(x, (int64_t)n, mode, result, (unsigned char*)ws.p, stream));
  return REPRO_OK;
}

}  // namespace

// ------------------------------------------------------------ binned states
constexpr size_t STATE_HDR = 32;

bool state_ptr_ok(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

template <typename T>
repro_status state_init_impl(void* state, int K, cudaStream_t stream) {
  if (K < 2 || K > Lim<T>::MAXK || !state_ptr_ok(state)) return REPRO_ERR_INVALID_ARG;
  repro_status st = validate_env(stream);
  if (st != REPRO_OK) return st;
  CK(launch_state_op<T>(0, (unsigned char*)state, nullptr, K, 0, nullptr, stream));
  return REPRO_OK;
}

template <typename T>
repro_status state_deposit_impl(void* state, const T* x, size_t n, int K, cudaStream_t stream) {
  repro_status st = check_sum_args(x, n, K);
  if (st != REPRO_OK) return st;
  if (!state_ptr_ok(state)) return REPRO_ERR_INVALID_ARG;
  if (n == 0) return REPRO_OK;
  st = validate_env(stream);
  if (st != REPRO_OK) return st;
  const int block = 256;
  if ((uint64_t)n <= SMALL_SUM_MAX) {
    CK(launch_sum_single<T>(x, (int64_t)n, K, nullptr, block, stream, (unsigned char*)state));
    return REPRO_OK;
  }
  const int grid = sum_grid((int64_t)n, block, 4 * (int)(16 / sizeof(T)), sum_blocks_per_sm<T>(K, block), nullptr);
  Scratch ws;
  ws.s = stream;
  CK(ws_alloc(&ws.p, sum_workspace_bytes(K, grid), stream));
  CK(cudaMemsetAsync(ws.p, 0, 256, stream));
  CK(launch_state_deposit<T>(x, (int64_t)n, K, (unsigned char*)ws.p, (unsigned char*)state, grid, block, stream));
  return REPRO_OK;
}

template <typename T>
repro_status state_merge_impl(void* dst, const void* src, int K, cudaStream_t stream) {
  if (K < 2 || K > Lim<T>::MAXK || !state_ptr_ok(dst) || !state_ptr_ok(src)) return REPRO_ERR_INVALID_ARG;
  repro_status st = validate_env(stream);
  if (st != REPRO_OK) return st;
  CK(launch_state_op<T>(1, (unsigned char*)dst, (const unsigned char*)src, K, 0, nullptr, stream));
  return REPRO_OK;
}

template <typename T>
repro_status state_finalize_impl(const void* state, int K, T* result_dev, cudaStream_t stream) {
  if (K < 2 || K > Lim<T>::MAXK || !state_ptr_ok(state) || !result_dev || !aligned(result_dev))
    return REPRO_ERR_INVALID_ARG;
  repro_status st = validate_env(stream);
  if (st != REPRO_OK) return st;
  CK(launch_state_op<T>(2, nullptr, (const unsigned char*)state, K, Lim<T>::COUNT, result_dev, stream));
  return REPRO_OK;
}

extern "C" {

const char* repro_strerror(repro_status s) {
  switch (s) {
    case REPRO_OK: return "ok";
    case REPRO_ERR_INVALID_ARG: return "invalid argument";
    case REPRO_ERR_CAPACITY: return "input count exceeds the reproducible capacity";
    case REPRO_ERR_OVERLAP: return "input and output overlap (only exact in-place is allowed)";
    case REPRO_ERR_ENV: return "device floating-point environment failed validation";
    case REPRO_ERR_CUDA: return "CUDA runtime error";
    case REPRO_ERR_DEVICE_TIMEOUT: return "device-side wait exceeded its bound";
  }
  return "unknown status";
}

int repro_last_cuda_error(void) { return g_last_cuda; }

uint64_t repro_max_count_f32(void) { return MAX_COUNT_F32; }
uint64_t repro_max_count_f64(void) { return MAX_COUNT_F64; }
int repro_max_k_f32(void) { return MAXK_F32; }
int repro_max_k_f64(void) { return MAXK_F64; }

repro_status repro_validate_environment(cudaStream_t stream) { return validate_env(stream); }

repro_status repro_sum_f32(const float* x, size_t n, int K, cudaStream_t s, float* r) {
  return sum_sync_impl<float>(x, n, K, s, r);
}
repro_status repro_sum_f64(const double* x, size_t n, int K, cudaStream_t s, double* r) {
  return sum_sync_impl<double>(x, n, K, s, r);
}
repro_status repro_sum_f32_async(const float* x, size_t n, int K, cudaStream_t s, float* r,
                                 const repro_launch* l) {
  return sum_async_impl<float>(x, n, K, s, r, l);
}
repro_status repro_sum_f64_async(const double* x, size_t n, int K, cudaStream_t s, double* r,
                                 const repro_launch* l) {
  return sum_async_impl<double>(x, n, K, s, r, l);
}

repro_status repro_cumsum_f32(const float* in, float* out, size_t n, int K, cudaStream_t s) {
  return cumsum_impl<float>(in, out, n, K, s, nullptr);
}
repro_status repro_cumsum_f64(const double* in, double* out, size_t n, int K, cudaStream_t s) {
  return cumsum_impl<double>(in, out, n, K, s, nullptr);
}
repro_status repro_cumsum_f32_ex(const float* in, float* out, size_t n, int K, cudaStream_t s,
                                 const repro_launch* l) {
  return cumsum_impl<float>(in, out, n, K, s, l);
}
repro_status repro_cumsum_f64_ex(const double* in, double* out, size_t n, int K, cudaStream_t s,
                                 const repro_launch* l) {
  return cumsum_impl<double>(in, out, n, K, s, l);
}

repro_status repro_segsum_f32(const float* x, int64_t rows, int64_t cols, int axis, int K, float* out,
                              cudaStream_t s) {
  if (axis != 0 && axis != 1) return REPRO_ERR_INVALID_ARG;
  if (K < 2 || K > MAXK_F32 || rows <= 0 || cols <= 0) return REPRO_ERR_INVALID_ARG;
  if ((uint64_t)(axis == 1 ? cols : rows) > MAX_COUNT_F32) return REPRO_ERR_CAPACITY;
  if (!x || !out || !aligned(x) || !aligned(out)) return REPRO_ERR_INVALID_ARG;
  repro_status st = validate_env(s);
  if (st != REPRO_OK) return st;
  int64_t grid = rows < 65535 * 16 ? rows : 65535 * 16;
  CK(launch_segsum(x, rows, cols, axis, K, out, (int)grid, 256, s));
  return REPRO_OK;
}

repro_status stable_var_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof, float* out,
                            float* mean_out, cudaStream_t s) {
  return var_impl(x, rows, cols, axis, ddof, out, mean_out, 0, s);
}
repro_status twoterm_var_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof, float* out,
                             cudaStream_t s) {
  return var_impl(x, rows, cols, axis, ddof, out, nullptr, 1, s);
}
repro_status stable_var_f32_variant(const float* x, int64_t rows, int64_t cols, int axis, int ddof, int variant,
                                    float* out, float* mean_out, cudaStream_t s) {
  return var_impl(x, rows, cols, axis, ddof, out, mean_out, variant, s);
}
repro_status stable_var_f64(const double* x, int64_t rows, int64_t cols, int axis, int ddof, double* out,
                            double* mean_out, cudaStream_t s) {
  return var_f64_impl(x, rows, cols, axis, ddof, out, mean_out, s);
}
repro_status stable_var_c64(const float* z, int64_t rows, int64_t cols, int axis, int ddof, float* out,
                            float* mean_out, cudaStream_t s) {
  return var_c64_impl(z, rows, cols, axis, ddof, out, mean_out, s);
}

repro_status repro_sum_naive_f32(const float* x, size_t n, float* r, cudaStream_t s) {
  return compare_impl<float>(x, n, 0, r, s);
}
repro_status repro_sum_naive_f64(const double* x, size_t n, double* r, cudaStream_t s) {
  return compare_impl<double>(x, n, 0, r, s);
}
repro_status repro_sum_pairwise_f32(const float* x, size_t n, float* r, cudaStream_t s) {
  return compare_impl<float>(x, n, 1, r, s);
}
repro_status repro_sum_pairwise_f64(const double* x, size_t n, double* r, cudaStream_t s) {
  return compare_impl<double>(x, n, 1, r, s);
}
repro_status repro_sum_kahan_f32(const float* x, size_t n, float* r, cudaStream_t s) {
  return compare_impl<float>(x, n, 2, r, s);
}
repro_status repro_sum_kahan_f64(const double* x, size_t n, double* r, cudaStream_t s) {
  return compare_impl<double>(x, n, 2, r, s);
}
repro_status repro_sum_neumaier_f32(const float* x, size_t n, float* r, cudaStream_t s) {
  return compare_impl<float>(x, n, 3, r, s);
}
repro_status repro_sum_neumaier_f64(const double* x, size_t n, double* r, cudaStream_t s) {
  return compare_impl<double>(x, n, 3, r, s);
}
int repro_compensated_chunk(void) { return COMPENSATED_CHUNK; }

size_t repro_state_bytes(int K) {
  if (K < 2 || K > MAXK_F64) return 0;
  return STATE_HDR + 16 * (size_t)K;
}
repro_status repro_state_init_f32(void* state, int K, cudaStream_t s) { return state_init_impl<float>(state, K, s); }
repro_status repro_state_init_f64(void* state, int K, cudaStream_t s) { return state_init_impl<double>(state, K, s); }
repro_status repro_state_deposit_f32(void* state, const float* x, size_t n, int K, cudaStream_t s) {
  return state_deposit_impl<float>(state, x, n, K, s);
}
repro_status repro_state_deposit_f64(void* state, const double* x, size_t n, int K, cudaStream_t s) {
  return state_deposit_impl<double>(state, x, n, K, s);
}
repro_status repro_state_merge_f32(void* dst, const void* src, int K, cudaStream_t s) {
  return state_merge_impl<float>(dst, src, K, s);
}
repro_status repro_state_merge_f64(void* dst, const void* src, int K, cudaStream_t s) {
  return state_merge_impl<double>(dst, src, K, s);
}
repro_status repro_state_finalize_f32(const void* state, int K, float* result_dev, cudaStream_t s) {
  return state_finalize_impl<float>(state, K, result_dev, s);
}
repro_status repro_state_finalize_f64(const void* state, int K, double* result_dev, cudaStream_t s) {
  return state_finalize_impl<double>(state, K, result_dev, s);
}
repro_status repro_cumsum_from_state_f32(const float* in, float* out, size_t n, int K, const void* state,
                                         cudaStream_t s) {
  return cumsum_from_state_impl<float>(in, out, n, K, state, s);
}
repro_status repro_cumsum_from_state_f64(const double* in, double* out, size_t n, int K, const void* state,
                                         cudaStream_t s) {
  return cumsum_from_state_impl<double>(in, out, n, K, state, s);
}

}  // extern "C"

namespace repro {
void set_last_cuda(cudaError_t e) { g_last_cuda = (int)e; }
bool env_fail_forced() {
  const char* force = std::getenv("REPRO_FORCE_ENV_FAIL");
  return force && force[0] == '1';
}
}  // namespace repro
