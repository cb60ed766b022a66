// Binned float sum that allocates nothing (declared in include/repro.h as
// repro_sum_f32_noalloc).
//
// Some callers cannot call cudaMalloc: their device memory is entirely held
// by another allocator (a framework's caching pool that reserved the GPU), or
// they run in a phase where an allocation must not happen because it can
// synchronize the device or fail under memory pressure.  This entry point
// runs the same binned sum kernel as repro_sum_f32_async, but its workspace
// (the grid ticket and the per-block partial states) lives in one file-scope
// device array of fixed size, so no call allocates device or host memory.
//
// Limits and sharing:
//  - the array holds NOALLOC_SCRATCH_BYTES (256 KiB); the grid is sized to fit
//    it, which covers every n up to the float capacity (4,294,966,784) and
//    every K from 2 to 21;
//  - every GPU that loads the library holds the array until the process exits;
//  - all calls on a device share the array and it keeps the last call's
//    contents: each call clears the part that must start at zero (the grid
//    ticket), and calls whose work overlaps on the GPU race on it, so callers
//    must order them (one stream, or events between streams);
//  - the first call on a device does the set-up (the array's device address
//    and the floating-point environment probe) and waits for it; make that
//    first call before any stream capture;
//  - the device address is kept for the life of the process: after a
//    cudaDeviceReset the array belongs to a context that no longer exists,
//    and the entry point must not be called again in that process;
//  - CUDA errors are reported like every other entry point's: status
//    REPRO_ERR_CUDA, code in repro_last_cuda_error().
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>
#include "../../include/repro.h"
#include "launch.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 256 * 1024;
constexpr int NOALLOC_MAX_DEVICES = 64;

// The workspace.  Host code must not use this name as an address: in host
// code it is a stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

struct DevInfo {
  bool ready = false;
  bool env_ok = false;
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
  int sms = 0;
};

std::mutex g_mu;
DevInfo g_dev[NOALLOC_MAX_DEVICES];

// Once per device, with that device current: the array's device address, the
// SM count and the environment probe (its one result word is written into the
// array itself, so nothing is allocated).
repro_status setup(int dev, cudaStream_t stream, DevInfo** out) {
  std::lock_guard<std::mutex> g(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      repro::set_last_cuda(e);
      return REPRO_ERR_CUDA;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      repro::set_last_cuda(e);
      return REPRO_ERR_CUDA;
    }
    unsigned probe = 0xFFFFFFFFu;
    e = repro::launch_env_probe((unsigned*)p, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&probe, p, sizeof(unsigned), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
      repro::set_last_cuda(e);
      return REPRO_ERR_CUDA;
    }
    d.scratch = (unsigned char*)p;
    d.sms = sms > 0 ? sms : 1;
    d.env_ok = (probe == 0);
    d.ready = true;
  }
  *out = &d;
  return REPRO_OK;
}

}  // namespace

extern "C" repro_status repro_sum_f32_noalloc(const float* x, size_t n, int K, cudaStream_t stream,
                                              float* result_dev) {
  if (K < 2 || K > 21) return REPRO_ERR_INVALID_ARG;
  if ((uint64_t)n > 4294966784ull) return REPRO_ERR_CAPACITY;
  if ((n > 0 && (x == nullptr || ((uintptr_t)x & 3))) || result_dev == nullptr || ((uintptr_t)result_dev & 3))
    return REPRO_ERR_INVALID_ARG;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    repro::set_last_cuda(e);
    return REPRO_ERR_CUDA;
  }
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return REPRO_ERR_INVALID_ARG;
  if (repro::env_fail_forced()) return REPRO_ERR_ENV;
  DevInfo* d = nullptr;
  repro_status st = setup(dev, stream, &d);
  if (st != REPRO_OK) return st;
  if (!d->env_ok) return REPRO_ERR_ENV;
  // Grid: fill the GPU (8 blocks of 256 per SM), no more blocks than the work
  // needs, and no more than the array holds.
  const int block = 256;
  const size_t stride = 16 + 16 * (size_t)K;
  int64_t work = ((int64_t)n + (int64_t)block * 16 - 1) / ((int64_t)block * 16);
  int64_t grid = (int64_t)d->sms * 8;
  if (work < grid) grid = work;
  int64_t fit = (int64_t)((NOALLOC_SCRATCH_BYTES - 256 - 64) / stride);
  if (grid > fit) grid = fit;
  if (grid < 1) grid = 1;
  // int64 lanes hold at most 2^23 deposits per thread
  if ((int64_t)n > grid * block * (int64_t)(1 << 23)) return REPRO_ERR_CAPACITY;
  if (256 + (size_t)grid * stride + 64 > NOALLOC_SCRATCH_BYTES) return REPRO_ERR_CAPACITY;
  // the grid ticket must start at zero
  e = cudaMemsetAsync(d->scratch, 0, 256, stream);
  if (e == cudaSuccess)
    e = repro::launch_sum<float>(x, (int64_t)n, K, (unsigned*)d->scratch, d->scratch + 256, result_dev, (int)grid,
                                 block, stream);
  if (e != cudaSuccess) {
    repro::set_last_cuda(e);
    return REPRO_ERR_CUDA;
  }
  return REPRO_OK;
}
