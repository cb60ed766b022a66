/*
 * repro: order-independent floating-point summation on one NVIDIA GB300.
 *
 * C ABI of librepro_gb300.so.  Every call takes plain pointers and sizes and a
 * CUDA stream; no C++ or framework types cross this boundary.
 *
 * Conventions shared by all calls
 *  - Pointers: inputs and outputs are caller-owned device pointers (also
 *    managed memory, or host memory as stated per call); the library never
 *    frees them.  Floating-point pointers must be aligned to their element
 *    size.  Temporary device memory is taken, stream-ordered on `stream`,
 *    from a memory pool the library creates per device (it keeps up to
 *    1 GiB mapped between calls; the process's default pool is not
 *    touched) and returned before the call's work completes on that stream.
 *    Small inputs need none: a sum of at most 16384 elements runs in one
 *    block, a K = 3 cumulative sum of at most 4096 in one tile.
 *  - Streams: work is enqueued on `stream` (0 = legacy default stream).
 *    Calls documented "synchronous" wait for their own work; the others
 *    return once the work is enqueued.
 *  - Control words: the sums and cumulative sums count and accumulate in a
 *    4 KiB page of device memory per device and stream, allocated and
 *    zeroed at a stream's first call, which every call leaves zero again
 *    (so no call needs a memset).  Calls on one stream therefore run one
 *    after another on it; calls on different streams use different pages.
 *    Pages are kept until the process exits.  A CUDA graph captured from a
 *    stream keeps that stream's page: its launches must not overlap one
 *    another or calls made directly on that stream, and the stream's first
 *    call must come before the capture (the page is allocated then).
 *  - Device reset: the library keeps per-device state (its memory pool,
 *    the control pages, cached device properties).  After cudaDeviceReset
 *    the library's calls must not be used again in that process.
 *  - Errors: a non-zero repro_status.  Argument and capacity checks happen
 *    before any pointer is touched or any memory allocated; an error leaves
 *    outputs unwritten.  repro_strerror() gives a static message.
 *  - Reproducibility: for the binned (ADN) calls the result bits depend only
 *    on the input values (for sums: on the multiset; for cumulative sums: on
 *    the sequence), never on launch configuration, scheduling or stream.
 *
 * Sources: "SyclReproSum" (sections "How It Works", "API Reference",
 * "Accumulator capacity", "Template Parameters", "Runtime environment
 * validation"); "Variance in float32 with a first-element shift, a local
 * centring and a compensated tree sum" (section 2); "Reduction order and
 * compensation solve related but different problems" and "Kahan's Summation
 * Formula" (comparison sums).
 */
#ifndef REPRO_GB300_H
#define REPRO_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cudaStream_t;

typedef enum {
  REPRO_OK = 0,
  REPRO_ERR_INVALID_ARG = 1,      /* null pointer with n > 0, K out of range, bad axis/ddof/shape, misaligned */
  REPRO_ERR_CAPACITY = 2,         /* n above the reproducible capacity */
  REPRO_ERR_OVERLAP = 3,          /* cumulative sum with partially overlapping input/output */
  REPRO_ERR_ENV = 4,              /* device floating-point environment failed validation */
  REPRO_ERR_CUDA = 5,             /* a CUDA runtime call failed (see repro_last_cuda_error) */
  REPRO_ERR_DEVICE_TIMEOUT = 6    /* a device-side wait exceeded its bound */
} repro_status;

/* Optional launch shape for the *_ex calls (0 fields = library default).
   Only the speed changes with it, never the result bits. */
typedef struct {
  int block;   /* threads per block: a multiple of 32 in [32, 1024] */
  int grid;    /* blocks; 0 = sized from n and the SM count */
} repro_launch;

/* Static description of a status code. */
const char* repro_strerror(repro_status s);
/* Last CUDA error code seen by this host thread (cudaError_t value). */
int repro_last_cuda_error(void);

/* ---- constants ("Accumulator capacity", "Template Parameters") ---------- */
/* Largest n for which results are reproducible: 4,294,966,784 (float) and
   9,223,372,036,854,773,760 (double). */
uint64_t repro_max_count_f32(void);
uint64_t repro_max_count_f64(void);
/* Largest fold count K: 21 (float), 52 (double); the smallest is 2. */
int repro_max_k_f32(void);
int repro_max_k_f64(void);

/* ---- environment ("Runtime environment validation") --------------------- */
/* Runs a probe kernel on the current device checking IEEE binary32/64
   layouts, round-to-nearest-even, unflushed subnormals, signed zero and
   Inf/NaN arithmetic.  The result is cached per device; every compute call
   of this library calls it on first use.  Synchronous.  REPRO_ERR_ENV when a
   check fails.  With the environment variable REPRO_FORCE_ENV_FAIL=1 every
   validation fails with REPRO_ERR_ENV before any device work (a test hook
   for the failure path). */
repro_status repro_validate_environment(cudaStream_t stream);

/* ---- binned sums ("How It Works": deposit, renormalize, merge) ---------- */
/* Reproducible sum of x[0..n) with K folds (2 <= K <= max K).  x may be a
   device, managed, pinned-host or plain host pointer (host data is copied to
   the device first).  Synchronous; *result is a host pointer.  n == 0 gives
   +0.0.  Any NaN, or both +Inf and -Inf, gives the canonical quiet NaN
   (0x7fc00000 / 0x7ff8000000000000); otherwise an Inf propagates; an exact
   zero is +0.0.  Result = correct rounding of the exact binned value.  The
   kernel writes the result to a pinned, mapped host slot owned by the
   calling host thread (allocated on its first call), so a call on device
   data makes no device allocation or copy for it. */
repro_status repro_sum_f32(const float* x, size_t n, int K, cudaStream_t stream, float* result);
repro_status repro_sum_f64(const double* x, size_t n, int K, cudaStream_t stream, double* result);
/* Same sum, stream-ordered: x is device-accessible, *result_dev is a device
   pointer written when the work completes; nothing waits on the host. */
repro_status repro_sum_f32_async(const float* x, size_t n, int K, cudaStream_t stream, float* result_dev,
                                 const repro_launch* launch);
repro_status repro_sum_f64_async(const double* x, size_t n, int K, cudaStream_t stream, double* result_dev,
                                 const repro_launch* launch);

/* Same binned float sum for callers that cannot allocate device memory (the
   pages have no counterpart to this call).  Some callers cannot call
   cudaMalloc: another allocator already holds the GPU's memory, or the call
   sits where an allocation could synchronize the device or fail.  The
   workspace is one file-scope device array of 256 KiB inside the library,
   held by every GPU that loads it until the process exits; nothing is
   allocated per call.  x is device-accessible, *result_dev a device pointer;
   stream-ordered.  Limits: K in 2..21, n up to the float capacity
   (4,294,966,784), else REPRO_ERR_INVALID_ARG / REPRO_ERR_CAPACITY.  All calls
   share the array (each clears what must start at zero): calls whose work
   overlaps on the GPU race, so order them on one stream or with events.  The
   first call on a device sets up (device address of the array, environment
   probe) and waits for it; make it before any stream capture.  The address
   is kept until the process exits: after cudaDeviceReset do not call this
   entry point again in that process.  A failed CUDA call gives
   REPRO_ERR_CUDA with its code in repro_last_cuda_error(); the environment
   check honours REPRO_FORCE_ENV_FAIL like every other (REPRO_ERR_ENV). */
repro_status repro_sum_f32_noalloc(const float* x, size_t n, int K, cudaStream_t stream, float* result_dev);

/* ---- binned states ("How It Works": deposit and merge; "API Reference":
   chunked sums) ------------------------------------------------------------ */
/* A binned state holds everything deposited into it as {bin index, K exact
   fold sums, Inf/NaN flags, element count}.  It lives in caller-owned device
   memory of repro_state_bytes(K) bytes, 16-byte aligned; the layout is a
   32-byte header (int32 index, int32 flags, int32 K, int32 type 1 = float /
   2 = double, uint64 count, 8 zero bytes) followed by K fold sums, each a
   little-endian 128-bit integer (low 64 bits first), in units of their
   fold's grid.  Depositing chunks and merging states in any split and any
   order, then finalizing, gives the same bits as repro_sum of the whole
   input: the merge aligns both states to the coarser index and adds the
   folds exactly.  States can be copied between devices and merged there
   (the layout has no pointers).  Calls that touch one state must be ordered
   (one stream, or events).  All calls are stream-ordered and use the
   same K and element type as the state's init; a different K or type, or
   more than the capacity (repro_max_count_*) elements in total, makes
   finalize give the canonical NaN.  Errors: REPRO_ERR_INVALID_ARG for K out
   of range, a null or misaligned state / result / input pointer;
   REPRO_ERR_CAPACITY for one deposit above the capacity. */
size_t repro_state_bytes(int K);   /* 32 + 16 K; 0 for K outside 2..52 */
repro_status repro_state_init_f32(void* state, int K, cudaStream_t stream);
repro_status repro_state_init_f64(void* state, int K, cudaStream_t stream);
/* state += binned x[0..n) (x device-accessible; n == 0 does nothing). */
repro_status repro_state_deposit_f32(void* state, const float* x, size_t n, int K, cudaStream_t stream);
repro_status repro_state_deposit_f64(void* state, const double* x, size_t n, int K, cudaStream_t stream);
/* dst += src (dst == src doubles the state). */
repro_status repro_state_merge_f32(void* dst, const void* src, int K, cudaStream_t stream);
repro_status repro_state_merge_f64(void* dst, const void* src, int K, cudaStream_t stream);
/* *result_dev (device pointer) = correctly rounded value of the state, the
   same special-value and signed-zero rules as repro_sum. */
repro_status repro_state_finalize_f32(const void* state, int K, float* result_dev, cudaStream_t stream);
repro_status repro_state_finalize_f64(const void* state, int K, double* result_dev, cudaStream_t stream);

/* Cumulative sum that continues from a binned state ("How It Works": the
   cumulative-sum scan carries binned prefixes; states merge exactly):
   out[i] = binned sum of (everything deposited into *state) and in[0..i],
   with the index of that combined prefix, so a shard's cumulative sum that
   starts from the merged states of all earlier shards equals the
   corresponding outputs of one cumulative sum over the whole input.  state is
   a repro_state of the same K and type (another K or type gives the
   canonical NaN in every output; no fold of it is read); it is only read.
   in, out and state are device-accessible (device, managed or pinned) memory;
   in == out is allowed, other overlaps give REPRO_ERR_OVERLAP.  Stream-ordered.
   These calls run the general per-fold kernels (not the fixed-index paths).
   Errors: as repro_cumsum, and REPRO_ERR_INVALID_ARG for a null or
   misaligned state or for plain host memory. */
repro_status repro_cumsum_from_state_f32(const float* in, float* out, size_t n, int K, const void* state,
                                         cudaStream_t stream);
repro_status repro_cumsum_from_state_f64(const double* in, double* out, size_t n, int K, const void* state,
                                         cudaStream_t stream);

/* ---- binned cumulative sums ("How It Works", cumsum paragraph; "API
   Reference": cumsum) ------------------------------------------------------ */
/* out[i] = reproducible sum of in[0..i] (each prefix with its own bin
   index, so out[n-1] equals repro_sum of the whole input).  in == out (exact
   in place) is allowed; any other overlap gives REPRO_ERR_OVERLAP.  Device,
   managed or pinned host pointers are used as they are and the call is
   stream-ordered (returns once enqueued).  Plain host memory ("Pointer type
   handling"): a host input is copied to temporary device memory, a host
   output is computed there and copied back, and the call then returns only
   when out holds the result.  The *_ex forms check the launch shape (an
   invalid one gives REPRO_ERR_INVALID_ARG) but the cumulative sums run
   their own block sizes. */
repro_status repro_cumsum_f32(const float* in, float* out, size_t n, int K, cudaStream_t stream);
repro_status repro_cumsum_f64(const double* in, double* out, size_t n, int K, cudaStream_t stream);
repro_status repro_cumsum_f32_ex(const float* in, float* out, size_t n, int K, cudaStream_t stream,
                                 const repro_launch* launch);
repro_status repro_cumsum_f64_ex(const double* in, double* out, size_t n, int K, cudaStream_t stream,
                                 const repro_launch* launch);

/* ---- segmented binned sums --------------------------------------------- */
/* One reproducible sum per slice of a row-major [rows, cols] float array:
   axis 1 sums each row (out has rows entries), axis 0 each column (cols
   entries).  Device pointers; stream-ordered. */
repro_status repro_segsum_f32(const float* x, int64_t rows, int64_t cols, int axis, int K, float* out,
                              cudaStream_t stream);

/* ---- float32 variance ("Variance in float32 with a first-element shift, a
   local centring and a compensated tree sum", section 2) ------------------ */
/* Per-slice variance of a row-major [rows, cols] float array along `axis`
   (1: each row, 0: each column), entirely in float32:
     y = x - x[0];  m = sum(y) / n;  d = y - m;
     s2 = compensated TwoSum tree over d*d (errors carried up a second array,
          result = final sum + final carry);  s1 = tree sum of d;
     var = max(s2/n - (s1/n)^2, 0) * n / (n - ddof);  mean = x[0] + m.
   Trees pair adjacent nodes (2i, 2i+1) level by level; an unpaired last node
   passes up unchanged.  0 <= ddof < n.  out gets one variance per slice;
   mean_out (nullable) the means.  Device pointers; stream-ordered. */
repro_status stable_var_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof, float* out,
                            float* mean_out, cudaStream_t stream);
/* The same kernel on float64 input, every step in float64 (variance page,
   section 2: "all in the input dtype"; section 5 lists float64 as not
   measured).  n <= 2^53; otherwise as stable_var_f32. */
repro_status stable_var_f64(const double* x, int64_t rows, int64_t cols, int axis, int ddof, double* out,
                            double* mean_out, cudaStream_t stream);
/* Complex64 input (section 2, last paragraph): z is a row-major [rows, cols]
   complex64 array (interleaved real, imaginary float32 pairs, 8-byte
   aligned).  Per slice, out = RN(var(re) + var(im)) with each part by the
   float32 kernel (ddof applied to each part), i.e. E|z - mean(z)|^2;
   mean_out (nullable, complex64, 8-byte aligned) gets (mean(re), mean(im)).
   Otherwise as stable_var_f32. */
repro_status stable_var_c64(const float* z, int64_t rows, int64_t cols, int axis, int ddof, float* out,
                            float* mean_out, cudaStream_t stream);
/* The kernel with steps changed, as in the variance page's section 4
   ("Which step does what"); variant:
     0  the kernel (= stable_var_f32);
     1  the formula of reference (= twoterm_var_f32; mean_out gets mean(x));
     2  shift + centring, plain tree for d^2, no two-term: var = s2/n;
     3  shift + centring, plain tree for d^2, two-term;
     4  no shift: the formula of reference with the TwoSum tree for d^2
        (var = max(RN(s2 RN(1/n)) - md^2, 0)); mean_out gets mean(x);
     5  shift + centring, TwoSum tree, no two-term;
     6  shift + centring, s2 by Kahan's sequential loop over d^2 in index
        order (one thread per slice: slow by design), two-term.
   Every tree and rounding step is the kernel's; the result is bit-identical
   to the oracle's restatement of each variant.  variant outside 0..6 gives
   REPRO_ERR_INVALID_ARG. */
repro_status stable_var_f32_variant(const float* x, int64_t rows, int64_t cols, int axis, int ddof, int variant,
                                    float* out, float* mean_out, cudaStream_t stream);

/* ---- comparison modes ("Reduction order and compensation solve related but
   different problems"; "Kahan's Summation Formula") ---------------------- */
/* Formula of reference for the variance (tf.nn.moments; variance page,
   section 1): m = mean(x); d = x - m; var = max(mean(d^2) - mean(d)^2, 0),
   mean(v) = RN(tree_sum(v) * RN(1/n)), same ddof rescale.  Stream-ordered. */
repro_status twoterm_var_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof, float* out,
                             cudaStream_t stream);
/* Non-reproducible comparison sums, result to a device pointer,
   stream-ordered:
   naive     - plain parallel float/double reduction (order depends on the
               launch shape: the usual non-reproducible baseline);
   pairwise  - the adjacent-pair tree over x[0..n) (deterministic for a given
               n);
   kahan     - Kahan's loop (y = x - c; t = s + y; c = (t - s) - y; s = t) over
               consecutive 4096-element chunks, chunk sums combined by the
               pairwise tree;
   neumaier  - Neumaier's loop over the same chunks (result s + c per chunk),
               combined by the pairwise tree. */
repro_status repro_sum_naive_f32(const float* x, size_t n, float* result_dev, cudaStream_t stream);
repro_status repro_sum_naive_f64(const double* x, size_t n, double* result_dev, cudaStream_t stream);
repro_status repro_sum_pairwise_f32(const float* x, size_t n, float* result_dev, cudaStream_t stream);
repro_status repro_sum_pairwise_f64(const double* x, size_t n, double* result_dev, cudaStream_t stream);
repro_status repro_sum_kahan_f32(const float* x, size_t n, float* result_dev, cudaStream_t stream);
repro_status repro_sum_kahan_f64(const double* x, size_t n, double* result_dev, cudaStream_t stream);
repro_status repro_sum_neumaier_f32(const float* x, size_t n, float* result_dev, cudaStream_t stream);
repro_status repro_sum_neumaier_f64(const double* x, size_t n, double* result_dev, cudaStream_t stream);
/* Chunk length used by the chunked Kahan / Neumaier comparison sums. */
int repro_compensated_chunk(void);

#ifdef __cplusplus
}
#endif
#endif /* REPRO_GB300_H */
