// Internal launchers (host side), called by the C-ABI layer.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace repro {

// binned sum.  ticket: a zero counter (zero again after the call); parts:
// one partial state of 16 + 16 K bytes per block (sum_workspace_bytes(K,
// grid) bytes suffice).
template <typename T>
cudaError_t launch_sum(const T* x, int64_t n, int K, unsigned* ticket, unsigned char* parts, T* result, int grid,
                       int block, cudaStream_t s);
// One block, no workspace: the single-block sum for small inputs.
template <typename T>
cudaError_t launch_sum_single(const T* x, int64_t n, int K, T* result, int block, cudaStream_t s,
                              unsigned char* state = nullptr);

// Binned states (32-byte header + K 128-bit folds in device memory).
// Deposit: the grid sum of x merged into *state (workspace as for
// launch_sum).  op 0: init dst; 1: merge src into dst; 2: finalize src to
// *result (canonical NaN past `capacity` elements or on a K/type mismatch).
template <typename T>
cudaError_t launch_state_deposit(const T* x, int64_t n, int K, unsigned char* ws, unsigned char* state, int grid,
                                 int block, cudaStream_t s);
template <typename T>
cudaError_t launch_state_op(int op, unsigned char* dst, const unsigned char* src, int K, uint64_t capacity,
                            T* result, cudaStream_t s);
size_t sum_workspace_bytes(int K, int grid);
template <typename T>
int sum_blocks_per_sm(int K, int block);
// double sum at a fixed index (K = 2..6): blocks per GPU for this block
// size (0: not available), size of the control words, launch.  The first
// pass (second = 0) guesses the index from a sample; launched right after
// it, the second pass (second = 1) runs only when an element lay above the
// guessed bin (or the first pass could not be used), at the index of the
// largest exponent, or to find which of Inf and NaN occur.  ctl points at
// sum_f64_fixed_ctl_bytes() zero bytes (16-byte aligned), which the two
// leave zero.
int sum_f64_fixed_grid(int K, int block, int sms);
size_t sum_f64_fixed_ctl_bytes();
cudaError_t launch_sum_f64_fixed(const double* x, int64_t n, int K, unsigned* ctl, double* result, int grid,
                                 int block, int second, cudaStream_t s);
cudaError_t launch_segsum(const float* x, int64_t rows, int64_t cols, int axis, int K, float* out, int grid,
                          int block, cudaStream_t s);

// binned cumulative sum
template <typename T>
size_t cumsum_workspace_bytes(int64_t n, int K);
// zc: 256 bytes of control words, zero at the call and left zero (the
// stream's control page).  carry: null, or a device binned state
// (repro_state layout) that every prefix includes; such calls take the
// general per-fold kernels.
template <typename T>
cudaError_t launch_cumsum(const T* in, T* out, int64_t n, int K, unsigned char* ws, unsigned char* zc, cudaStream_t s,
                          const unsigned char* carry = nullptr);
// The general per-fold kernels for K = 4..6 on doubles, optionally gated (see
// adn_cumsum.cu), and their workspace.
template <typename T>
cudaError_t launch_cumsum_general(const T* in, T* out, int64_t n, int K, unsigned char* ws, cudaStream_t s,
                                  const unsigned* gate);
size_t cumsum_general_bytes(int64_t n, int K);
// Doubles with K = 4..6 (cumsum_fx.cu): the fixed-index path for long inputs,
// the general kernels otherwise.
size_t cumsum_fx_workspace_bytes(int64_t n, int K);
cudaError_t launch_cumsum_fx(const double* in, double* out, int64_t n, int K, unsigned char* ws, unsigned char* zc,
                             cudaStream_t s);
template <typename T>
size_t cumsum_k3_workspace_bytes(int64_t n);
template <typename T>
size_t cumsum_k3_general_bytes(int64_t n);
template <typename T>
size_t cumsum_carry_workspace_bytes(int64_t n, int K);
template <typename T>
cudaError_t launch_cumsum_k3(const T* in, T* out, int64_t n, unsigned char* ws, unsigned char* zc, cudaStream_t s,
                             const unsigned char* carry = nullptr);

// variance
cudaError_t launch_var(const float* x, int64_t rows, int64_t cols, int axis, int ddof, float* out, float* mean,
                       int variant, unsigned char* ws, cudaStream_t s);
// The kernel on float64 input (every step in float64).
cudaError_t launch_var_f64(const double* x, int64_t rows, int64_t cols, int axis, int ddof, double* out,
                           double* mean, cudaStream_t s);
// Complex64 input (interleaved re, im): var(re) + var(im) per slice; mean
// interleaved.
cudaError_t launch_var_c64(const float* z, int64_t rows, int64_t cols, int axis, int ddof, float* out,
                           float* mean, cudaStream_t s);
size_t var_workspace_bytes(int64_t rows, int64_t cols, int axis);

// comparison sums: mode 0 naive, 1 pairwise, 2 kahan, 3 neumaier
template <typename T>
cudaError_t launch_compare(const T* x, int64_t n, int mode, T* result, unsigned char* ws, cudaStream_t s);
template <typename T>
size_t compare_workspace_bytes(int64_t n, int mode);
constexpr int COMPENSATED_CHUNK = 4096;

// environment probe: writes check bits to *out (device), 0 = all passed
cudaError_t launch_env_probe(unsigned* out, cudaStream_t s);
// true when REPRO_FORCE_ENV_FAIL=1 asks every environment check to fail
bool env_fail_forced();

// The calling host thread's last CUDA error, the one repro_last_cuda_error()
// returns; every entry point that returns REPRO_ERR_CUDA records its code here.
void set_last_cuda(cudaError_t e);

}  // namespace repro
