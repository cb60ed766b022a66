/*
 * Oracle for order-independent floating-point summation: a plain, slow,
 * single-threaded CPU restatement of what the GPU path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library: every constant below is
 * restated from the pages it cites.
 *
 * Sources (by page title and section):
 *  - "SyclReproSum": "How It Works" (deposit / renormalize / merge,
 *    Inf/NaN rules, absorption threshold), "Accumulator capacity",
 *    "Template Parameters" (bin width W, max K, error term), "Quick Start".
 *  - "Variance in float32 with a first-element shift, a local centring and a
 *    compensated tree sum": section 1 (formula of reference), section 2 (the
 *    four steps), section 3 (identical-value table).
 *  - "Reduction order and compensation solve related but different problems":
 *    sequential, pairwise, Kahan and Neumaier sums.
 *  - "Kahan's Summation Formula": the Kahan loop and its printed results.
 *
 * Parity status of every function is stated at its definition; functions
 * with no pin to the pages or to mathematics say "parity unpinned".
 */
#ifndef REPRO_ORACLE_H
#define REPRO_ORACLE_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_MAXK 52

/* ---- exact sums (superaccumulator) ---------------------------------- */
/* Exact sum of finite inputs, rounded once to nearest-even. Returns 0 on
   success, 1 if an input is Inf/NaN (the result is then not written). */
int orc_exact_sum_f64(const double* x, int64_t n, double* out);
int orc_exact_sum_f32(const float* x, int64_t n, float* out);
/* Exact sum exported as a two's-complement limb array: value =
   sum_i limb[i] * 2^(64 i + *lsb).  Returns the number of limbs written. */
int orc_exact_sum_limbs_f64(const double* x, int64_t n, uint64_t* limbs, int max_limbs, int* lsb);
int orc_exact_sum_limbs_f32(const float* x, int64_t n, uint64_t* limbs, int max_limbs, int* lsb);

/* ---- ADN binned sum --------------------------------------------------- */
uint64_t orc_max_count_f32(void);
uint64_t orc_max_count_f64(void);
int orc_max_k_f32(void);
int orc_max_k_f64(void);
int orc_bin_width_f32(void);
int orc_bin_width_f64(void);
/* Bin index of one finite non-zero value (0 = coarsest). */
int orc_bin_index_f64(double x);
int orc_bin_index_f32(float x);

/* Closed form: index from max|x|, chained round-half-away pieces per value,
   exact per-fold integer sums, one correct rounding. */
double orc_adn_sum_closed_f64(const double* x, int64_t n, int K);
float  orc_adn_sum_closed_f32(const float* x, int64_t n, int K);
/* Same, also exporting the state: *I, fold sums F[k] (units of the fold's
   grid) as (hi, lo) 64-bit halves of a 128-bit two's-complement integer, and
   special-value flags (bit0 NaN, bit1 +Inf, bit2 -Inf). */
void orc_adn_state_closed_f64(const double* x, int64_t n, int K, int* I,
                              int64_t* F_hi, uint64_t* F_lo, int* flags);
void orc_adn_state_closed_f32(const float* x, int64_t n, int K, int* I,
                              int64_t* F_hi, uint64_t* F_lo, int* flags);
/* Sequential floating-point form: primaries, sticky-bit deposit,
   renormalisation into carries, one-pass index raise. */
double orc_adn_sum_fp_f64(const double* x, int64_t n, int K);
float  orc_adn_sum_fp_f32(const float* x, int64_t n, int K);
/* Cumulative sums: out[i] = ADN sum of x[0..i]. */
void orc_adn_cumsum_f64(const double* x, double* out, int64_t n, int K);
void orc_adn_cumsum_f32(const float* x, float* out, int64_t n, int K);
/* Cumulative sums evaluated only at sorted positions pos[0..m) (one pass). */
void orc_adn_cumsum_at_f64(const double* x, int64_t n, int K, const int64_t* pos, int64_t m, double* out);
void orc_adn_cumsum_at_f32(const float* x, int64_t n, int K, const int64_t* pos, int64_t m, float* out);

/* ---- comparison modes ------------------------------------------------- */
double orc_sum_naive_f64(const double* x, int64_t n);
float  orc_sum_naive_f32(const float* x, int64_t n);
double orc_sum_pairwise_f64(const double* x, int64_t n);
float  orc_sum_pairwise_f32(const float* x, int64_t n);
double orc_sum_kahan_f64(const double* x, int64_t n);
float  orc_sum_kahan_f32(const float* x, int64_t n);
double orc_sum_neumaier_f64(const double* x, int64_t n);
float  orc_sum_neumaier_f32(const float* x, int64_t n);
/* Chunked compensated sums: compensated sum of each `chunk`-element run in
   order, chunk results combined by the pairwise tree. */
double orc_sum_kahan_chunked_f64(const double* x, int64_t n, int64_t chunk);
float  orc_sum_kahan_chunked_f32(const float* x, int64_t n, int64_t chunk);
double orc_sum_neumaier_chunked_f64(const double* x, int64_t n, int64_t chunk);
float  orc_sum_neumaier_chunked_f32(const float* x, int64_t n, int64_t chunk);

/* ---- variance ----------------------------------------------------------- */
/* x is row-major [rows, cols]; axis 1 reduces along a row, axis 0 along a
   column.  Outputs have one entry per slice. mean_out may be NULL. */
void orc_var_kernel_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof,
                        float* var_out, float* mean_out);
void orc_var_twoterm_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof,
                         float* var_out);
void orc_var_naive_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof,
                       float* var_out);
void orc_var_f64(const float* x, int64_t rows, int64_t cols, int axis, int ddof,
                 double* var_out, double* mean_out);
/* Per-slice ADN sum (segmented), same layout conventions. */
void orc_segsum_f32(const float* x, int64_t rows, int64_t cols, int axis, int K, float* out);
/* Complex variance: var(re) + var(im), each by the float32 kernel. */
void orc_var_kernel_c64(const float* re, const float* im, int64_t n, int ddof, float* var_out);
/* The same per slice of a complex64 [rows, cols] array (interleaved re, im);
   mean_out (interleaved, may be NULL) gets (mean(re), mean(im)). */
void orc_var_kernel_c64_2d(const float* z, int64_t rows, int64_t cols, int axis, int ddof,
                           float* var_out, float* mean_out);
/* Section 4 variants of the float32 kernel ("Which step does what"):
     0 the kernel: shift + centring, TwoSum tree, two-term;
     2 shift + centring, plain tree, no two-term (var = s2/n);
     3 shift + centring, plain tree, two-term;
     4 no shift: the formula of reference (means as the tree sum times
       RN(1/n), d = x - mean, two-term) with the TwoSum tree for d^2 (the
       reading that matches its row: at most equal to the reference on 4/4
       datasets, NaN for [1e38]*3 on the GPU); mean = the reference's mean;
     5 shift + centring, TwoSum tree, no two-term;
     6 shift + centring, s2 by Kahan's sequential loop over d^2 in index
       order, two-term (only step 3 changes: "one step changed at a time").
   Variant 1 is the formula of reference (orc_var_twoterm_f32, with its
   mean).  Pins: exact
   variance on small-integer data; the [1e38]*3 column of section 4 (0 with
   the shift, NaN for variant 4); identical values give 0 with the shift;
   float64 closeness; variant 0 equals orc_var_kernel_f32 bit for bit. */
void orc_var_variant_f32(const float* x, int64_t rows, int64_t cols, int axis, int ddof, int variant,
                         float* var_out, float* mean_out);
/* The kernel on float64 input, every step in float64.  Pins: exact
   variance on small-integer data, identical values (including [1e307]*3)
   give 0, closeness to the exact rational variance. */
void orc_var_kernel_f64(const double* x, int64_t rows, int64_t cols, int axis, int ddof,
                        double* var_out, double* mean_out);
/* TwoSum of the compensated tree (section 2, step 3): *s = RN(a + b) and
   *e the exact rounding error, so that *s + *e = a + b.  Pins: the exact
   identity on random pairs of every exponent spread, and the tree's s2
   equal to the correctly rounded sum of the squared residuals on slices
   where the carries are exact and the plain tree rounds. */
void orc_two_sum_f32(float a, float b, float* s, float* e);
void orc_two_sum_f64(double a, double b, double* s, double* e);

#ifdef __cplusplus
}
#endif
#endif
