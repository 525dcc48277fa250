/*
 * dspark_markov_check.h -- checking aids of libdspark_markov.so.
 *
 * Each entry point runs, element by element on the GPU, one of the device
 * functions the Markov step kernel inlines, so that tests can compare them
 * bit for bit with an independent implementation over exhaustive input
 * ranges.  They are not part of the sampling path.
 *
 * All pointers are device pointers; n >= 0; each call enqueues one kernel on
 * `stream` and returns DSPARK_OK or a DSPARK_ERR_* code (dspark_markov.h).
 */
#ifndef DSPARK_MARKOV_CHECK_H
#define DSPARK_MARKOV_CHECK_H

#include "dspark_markov.h"

#ifdef __cplusplus
extern "C" {
#endif

/* L[i] = log(-log(1 - u(h0 + i))), u(h) = RN((h + 0.5) / 2^32): the noise of
 * [P3] _gumbel with this library's own logarithm; h0 + i wraps modulo 2^32. */
DSPARK_API int dspark_check_noise_range(uint32_t h0, float *L, int64_t n, cudaStream_t stream);

/* Murmur3 noise hash of [P3] _StepKernel.kernel for ids[i]:
 * out[i] = MurmurHash3_x86_32(seed 0; lo(s'), hi(s'), lo(pos - 1 + salt), ids[i]),
 * s' = seed XOR (step << 32). */
DSPARK_API int dspark_check_hash(int64_t seed, int32_t step, int64_t pos, uint32_t salt, const uint32_t *ids,
                                 uint32_t *out, int64_t n, cudaStream_t stream);

/* Output transform of [P3] _logit: c[i] = cached BF16 of (base[i], bias[i]),
 * l[i] its FP32 value; cap = 0 means no soft cap. */
DSPARK_API int dspark_check_logit(const uint16_t *base, const uint16_t *bias, uint16_t *c, float *l, int64_t n,
                                  float mult, float cap, cudaStream_t stream);

/* key[i] = RN(RN(l[i] / temp) - L(h[i])) for temp != 0, else l[i] ([P2] _gumbel_key). */
DSPARK_API int dspark_check_key(const float *l, float temp, const uint32_t *h, float *key, int64_t n,
                                cudaStream_t stream);

/* own log and tanh of the library, elementwise. */
DSPARK_API int dspark_check_logf(const float *x, float *y, int64_t n, cudaStream_t stream);
DSPARK_API int dspark_check_tanhf(const float *x, float *y, int64_t n, cudaStream_t stream);

/* own exp of the library for x <= 0 (the logits-to-probabilities weights and
 * the confidence logistic), elementwise. */
DSPARK_API int dspark_check_expf(const float *x, float *y, int64_t n, cudaStream_t stream);

/* The library's division by one divisor (a correctly rounded reciprocal, the
 * quotient and one remainder correction -- Markstein's method -- in the range
 * where that is exact, the IEEE division elsewhere): y[i] = x[i] / d. */
DSPARK_API int dspark_check_div(const float *x, float d, float *y, int64_t n, cudaStream_t stream);

/* The same division against the IEEE quotient for every float whose bits lie
 * in [lo, lo + n) (n <= 2^32, wrapping): adds to out[0] the number whose bits
 * differ (two NaNs agree) and lowers out[1] to the smallest such bit
 * pattern.  out: two device words the caller sets to 0 and ~0 first. */
DSPARK_API int dspark_check_div_sweep(float d, uint32_t lo, int64_t n, unsigned long long *out,
                                      cudaStream_t stream);

/* The step kernel's bounds of the Gumbel noise -L(h), which let it skip
 * elements that cannot be the argmax (no counterpart in the pages: the pages
 * evaluate every key).  Host code only, no GPU and no stream: fills HOST
 * arrays ub[n], lb[n] with n >= 512; bucket b = 16 k + m of g = h | 1, k the
 * position of g's leading one and m the 4 bits after it; for every h of
 * bucket b, lb[b] <= -L(h) <= ub[b]; empty buckets hold 0.  Returns the
 * number of buckets (512) or DSPARK_ERR_INVALID_ARG. */
DSPARK_API int dspark_noise_bound_tables(float *ub, float *lb, int32_t n);

#ifdef __cplusplus
}
#endif
#endif
