/*
 * fattn_testing.h -- test and measurement hooks exported by libfattn.
 *
 * These two calls are NOT part of the attention interface (fattn.h): the
 * library's own tests use the first to exercise its failure reporting, and the
 * benchmark uses the second to measure a ceiling of the forward kernel.  No
 * product code path calls either.  The pages have no counterpart to them.
 */
#ifndef FATTN_TESTING_H_
#define FATTN_TESTING_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Failure-path check: launches one warp that waits, through the kernels'
 * bounded-wait routine, on a barrier that nothing completes, with a short
 * limit (2^21 SM clock cycles, about 1 ms).  The wait then records code 0x301
 * in the device error word (fattn_device_error then returns
 * FATTN_ERR_TIMEOUT with that code) and the kernel returns; the context stays
 * usable.  Asynchronous on stream.  Returns FATTN_OK, FATTN_ERR_UNSUPPORTED
 * or FATTN_ERR_CUDA; with FATTN_DEBUG set, FATTN_ERR_TIMEOUT (the post-call
 * check of fattn.h sees the word). */
int fattn_check_wait_timeout(void* stream);

/* Measured throughput of the exponential unit of the current device, in ex2
 * evaluations per second: a kernel of independent ex2.approx chains on every
 * SM, timed with events on `stream` (a warm-up launch, then one timed launch;
 * the call synchronises with the timed launch).  It is the second ceiling of
 * the forward pass, which takes one exponential per visible score.  Returns
 * FATTN_OK, FATTN_ERR_INVALID_ARG (per_second NULL) or FATTN_ERR_CUDA. */
int fattn_ex2_throughput(double* per_second, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_TESTING_H_ */
