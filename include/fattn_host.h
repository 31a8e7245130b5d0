/*
 * fattn_host.h -- C-ABI of libfattn_host: exact flash-style attention on the
 * host CPU cores, fp32.
 *
 * The same operation as fattn_fwd in fattn.h, for every (batch b, head h):
 *
 *     S = scale * Q K^T            (never stored)
 *     P = softmax(S) row by row    (causal: key j visible to query i iff j <= i)
 *     O = P V,   LSE_i = m_i + ln l_i = ln sum_j exp(S_ij)
 *
 * computed with the online-softmax recurrence over blocks of 64 keys for
 * tiles of 64 queries, so that the working set of a tile stays in the core's
 * caches and the keys and values stream past once ("tm_flash_attention_math",
 * "The block-wise update, and the full algorithm" and "Why the same math
 * matters on a CPU").  This is a separate library with host pointers only; it
 * is not a fallback for the GPU entry points of libfattn, which never call it.
 *
 * Layout.  q, k, v, o are HOST pointers to contiguous fp32 [B, H, N, d]
 * (row-major, d innermost); lse is a HOST pointer to fp32 [B, H, N].  No
 * alignment is required.  o and lse must not overlap q, k or v.
 *
 * Numerics.  fp32 throughout, multiply-adds fused where the host has a fused
 * multiply-add (every AArch64 host; x86-64 with AVX2/FMA), the exponential
 * evaluated by the library's own exp2 (a degree-7 Taylor polynomial of 2^f
 * after range reduction; within 1.5 ulp of 2^t on [-126, 0], 0 below -126.5).
 * Every reduction runs in a fixed order: the result is the same, bit for bit,
 * for any thread count.  Inputs must be finite.
 *
 * Threads.  n_threads <= 0 means the OpenMP default (all cores the process may
 * use).  The call is synchronous and returns when O and LSE are written.  It
 * allocates, for the duration of the call, packed copies of K and V (about
 * 2 * B*H*ceil(N/64)*64 * ceil(d/16)*16 floats) and a few 16-KB tiles per
 * thread.
 */
#ifndef FATTN_HOST_H_
#define FATTN_HOST_H_

#ifdef __cplusplus
extern "C" {
#endif

#define FATTN_HOST_MAX_D 256

enum {
  FATTN_HOST_OK = 0,
  FATTN_HOST_ERR_INVALID_ARG = 1, /* negative size, null pointer, scale not finite and > 0 */
  FATTN_HOST_ERR_UNSUPPORTED = 2, /* d < 1 or d > FATTN_HOST_MAX_D */
  FATTN_HOST_ERR_NO_MEMORY = 6    /* the packed copies or a thread's tiles could not be allocated */
};

/* Forward pass.  Writes o [B,H,N,d] and lse [B,H,N] (natural log, in units of
 * scaled scores).  B*H = 0 or N = 0 is a valid empty call.  Returns one of the
 * codes above; on an argument error nothing is written. */
int fattn_host_fwd(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                   int H, int N, int d, float scale, int causal, int n_threads);

/* The number of threads n_threads <= 0 stands for. */
int fattn_host_max_threads(void);

/* Measured fp32 multiply-add throughput of n_threads threads (<= 0: all), in
 * GFLOP/s (2 FLOP per fmaf), from a register-resident loop of independent
 * fmaf chains run for about `seconds`: the peak the forward pass is compared
 * with. */
double fattn_host_fma_peak_gflops(int n_threads, double seconds);

/* y[i] = 2^t[i] by the library's exp2, for t[i] <= 0 (diagnostic, so the
 * approximation can be tested against its stated bound). */
void fattn_host_exp2(const float* t, float* y, long long n);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_HOST_H_ */
