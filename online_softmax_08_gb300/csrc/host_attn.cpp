// host_attn.cpp -- flash-style exact attention on the host CPU cores, fp32.
//
// The online-softmax recurrence of the GPU forward pass, with the CPU's caches
// in the role of shared memory ("tm_flash_attention_math", "Why the same math
// matters on a CPU"): a tile of BQ queries keeps its running max m, running sum
// l and unnormalised output o~ resident while blocks of BK keys and values
// stream past once; the N x N score matrix never exists.  For every key block
// ("The block-wise update, and the full algorithm"):
//
//     S      = scale Q K^T, masked entries set to -inf before the block max
//     m_new  = max(m, rowmax S),  alpha = exp(m - m_new),  P = exp(S - m_new)
//     l      = alpha l + rowsum P,  o~ = alpha o~ + P V
//
// and after the last block O = o~ / l, LSE = m + ln l.  A row that has seen no
// visible key yet (m_new = -inf) keeps alpha = 1 and P = 0, since
// exp(-inf - (-inf)) is undefined.
//
// Scores are kept in base-2 units (Q is multiplied by scale * log2(e) once) so
// every exponential is an exp2.  That exp2 is this file's own: t = n + f with
// n the integer nearest to t (found by adding and subtracting 1.5 * 2^23) and
// f in [-1/2, 1/2]; 2^f from the Taylor series of e^(f ln 2) to degree 7
// (truncation error below 6e-9 relative), evaluated by Horner's rule; 2^n
// written into the exponent field.  Arguments are never positive (every score
// is at most the running max: "Proof of numerical stability"), and below
// -126.5 the result is 0.
//
// The arithmetic is written with vector types of CJ floats, one multiply-add
// per statement (the build contracts each into a fused multiply-add where the
// host has one), and every reduction runs in one fixed order, so the result
// does not depend on the thread count.
//
// Layout of the work.  A pre-pass packs K, per (head, key block), transposed
// and zero-padded ([Dp][BK], Dp = d rounded up to CJ) and V zero-padded
// ([BK][Dp]); the main pass runs one task per (head, query tile) over the
// threads, longest causal tiles first.
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <chrono>

#ifdef _OPENMP
#include <omp.h>
#endif

#include "fattn_host.h"

namespace {

constexpr int BQ = 64;   // query rows per task
constexpr int BK = 64;   // keys per block
constexpr int CJ = 16;   // floats per vector (one AVX-512 register, four NEON registers)
constexpr int RB = 4;    // query rows per register block
constexpr int DMAX = FATTN_HOST_MAX_D;

constexpr double kLn2 = 0.693147180559945309417232121458176568;
constexpr double kLog2e = 1.442695040888963407359924681001892137;

// Taylor coefficients of 2^f = e^(f ln 2): (ln 2)^k / k!
constexpr double taylor(int k) {
  double c = 1.0;
  for (int i = 1; i <= k; ++i) c = c * kLn2 / i;
  return c;
}
constexpr float kC0 = (float)taylor(0), kC1 = (float)taylor(1), kC2 = (float)taylor(2),
                kC3 = (float)taylor(3), kC4 = (float)taylor(4), kC5 = (float)taylor(5),
                kC6 = (float)taylor(6), kC7 = (float)taylor(7);
// adding 1.5 * 2^23 rounds a float of magnitude below 2^22 to an integer
constexpr float kRound = 12582912.f;

// GCC vector extensions: the compiler maps them onto whatever vector unit the
// target has (AVX-512, AVX2, SSE, NEON); no intrinsics
typedef float vf __attribute__((vector_size(CJ * sizeof(float))));
typedef int vi __attribute__((vector_size(CJ * sizeof(int))));
typedef float vf_u __attribute__((vector_size(CJ * sizeof(float)), aligned(4)));

#if defined(__x86_64__) && defined(__GNUC__) && !defined(__clang__)
// the hot functions are also compiled for x86-64-v3 (AVX2 + FMA) and
// x86-64-v4 (AVX-512); the loader picks the best the host supports
#define HOST_CLONES __attribute__((target_clones("arch=x86-64-v4", "arch=x86-64-v3", "default")))
#else
#define HOST_CLONES
#endif
#define HOST_INLINE static inline __attribute__((always_inline))

HOST_INLINE vf load(const float* p) { return *(const vf_u*)p; }
HOST_INLINE void store(float* p, vf x) { *(vf_u*)p = x; }
HOST_INLINE vf splat(float x) { return vf{} + x; }

// 2^t for t <= 0, lane by lane
HOST_INLINE vf exp2_nonpos(vf t) {
  t = t < -127.f ? splat(-127.f) : t;  // also maps -inf; 2^-127 and below become 0 below
  const vf n = (t + kRound) - kRound;  // nearest integer
  const vf f = t - n;                  // exact, in [-1/2, 1/2]
  vf p = splat(kC7);
  p = p * f + kC6;
  p = p * f + kC5;
  p = p * f + kC4;
  p = p * f + kC3;
  p = p * f + kC2;
  p = p * f + kC1;
  p = p * f + kC0;
  const vi e = __builtin_convertvector(n, vi) + 127;  // 0 for n = -127: the scale is then +0
  return p * (vf)(e << 23);
}

struct Problem {
  const float *q, *k, *v;
  float *o, *lse;
  long long BH;
  int N, d, Dp, nkb, nqt;
  float qscale;  // scale * log2(e)
  int causal;
  float *kt, *vp;  // packed blocks: [BH][nkb][Dp][BK] and [BH][nkb][BK][Dp]
};

HOST_CLONES void pack_block(const Problem& pr, long long bh, int kb) {
  const int j0 = kb * BK, kn = std::min(BK, pr.N - j0), d = pr.d, Dp = pr.Dp;
  const size_t blk = ((size_t)bh * pr.nkb + kb) * (size_t)Dp * BK;
  float* __restrict kt = pr.kt + blk;
  float* __restrict vp = pr.vp + blk;
  const float* __restrict k = pr.k + ((size_t)bh * pr.N + j0) * d;
  const float* __restrict v = pr.v + ((size_t)bh * pr.N + j0) * d;
  for (int jj = 0; jj < BK; ++jj) {
    float* vr = vp + (size_t)jj * Dp;
    const int live = jj < kn ? d : 0;
    if (live) memcpy(vr, v + (size_t)jj * d, sizeof(float) * d);
    for (int c = live; c < Dp; ++c) vr[c] = 0.f;
  }
  // transpose in CJ x CJ squares so both sides stay within a few cache lines
  for (int c0 = 0; c0 < Dp; c0 += CJ)
    for (int jb = 0; jb < BK; jb += CJ)
      for (int c = c0; c < c0 + CJ; ++c)
        for (int jj = jb; jj < jb + CJ; ++jj)
          kt[(size_t)c * BK + jj] = (jj < kn && c < d) ? k[(size_t)jj * d + c] : 0.f;
}

struct Scratch {
  float* q;      // [BQ][Dp] pre-scaled queries (padded rows and columns zero)
  float* o;      // [BQ][Dp] unnormalised output o~
  float* s;      // [BQ][BK] scores, then probabilities
  float m[BQ], l[BQ], alpha[BQ];
};

// s[r][:] = q[r] . kt, for RB rows at a time
HOST_INLINE void block_scores(const float* __restrict q, const float* __restrict kt,
                              float* __restrict s, int Dp, int rows) {
  for (int r0 = 0; r0 < rows; r0 += RB) {
    const float* q0 = q + (size_t)r0 * Dp;
    for (int j0 = 0; j0 < BK; j0 += CJ) {
      vf acc[RB];
#pragma GCC unroll 4
      for (int rr = 0; rr < RB; ++rr) acc[rr] = vf{};
      const float* kc = kt + j0;
      for (int c = 0; c < Dp; ++c, kc += BK) {
        const vf kv = load(kc);
#pragma GCC unroll 4
        for (int rr = 0; rr < RB; ++rr) acc[rr] = q0[(size_t)rr * Dp + c] * kv + acc[rr];
      }
#pragma GCC unroll 4
      for (int rr = 0; rr < RB; ++rr) store(s + (size_t)(r0 + rr) * BK + j0, acc[rr]);
    }
  }
}

// o[r] = alpha[r] o[r] + sum_jj p[r][jj] vp[jj], for RB rows at a time
HOST_INLINE void block_accumulate(const float* __restrict p, const float* __restrict vp,
                                  float* __restrict o, const float* __restrict alpha, int Dp,
                                  int rows) {
  for (int r0 = 0; r0 < rows; r0 += RB) {
    const float* p0 = p + (size_t)r0 * BK;
    for (int c0 = 0; c0 < Dp; c0 += CJ) {
      vf acc[RB];
#pragma GCC unroll 4
      for (int rr = 0; rr < RB; ++rr)
        acc[rr] = load(o + (size_t)(r0 + rr) * Dp + c0) * alpha[r0 + rr];
      const float* vr = vp + c0;
      for (int jj = 0; jj < BK; ++jj, vr += Dp) {
        const vf vv = load(vr);
#pragma GCC unroll 4
        for (int rr = 0; rr < RB; ++rr) acc[rr] = p0[(size_t)rr * BK + jj] * vv + acc[rr];
      }
#pragma GCC unroll 4
      for (int rr = 0; rr < RB; ++rr) store(o + (size_t)(r0 + rr) * Dp + c0, acc[rr]);
    }
  }
}

// lanes of x combined pairwise in a fixed order: (0..7 with 8..15), then halves again
HOST_INLINE float lane_max(vf x) {
  for (int w = CJ / 2; w > 0; w >>= 1)
    for (int u = 0; u < w; ++u) x[u] = x[u + w] > x[u] ? x[u + w] : x[u];
  return x[0];
}
HOST_INLINE float lane_sum(vf x) {
  for (int w = CJ / 2; w > 0; w >>= 1)
    for (int u = 0; u < w; ++u) x[u] = x[u] + x[u + w];
  return x[0];
}

// the online update of (m, l) for one row of scores; the row becomes P
HOST_INLINE void row_update(float* __restrict sr, float& m, float& l, float& alpha) {
  vf mx = load(sr);
#pragma GCC unroll 4
  for (int j = CJ; j < BK; j += CJ) {
    const vf x = load(sr + j);
    mx = x > mx ? x : mx;
  }
  const float mb = lane_max(mx);
  const float m_new = mb > m ? mb : m;
  if (m_new == -INFINITY) {  // nothing visible in this row yet
    alpha = 1.f;
    for (int j = 0; j < BK; j += CJ) store(sr + j, vf{});
    return;
  }
  alpha = exp2_nonpos(splat(m - m_new))[0];  // 0 on the first visible block (m = -inf)
  vf ls = vf{};
#pragma GCC unroll 4
  for (int j = 0; j < BK; j += CJ) {
    const vf pj = exp2_nonpos(load(sr + j) - m_new);
    store(sr + j, pj);
    ls += pj;
  }
  l = alpha * l + lane_sum(ls);
  m = m_new;
}

HOST_CLONES void run_task(const Problem& pr, Scratch& sc, long long bh, int qt) {
  const int d = pr.d, Dp = pr.Dp, N = pr.N;
  const int i0 = qt * BQ, rows = std::min(BQ, N - i0);
  const int rows_p = (rows + RB - 1) / RB * RB;
  const float* qg = pr.q + ((size_t)bh * N + i0) * d;
  for (int r = 0; r < rows_p; ++r) {
    float* qr = sc.q + (size_t)r * Dp;
    float* orow = sc.o + (size_t)r * Dp;
    for (int c = 0; c < Dp; ++c) {
      qr[c] = (r < rows && c < d) ? qg[(size_t)r * d + c] * pr.qscale : 0.f;
      orow[c] = 0.f;
    }
    sc.m[r] = -INFINITY;
    sc.l[r] = 0.f;
  }
  // key blocks: all of them, or (causal) those that start at or before the tile's last row
  const int kb_end = pr.causal ? (i0 + rows - 1) / BK + 1 : pr.nkb;
  for (int kb = 0; kb < kb_end; ++kb) {
    const int j0 = kb * BK;
    const size_t blk = ((size_t)bh * pr.nkb + kb) * (size_t)Dp * BK;
    block_scores(sc.q, pr.kt + blk, sc.s, Dp, rows_p);
    // masks before the block max: keys past N, and (causal) keys after the query
    const bool ragged = j0 + BK > N;
    const bool diag = pr.causal && j0 + BK - 1 > i0;
    if (ragged || diag) {
      for (int r = 0; r < rows_p; ++r) {
        float* sr = sc.s + (size_t)r * BK;
        const int lim = std::min(N, pr.causal ? i0 + r + 1 : N) - j0;  // visible: jj < lim
        for (int jj = std::max(lim, 0); jj < BK; ++jj) sr[jj] = -INFINITY;
      }
    }
    for (int r = 0; r < rows_p; ++r) {
      if (r < rows) {
        row_update(sc.s + (size_t)r * BK, sc.m[r], sc.l[r], sc.alpha[r]);
      } else {  // padding rows stay zero
        sc.alpha[r] = 1.f;
        for (int jj = 0; jj < BK; ++jj) sc.s[(size_t)r * BK + jj] = 0.f;
      }
    }
    block_accumulate(sc.s, pr.vp + blk, sc.o, sc.alpha, Dp, rows_p);
  }
  // O = o~ / l;  LSE = m + ln l, back from base-2 units
  float* og = pr.o + ((size_t)bh * N + i0) * d;
  for (int r = 0; r < rows; ++r) {
    const float l = sc.l[r];
    const float* orow = sc.o + (size_t)r * Dp;
    for (int c = 0; c < d; ++c) og[(size_t)r * d + c] = orow[c] / l;
    pr.lse[(size_t)bh * N + i0 + r] = (float)(((double)sc.m[r] + log2((double)l)) * kLn2);
  }
}

int threads_for(int n_threads) {
#ifdef _OPENMP
  return n_threads > 0 ? n_threads : omp_get_max_threads();
#else
  (void)n_threads;
  return 1;
#endif
}

void* alloc_floats(size_t n) {
  const size_t bytes = (n * sizeof(float) + 63) / 64 * 64;
  return aligned_alloc(64, bytes ? bytes : 64);
}

// multiply-add throughput: KV independent vector chains, enough to cover the
// latency of every FMA pipe
constexpr int KV = 8;

HOST_CLONES float fma_loop(long long iters, float a, float b) {
  vf acc[KV];
  for (int u = 0; u < KV; ++u) acc[u] = splat((float)u * 1e-3f);
  const vf va = splat(a), vb = splat(b);
  for (long long it = 0; it < iters; ++it)
#pragma GCC unroll 8
    for (int u = 0; u < KV; ++u) acc[u] = acc[u] * va + vb;
  vf s = vf{};
  for (int u = 0; u < KV; ++u) s += acc[u];
  return lane_sum(s);
}

HOST_CLONES void exp2_array(const float* __restrict t, float* __restrict y, long long n) {
  long long i = 0;
  for (; i + CJ <= n; i += CJ) store(y + i, exp2_nonpos(load(t + i)));
  if (i < n) {
    float buf[CJ];
    for (int u = 0; u < CJ; ++u) buf[u] = i + u < n ? t[i + u] : 0.f;
    const vf r = exp2_nonpos(load(buf));
    for (long long u = 0; i + u < n; ++u) y[i + u] = r[u];
  }
}

}  // namespace

extern "C" {

int fattn_host_fwd(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                   int H, int N, int d, float scale, int causal, int n_threads) {
  if (B < 0 || H < 0 || N < 0) return FATTN_HOST_ERR_INVALID_ARG;
  if (d < 1 || d > DMAX) return FATTN_HOST_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_HOST_ERR_INVALID_ARG;
  const long long BH = (long long)B * H;
  if (BH == 0 || N == 0) return FATTN_HOST_OK;
  if (!q || !k || !v || !o || !lse) return FATTN_HOST_ERR_INVALID_ARG;

  Problem pr{};
  pr.q = q, pr.k = k, pr.v = v, pr.o = o, pr.lse = lse;
  pr.BH = BH, pr.N = N, pr.d = d;
  pr.Dp = (d + CJ - 1) / CJ * CJ;
  pr.nkb = (N + BK - 1) / BK;
  pr.nqt = (N + BQ - 1) / BQ;
  pr.qscale = (float)((double)scale * kLog2e);
  pr.causal = causal ? 1 : 0;
  const size_t packed = (size_t)BH * pr.nkb * pr.Dp * BK;
  pr.kt = (float*)alloc_floats(packed);
  pr.vp = (float*)alloc_floats(packed);
  if (!pr.kt || !pr.vp) {
    free(pr.kt);
    free(pr.vp);
    return FATTN_HOST_ERR_NO_MEMORY;
  }
  const long long n_blocks = BH * pr.nkb;
  const long long n_tasks = BH * pr.nqt;
  const int nt = (int)std::max(1LL, std::min<long long>(threads_for(n_threads), n_tasks));
  int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nt) reduction(| : failed)
#endif
  {
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
    for (long long t = 0; t < n_blocks; ++t) pack_block(pr, t / pr.nkb, (int)(t % pr.nkb));

    Scratch sc;
    sc.q = (float*)alloc_floats((size_t)BQ * pr.Dp);
    sc.o = (float*)alloc_floats((size_t)BQ * pr.Dp);
    sc.s = (float*)alloc_floats((size_t)BQ * BK);
    const bool ok = sc.q && sc.o && sc.s;
    if (!ok) failed = 1;
    // (the implicit barrier of the loop above orders the packing before any task)
    // causal: the last query tiles see the most keys, so they go first
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (long long t = 0; t < n_tasks; ++t) {
      if (!ok) continue;
      const int qt = pr.causal ? pr.nqt - 1 - (int)(t / BH) : (int)(t / BH);
      run_task(pr, sc, t % BH, qt);
    }
    free(sc.q);
    free(sc.o);
    free(sc.s);
  }
  free(pr.kt);
  free(pr.vp);
  return failed ? FATTN_HOST_ERR_NO_MEMORY : FATTN_HOST_OK;
}

int fattn_host_max_threads(void) { return threads_for(0); }

double fattn_host_fma_peak_gflops(int n_threads, double seconds) {
  const int nt = threads_for(n_threads);
  if (!(seconds > 0.0)) seconds = 0.2;
  // calibrate the iteration count on one thread
  long long iters = 1 << 16;
  double el = 0.0;
  volatile float sink = 0.f;
  for (;;) {
    const auto t0 = std::chrono::steady_clock::now();
    sink = sink + fma_loop(iters, 0.999999f, 1e-6f);
    el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
    if (el >= seconds * 0.25 || iters >= (1LL << 40)) break;
    iters *= 2;
  }
  iters = (long long)(iters * (seconds / std::max(el, 1e-9)));
  if (iters < 1) iters = 1;
  const auto t0 = std::chrono::steady_clock::now();
  float total = 0.f;
#ifdef _OPENMP
#pragma omp parallel num_threads(nt) reduction(+ : total)
#endif
  total += fma_loop(iters, 0.999999f, 1e-6f);
  el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  sink = sink + total;
  return 2.0 * KV * CJ * (double)iters * nt / el / 1e9;
}

void fattn_host_exp2(const float* t, float* y, long long n) {
  if (t && y && n > 0) exp2_array(t, y, n);
}

}  // extern "C"
