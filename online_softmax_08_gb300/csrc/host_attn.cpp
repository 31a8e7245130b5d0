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
constexpr int CJ = 16;   // columns per chunk: the unit of every vector loop and reduction
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

#define HOST_INLINE static inline __attribute__((always_inline))

// GCC vector extensions of W floats, W the width of the target's vector
// registers (4 for NEON and SSE, 8 for AVX2, 16 for AVX-512), so that every
// vector lives in a register; no intrinsics.  A chunk of CJ columns is CJ / W
// vectors.
template <int W>
struct Vec {
  typedef float f __attribute__((vector_size(W * sizeof(float))));
  typedef int i __attribute__((vector_size(W * sizeof(int))));
  typedef float fu __attribute__((vector_size(W * sizeof(float)), aligned(4)));
};

template <int W>
HOST_INLINE typename Vec<W>::f vload(const float* p) {
  return *(const typename Vec<W>::fu*)p;
}
template <int W>
HOST_INLINE void vstore(float* p, typename Vec<W>::f x) {
  *(typename Vec<W>::fu*)p = x;
}
template <int W>
HOST_INLINE typename Vec<W>::f vsplat(float x) {
  return typename Vec<W>::f{} + x;
}

// 2^t for t <= 0, lane by lane
template <int W>
HOST_INLINE typename Vec<W>::f exp2_nonpos(typename Vec<W>::f t) {
  typedef typename Vec<W>::f vf;
  typedef typename Vec<W>::i vi;
  t = t < -127.f ? vsplat<W>(-127.f) : t;  // also maps -inf; 2^-127 and below become 0 below
  const vf n = (t + kRound) - kRound;      // nearest integer
  const vf f = t - n;                      // exact, in [-1/2, 1/2]
  vf p = vsplat<W>(kC7);
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

// Reductions of a chunk's CJ logical lanes (lane u = x[u / W][u % W]) by one
// fixed tree: for w = CJ/2, ..., 1, lane u takes op(lane u, lane u + w).  The
// steps with w >= W combine whole vectors, the rest run inside x[0]; the tree,
// and so the result, is the same for every W.
template <int W, class Op>
HOST_INLINE float chunk_reduce(typename Vec<W>::f (&x)[CJ / W], Op op) {
  for (int w = CJ / 2; w >= W; w >>= 1)
    for (int t = 0; t < w / W; ++t) x[t] = op(x[t], x[t + w / W]);
  for (int w = W / 2; w > 0; w >>= 1)
    for (int u = 0; u < w; ++u) x[0][u] = op(x[0][u], x[0][u + w]);
  return x[0][0];
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

void pack_block(const Problem& pr, long long bh, int kb) {
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

// s[r][:] = q[r] . kt, for RB rows and NVB vectors of keys at a time.  LANES:
// take four consecutive q values of a row as one vector and multiply by its
// lanes (one load per four multiply-adds per row; AArch64 has a multiply-add
// by vector lane); otherwise broadcast each q value from memory (x86).
template <int W, int RB, int NVB, bool LANES>
HOST_INLINE void block_scores(const float* __restrict q, const float* __restrict kt,
                              float* __restrict s, int Dp, int rows) {
  typedef typename Vec<W>::f vf;
  typedef typename Vec<4>::f v4;
  constexpr int NV = NVB;  // vectors per register block: NV * W keys
  static_assert(CJ % (NV * W) == 0, "register block inside a chunk");
  for (int j0 = 0; j0 < BK; j0 += NV * W) {  // this chunk's K strip stays in L1 across row blocks
    for (int r0 = 0; r0 < rows; r0 += RB) {
      const float* q0 = q + (size_t)r0 * Dp;
      vf acc[RB][NV];
#pragma GCC unroll 16
      for (int rr = 0; rr < RB; ++rr)
#pragma GCC unroll 16
        for (int t = 0; t < NV; ++t) acc[rr][t] = vf{};
      if (LANES) {  // Dp is a multiple of CJ, hence of 4
        for (int c = 0; c < Dp; c += 4) {
          v4 qv[RB];
#pragma GCC unroll 16
          for (int rr = 0; rr < RB; ++rr) qv[rr] = vload<4>(q0 + (size_t)rr * Dp + c);
#pragma GCC unroll 16
          for (int cc = 0; cc < 4; ++cc) {
            const float* kc = kt + (size_t)(c + cc) * BK + j0;
            vf kv[NV];
#pragma GCC unroll 16
            for (int t = 0; t < NV; ++t) kv[t] = vload<W>(kc + t * W);
#pragma GCC unroll 16
            for (int rr = 0; rr < RB; ++rr)
#pragma GCC unroll 16
              for (int t = 0; t < NV; ++t) acc[rr][t] = kv[t] * qv[rr][cc] + acc[rr][t];
          }
        }
      } else {
        const float* kc = kt + j0;
        for (int c = 0; c < Dp; ++c, kc += BK) {
          vf kv[NV];
#pragma GCC unroll 16
          for (int t = 0; t < NV; ++t) kv[t] = vload<W>(kc + t * W);
#pragma GCC unroll 16
          for (int rr = 0; rr < RB; ++rr) {
            const float a = q0[(size_t)rr * Dp + c];
#pragma GCC unroll 16
            for (int t = 0; t < NV; ++t) acc[rr][t] = a * kv[t] + acc[rr][t];
          }
        }
      }
#pragma GCC unroll 16
      for (int rr = 0; rr < RB; ++rr)
#pragma GCC unroll 16
        for (int t = 0; t < NV; ++t) vstore<W>(s + (size_t)(r0 + rr) * BK + j0 + t * W, acc[rr][t]);
    }
  }
}

// o[r] = alpha[r] o[r] + sum_jj p[r][jj] vp[jj], for RB rows and NVB vectors of
// columns at a time; LANES as in block_scores, over four consecutive p values
template <int W, int RB, int NVB, bool LANES>
HOST_INLINE void block_accumulate(const float* __restrict p, const float* __restrict vp,
                                  float* __restrict o, const float* __restrict alpha, int Dp,
                                  int rows) {
  typedef typename Vec<W>::f vf;
  typedef typename Vec<4>::f v4;
  constexpr int NV = NVB;  // vectors per register block: NV * W columns
  static_assert(CJ % (NV * W) == 0, "register block inside a chunk");
  for (int c0 = 0; c0 < Dp; c0 += NV * W) {  // this chunk's V strip stays in L1 across row blocks
    for (int r0 = 0; r0 < rows; r0 += RB) {
      const float* p0 = p + (size_t)r0 * BK;
      vf acc[RB][NV];
#pragma GCC unroll 16
      for (int rr = 0; rr < RB; ++rr) {
        const float a = alpha[r0 + rr];
#pragma GCC unroll 16
        for (int t = 0; t < NV; ++t) acc[rr][t] = vload<W>(o + (size_t)(r0 + rr) * Dp + c0 + t * W) * a;
      }
      if (LANES) {
        for (int jj = 0; jj < BK; jj += 4) {
          v4 pv[RB];
#pragma GCC unroll 16
          for (int rr = 0; rr < RB; ++rr) pv[rr] = vload<4>(p0 + (size_t)rr * BK + jj);
#pragma GCC unroll 16
          for (int j2 = 0; j2 < 4; ++j2) {
            const float* vr = vp + (size_t)(jj + j2) * Dp + c0;
            vf vv[NV];
#pragma GCC unroll 16
            for (int t = 0; t < NV; ++t) vv[t] = vload<W>(vr + t * W);
#pragma GCC unroll 16
            for (int rr = 0; rr < RB; ++rr)
#pragma GCC unroll 16
              for (int t = 0; t < NV; ++t) acc[rr][t] = vv[t] * pv[rr][j2] + acc[rr][t];
          }
        }
      } else {
        const float* vr = vp + c0;
        for (int jj = 0; jj < BK; ++jj, vr += Dp) {
          vf vv[NV];
#pragma GCC unroll 16
          for (int t = 0; t < NV; ++t) vv[t] = vload<W>(vr + t * W);
#pragma GCC unroll 16
          for (int rr = 0; rr < RB; ++rr) {
            const float pv = p0[(size_t)rr * BK + jj];
#pragma GCC unroll 16
            for (int t = 0; t < NV; ++t) acc[rr][t] = pv * vv[t] + acc[rr][t];
          }
        }
      }
#pragma GCC unroll 16
      for (int rr = 0; rr < RB; ++rr)
#pragma GCC unroll 16
        for (int t = 0; t < NV; ++t) vstore<W>(o + (size_t)(r0 + rr) * Dp + c0 + t * W, acc[rr][t]);
    }
  }
}

// the online update of (m, l) for one row of scores; the row becomes P
template <int W>
HOST_INLINE void row_update(float* __restrict sr, float& m, float& l, float& alpha) {
  typedef typename Vec<W>::f vf;
  constexpr int NV = CJ / W;
  auto vmax = [](auto a, auto b) { return b > a ? b : a; };
  auto vadd = [](auto a, auto b) { return a + b; };
  vf mx[NV];
  for (int t = 0; t < NV; ++t) mx[t] = vload<W>(sr + t * W);
  for (int j = CJ; j < BK; j += CJ)
    for (int t = 0; t < NV; ++t) {
      const vf x = vload<W>(sr + j + t * W);
      mx[t] = x > mx[t] ? x : mx[t];
    }
  const float mb = chunk_reduce<W>(mx, vmax);
  const float m_new = mb > m ? mb : m;
  if (m_new == -INFINITY) {  // nothing visible in this row yet
    alpha = 1.f;
    for (int j = 0; j < BK; ++j) sr[j] = 0.f;
    return;
  }
  alpha = exp2_nonpos<W>(vsplat<W>(m - m_new))[0];  // 0 on the first visible block (m = -inf)
  vf ls[NV];
  for (int t = 0; t < NV; ++t) ls[t] = vf{};
  for (int j = 0; j < BK; j += CJ)
    for (int t = 0; t < NV; ++t) {
      const vf pj = exp2_nonpos<W>(vload<W>(sr + j + t * W) - m_new);
      vstore<W>(sr + j + t * W, pj);
      ls[t] += pj;
    }
  l = alpha * l + chunk_reduce<W>(ls, vadd);
  m = m_new;
}

template <int W, int RB, int NVB, bool LANES>
HOST_INLINE void run_task_w(const Problem& pr, Scratch& sc, long long bh, int qt) {
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
    block_scores<W, RB, NVB, LANES>(sc.q, pr.kt + blk, sc.s, Dp, rows_p);
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
        row_update<W>(sc.s + (size_t)r * BK, sc.m[r], sc.l[r], sc.alpha[r]);
      } else {  // padding rows stay zero
        sc.alpha[r] = 1.f;
        for (int jj = 0; jj < BK; ++jj) sc.s[(size_t)r * BK + jj] = 0.f;
      }
    }
    block_accumulate<W, RB, NVB, LANES>(sc.s, pr.vp + blk, sc.o, sc.alpha, Dp, rows_p);
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

// multiply-add throughput: KV independent vector chains (enough to cover the
// latency of every FMA pipe) on W-float vectors
template <int W, int KV>
HOST_INLINE float fma_loop_w(long long iters, float a, float b) {
  typedef typename Vec<W>::f vf;
  vf acc[KV];
  for (int u = 0; u < KV; ++u) acc[u] = vsplat<W>((float)u * 1e-3f);
  const vf va = vsplat<W>(a), vb = vsplat<W>(b);
  // the running value is the addend (acc += va * vb), the form the kernels use:
  // a multiply-add that accumulates into its destination register
  for (long long it = 0; it < iters; ++it)
#pragma GCC unroll 16
    for (int u = 0; u < KV; ++u) acc[u] = va * vb + acc[u];
  // whole-vector adds, then the lanes of one vector (indexing the array by a
  // run-time lane would keep it in memory through the loop above)
  vf t = acc[0];
#pragma GCC unroll 16
  for (int u = 1; u < KV; ++u) t += acc[u];
  float s = 0.f;
#pragma GCC unroll 16
  for (int i = 0; i < W; ++i) s += t[i];
  return s;
}

template <int W>
HOST_INLINE void exp2_array_w(const float* __restrict t, float* __restrict y, long long n) {
  long long i = 0;
  for (; i + W <= n; i += W) vstore<W>(y + i, exp2_nonpos<W>(vload<W>(t + i)));
  if (i < n) {
    float buf[W];
    for (int u = 0; u < W; ++u) buf[u] = i + u < n ? t[i + u] : 0.f;
    const typename Vec<W>::f r = exp2_nonpos<W>(vload<W>(buf));
    for (long long u = 0; i + u < n; ++u) y[i + u] = r[u];
  }
}

// One instance per vector unit.  Each is compiled for its own target, with the
// templates above inlined into it, and picked at run time.
struct Kernels {
  void (*run_task)(const Problem&, Scratch&, long long, int);
  float (*fma_loop)(long long, float, float);
  void (*exp2_array)(const float*, float*, long long);
  int flops_per_iter;  // 2 * KV * W
};

#define DEFINE_KERNELS(NAME, TARGET, W, RB, NVB, LANES, KV)                              \
  TARGET void NAME##_run(const Problem& pr, Scratch& sc, long long bh, int qt) {         \
    run_task_w<W, RB, NVB, LANES>(pr, sc, bh, qt);                                       \
  }                                                                                      \
  TARGET float NAME##_fma(long long it, float a, float b) {                              \
    return fma_loop_w<W, KV>(it, a, b);                                                  \
  }                                                                                      \
  TARGET void NAME##_exp2(const float* t, float* y, long long n) { exp2_array_w<W>(t, y, n); } \
  const Kernels NAME = {NAME##_run, NAME##_fma, NAME##_exp2, 2 * KV * W};

#if defined(__x86_64__) && defined(__GNUC__) && !defined(__clang__)
// AVX-512 (32 registers of 16 floats), AVX2 + FMA (16 of 8), SSE (16 of 4)
// register blocks: rows x (vectors x width) of the score and output tiles
DEFINE_KERNELS(k_avx512, __attribute__((target("arch=x86-64-v4"))), 16, 8, 1, false, 8)
DEFINE_KERNELS(k_avx2, __attribute__((target("arch=x86-64-v3"))), 8, 4, 2, false, 8)
DEFINE_KERNELS(k_sse, , 4, 2, 4, false, 8)
const Kernels& kernels() {
  static const Kernels* k = [] {
    __builtin_cpu_init();
    if (__builtin_cpu_supports("x86-64-v4")) return &k_avx512;
    if (__builtin_cpu_supports("x86-64-v3")) return &k_avx2;
    return &k_sse;
  }();
  return *k;
}
#else
// AArch64 NEON: 32 registers of 4 floats, four FMA pipes of four-cycle latency
// 8 rows x 8 columns, multiply-add by vector lane: measured 6-7 % faster on
// Neoverse V2 than 4 rows x 16 columns with broadcast loads
DEFINE_KERNELS(k_neon, , 4, 8, 2, true, 16)
const Kernels& kernels() { return k_neon; }
#endif

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
  const Kernels& kern = kernels();
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
      kern.run_task(pr, sc, t % BH, qt);
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
  const Kernels& kern = kernels();
  if (!(seconds > 0.0)) seconds = 0.2;
  // calibrate the iteration count on one thread
  long long iters = 1 << 16;
  double el = 0.0;
  volatile float sink = 0.f;
  for (;;) {
    const auto t0 = std::chrono::steady_clock::now();
    sink = sink + kern.fma_loop(iters, 0.999999f, 1e-6f);
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
  total += kern.fma_loop(iters, 0.999999f, 1e-6f);
  el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  sink = sink + total;
  return (double)kern.flops_per_iter * (double)iters * nt / el / 1e9;
}

void fattn_host_exp2(const float* t, float* y, long long n) {
  if (t && y && n > 0) kernels().exp2_array(t, y, n);
}

}  // extern "C"
