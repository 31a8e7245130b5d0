/*
 * oracle.c -- plain, slow fp64 CPU attention.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, the smoke check in __graft_entry__.py and the cpu_baseline
 * leg of bench.py may load this library.  It shares no code with the CUDA
 * path under online_softmax_08_gb300/ and never calls into it.
 *
 * What it computes is the textbook definition of scaled dot-product
 * attention, written out with every intermediate materialised:
 *
 *   S = Q K^T * scale           "FlashAttention tiles exact softmax..." (page 1),
 *                               opening equations; "tm_flash_attention_math"
 *                               (page 3), "What we must compute, and why storage is the problem"
 *   P = softmax(S) by rows      three-pass safe softmax: max, sum, normalise
 *                               (page 3, "Safe softmax: the max-subtraction we cannot give up")
 *   O = P V,  LSE = m + ln l    the per-row statistic the backward pass keeps
 *                               ("Decoding flash attention", "The backward pass")
 *
 * Causal masking: key j is visible to query i iff j <= i; a masked score is
 * -inf before the row maximum is taken (page 1, "Causal masking fits inside
 * the tiled computation").
 *
 * The backward pass is the calculus of that definition (the pages give no
 * gradient formulas): dV = P^T dO, dP = dO V^T, D_i = sum_j P_ij dP_ij,
 * dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
 *
 * All tensors are contiguous [BH, N, d] fp64 (BH = batch * heads), row-major.
 * Compiled with -ffp-contract=off so that x86 and Arm hosts give the same bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef int64_t i64;

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Row i of S = scale * Q K^T for one head, with the causal mask applied as -inf. */
static void score_row(const double *qi, const double *kh, i64 N, i64 d, double scale,
                      int causal, i64 i, double *s) {
    for (i64 j = 0; j < N; ++j) {
        if (causal && j > i) {
            s[j] = -INFINITY;
            continue;
        }
        const double *kj = kh + j * d;
        double acc = 0.0;
        for (i64 c = 0; c < d; ++c) acc += qi[c] * kj[c];
        s[j] = scale * acc;
    }
}

/* Three-pass safe softmax of one materialised row, in place (s -> p).
 * Pass 1: m = max_j s_j.  Pass 2: l = sum_j exp(s_j - m).  Pass 3: p_j = exp(s_j - m) / l.
 * Every row here has at least one visible key (key 0 is visible to every
 * query, causal or not), so m is finite and l >= 1. */
static void safe_softmax_row(double *s, i64 N, double *m_out, double *l_out) {
    double m = -INFINITY;
    for (i64 j = 0; j < N; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (i64 j = 0; j < N; ++j) l += exp(s[j] - m);
    for (i64 j = 0; j < N; ++j) s[j] = exp(s[j] - m) / l;
    *m_out = m;
    *l_out = l;
}

/* Full forward for every head: materialise S for one head, softmax its rows,
 * then O = P V.  lse[bh, i] = m_i + ln l_i (natural log, scaled-logit units). */
int oracle_attn_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
                    i64 BH, i64 N, i64 d, double scale, int causal, int nthreads) {
    if (BH < 0 || N < 1 || d < 1) return 1;
    set_threads(nthreads);
    double *S = (double *)malloc((size_t)N * (size_t)N * sizeof(double));
    if (!S) return 2;
    for (i64 bh = 0; bh < BH; ++bh) {
        const double *qh = q + bh * N * d, *kh = k + bh * N * d, *vh = v + bh * N * d;
        double *oh = o + bh * N * d, *lh = lse + bh * N;
#pragma omp parallel for schedule(static)
        for (i64 i = 0; i < N; ++i) score_row(qh + i * d, kh, N, d, scale, causal, i, S + i * N);
#pragma omp parallel for schedule(static)
        for (i64 i = 0; i < N; ++i) {
            double m, l;
            safe_softmax_row(S + i * N, N, &m, &l);
            lh[i] = m + log(l);
        }
        /* O = P V */
#pragma omp parallel for schedule(static)
        for (i64 i = 0; i < N; ++i) {
            double *oi = oh + i * d;
            for (i64 c = 0; c < d; ++c) oi[c] = 0.0;
            const double *pi = S + i * N;
            for (i64 j = 0; j < N; ++j) {
                const double pij = pi[j];
                const double *vj = vh + j * d;
                for (i64 c = 0; c < d; ++c) oi[c] += pij * vj[c];
            }
        }
    }
    free(S);
    return 0;
}

/* The same definition for a list of (head, query row) samples: each sample
 * materialises its own row of S (the single-query form of page 3), softmaxes
 * it in three passes and forms o = sum_j p_j v_j.  o_out is [count, d]. */
int oracle_attn_fwd_rows(const double *q, const double *k, const double *v, i64 BH, i64 N, i64 d,
                         double scale, int causal, const i64 *bh_idx, const i64 *row_idx,
                         i64 count, double *o_out, double *lse_out, int nthreads) {
    if (N < 1 || d < 1) return 1;
    for (i64 t = 0; t < count; ++t)
        if (bh_idx[t] < 0 || bh_idx[t] >= BH || row_idx[t] < 0 || row_idx[t] >= N) return 1;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)N * sizeof(double));
        if (!s) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (i64 t = 0; t < count; ++t) {
            if (!s) continue;
            const i64 bh = bh_idx[t], i = row_idx[t];
            const double *qh = q + bh * N * d, *kh = k + bh * N * d, *vh = v + bh * N * d;
            score_row(qh + i * d, kh, N, d, scale, causal, i, s);
            double m, l;
            safe_softmax_row(s, N, &m, &l);
            lse_out[t] = m + log(l);
            double *ot = o_out + t * d;
            for (i64 c = 0; c < d; ++c) ot[c] = 0.0;
            for (i64 j = 0; j < N; ++j) {
                const double *vj = vh + j * d;
                for (i64 c = 0; c < d; ++c) ot[c] += s[j] * vj[c];
            }
        }
        free(s);
    }
    return err;
}

/* Textbook backward for the heads listed in heads[0..nheads) (all heads when
 * heads == NULL).  Outputs dq, dk, dv are [nheads, N, d], in the order listed. */
int oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout, i64 BH,
                    i64 N, i64 d, double scale, int causal, const i64 *heads, i64 nheads,
                    double *dq, double *dk, double *dv, int nthreads) {
    if (N < 1 || d < 1) return 1;
    if (!heads) nheads = BH;
    for (i64 t = 0; t < nheads; ++t)
        if (heads && (heads[t] < 0 || heads[t] >= BH)) return 1;
    set_threads(nthreads);
    double *P = (double *)malloc((size_t)N * (size_t)N * sizeof(double));
    double *dS = (double *)malloc((size_t)N * (size_t)N * sizeof(double));
    double *D = (double *)malloc((size_t)N * sizeof(double));
    if (!P || !dS || !D) {
        free(P);
        free(dS);
        free(D);
        return 2;
    }
    for (i64 t = 0; t < nheads; ++t) {
        const i64 bh = heads ? heads[t] : t;
        const double *qh = q + bh * N * d, *kh = k + bh * N * d, *vh = v + bh * N * d;
        const double *doh = dout + bh * N * d;
        double *dqh = dq + t * N * d, *dkh = dk + t * N * d, *dvh = dv + t * N * d;
        /* P = softmax(scale Q K^T) with the causal mask */
#pragma omp parallel for schedule(static)
        for (i64 i = 0; i < N; ++i) {
            double m, l;
            score_row(qh + i * d, kh, N, d, scale, causal, i, P + i * N);
            safe_softmax_row(P + i * N, N, &m, &l);
        }
        /* dP = dO V^T, D_i = sum_j P_ij dP_ij, dS = P o (dP - D) */
#pragma omp parallel for schedule(static)
        for (i64 i = 0; i < N; ++i) {
            const double *doi = doh + i * d;
            double *dsi = dS + i * N;
            const double *pi = P + i * N;
            double Di = 0.0;
            for (i64 j = 0; j < N; ++j) {
                const double *vj = vh + j * d;
                double acc = 0.0;
                for (i64 c = 0; c < d; ++c) acc += doi[c] * vj[c];
                dsi[j] = acc;
                Di += pi[j] * acc;
            }
            D[i] = Di;
            for (i64 j = 0; j < N; ++j) dsi[j] = pi[j] * (dsi[j] - Di);
        }
        /* dQ = scale * dS K */
#pragma omp parallel for schedule(static)
        for (i64 i = 0; i < N; ++i) {
            double *dqi = dqh + i * d;
            for (i64 c = 0; c < d; ++c) dqi[c] = 0.0;
            const double *dsi = dS + i * N;
            for (i64 j = 0; j < N; ++j) {
                const double *kj = kh + j * d;
                for (i64 c = 0; c < d; ++c) dqi[c] += dsi[j] * kj[c];
            }
            for (i64 c = 0; c < d; ++c) dqi[c] *= scale;
        }
        /* dV = P^T dO and dK = scale * dS^T Q: each thread owns a range of keys j
         * and walks every query row i. */
#pragma omp parallel
        {
#ifdef _OPENMP
            const i64 nt = omp_get_num_threads(), id = omp_get_thread_num();
#else
            const i64 nt = 1, id = 0;
#endif
            const i64 j0 = N * id / nt, j1 = N * (id + 1) / nt;
            for (i64 j = j0; j < j1; ++j)
                for (i64 c = 0; c < d; ++c) dvh[j * d + c] = dkh[j * d + c] = 0.0;
            for (i64 i = 0; i < N; ++i) {
                const double *pi = P + i * N, *dsi = dS + i * N;
                const double *doi = doh + i * d, *qi = qh + i * d;
                for (i64 j = j0; j < j1; ++j) {
                    const double pij = pi[j], dsij = dsi[j];
                    double *dvj = dvh + j * d, *dkj = dkh + j * d;
                    for (i64 c = 0; c < d; ++c) {
                        dvj[c] += pij * doi[c];
                        dkj[c] += dsij * qi[c];
                    }
                }
            }
            for (i64 j = j0; j < j1; ++j)
                for (i64 c = 0; c < d; ++c) dkh[j * d + c] *= scale;
        }
    }
    free(P);
    free(dS);
    free(D);
    return 0;
}

/* Tile classification of one head's (query tile, key tile) grid, by brute
 * enumeration.  Query tiles hold rows [i0, min(i0+block_q, N) - 1], key tiles
 * columns [j0, min(j0+block_k, N) - 1].  A tile is
 *   skipped iff causal and j0 > i_max (wholly above the diagonal, so no key of
 *           it is visible: page 1, "Causal masking fits inside the tiled
 *           computation"),
 *   masked  iff not skipped and (causal and j_max > i0, i.e. it crosses the
 *           diagonal, or it runs past N, the ragged last key tile),
 *   full    otherwise.
 * out[0] = full, out[1] = masked, out[2] = skipped. */
int oracle_tile_counts(i64 N, int causal, i64 block_q, i64 block_k, i64 *out) {
    if (N < 1 || block_q < 1 || block_k < 1) return 1;
    i64 full = 0, masked = 0, skipped = 0;
    for (i64 i0 = 0; i0 < N; i0 += block_q) {
        const i64 i_max = (i0 + block_q < N ? i0 + block_q : N) - 1;
        for (i64 j0 = 0; j0 < N; j0 += block_k) {
            const i64 j_max = (j0 + block_k < N ? j0 + block_k : N) - 1;
            if (causal && j0 > i_max)
                ++skipped;
            else if ((causal && j_max > i0) || j0 + block_k > N)
                ++masked;
            else
                ++full;
        }
    }
    out[0] = full;
    out[1] = masked;
    out[2] = skipped;
    return 0;
}
