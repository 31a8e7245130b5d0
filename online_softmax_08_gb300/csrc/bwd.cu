// bwd.cu -- FlashAttention backward main kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// The backward keeps only LSE from the forward pass and recomputes score
// tiles ("FlashAttention tiles exact softmax without materializing the score
// matrix", "Backward computation can trade recomputation for stored
// intermediates"; "Decoding flash attention", "The backward pass").  The
// pages give no gradient formulas; this kernel evaluates the calculus of the
// definition tile by tile:
//
//   P^T  = exp(scale K Q_i^T - LSE_i)        recomputed, never stored in HBM
//   dV  += P^T dO_i
//   dP^T = V dO_i^T
//   dS^T = P^T o (dP^T - D_i)                D_i = rowsum(dO_i o O_i), precomputed
//   dK  += dS^T Q_i                          (x scale in the epilogue)
//   dQ_i += dS K                             (fp32 partials added into a workspace;
//                                             x scale in the convert kernel)
//
// One CTA owns one 128-key block K_j, V_j of one (batch, head); its dK_j and
// dV_j accumulate in TMEM while the query blocks Q_i, dO_i (BQ rows) stream
// through a three-stage TMA ring.  With causal masking only query blocks i
// with queries >= the block's first key are visited.
//
// dQ strategy: each CTA forms a partial dQ_i^T = K^T dS_i^T per visited query
// block in TMEM; a drain warpgroup stages it in shared memory, 32 query rows at
// a time, and adds it into an fp32 accumulator with one bulk tensor reduce per
// half tile (measured 10-15 % faster than per-element red.global.add).  The alternative, a
// second pass parallel over query blocks, would recompute S and dP (two more
// matmuls per tile, 7 instead of 5).
//
// Steps are BQ = 64 queries; every MMA has M = 128 (at d = 64 the dQ^T MMA
// computes 64 padding rows).  TMEM (512 columns at d = 128): dK, dV, two S^T
// buffers, dP^T, dQ^T.  S^T of step i+1 is computed into the other buffer while
// step i's P is formed, so the tensor pipe never waits for the softmax of the
// same buffer.  P^T (bf16) overwrites the first half of its S^T buffer and feeds
// dV += P^T dO as the TMEM A operand; the fp32 P goes through shared memory to
// the warpgroup that forms dS.
//
// Warp roles (512 threads): warps 0-3 form P, warps 4-7 form dS (thread t of a
// warpgroup owns key row t = TMEM lane t), warps 8-11 drain dQ, warp 12 issues MMAs (the whole warp runs the
// loop, elect.sync picks the issuing lane), warp 13 issues TMA loads and
// stages LSE and D, warps 14-15 idle.
#define FATTN_INLINE_WAIT_SLOW_PATH
#include "common.cuh"
#include "ptx.cuh"

namespace fattn {
namespace {

template <int D>
struct Bwd {
  static constexpr int BK = 128;                    // keys per CTA
  static constexpr int BQ = 64;                     // queries per step
  static constexpr int NCH = BQ / 32;               // 32-column chunks of one step
  static constexpr int QST = 3;                     // Q/dO ring stages
  static constexpr int KHALF = BK * 128;            // 64-column half of a K/V or dS^T tile
  static constexpr int QHALF = BQ * 128;            // 64-column half of a Q/dO tile
  static constexpr int TILE_K = BK * D * 2;
  static constexpr int TILE_Q = BQ * D * 2;
  static constexpr int PT = BK * BQ * 2;            // dS^T tile (bf16)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_K;
  static constexpr int OFF_Q = OFF_V + TILE_K;                 // [QST]
  static constexpr int OFF_DO = OFF_Q + QST * TILE_Q;          // [QST]
  static constexpr int OFF_DS = OFF_DO + QST * TILE_Q;
  static constexpr int OFF_P = OFF_DS + PT;                    // fp32 P [BQ/4][128 keys][4]
  static constexpr int OFF_STAT = OFF_P + BK * BQ * 4;         // [QST] x {lse2[BQ], delta[BQ]}
  static constexpr int OFF_DQ = OFF_STAT + QST * 2 * BQ * 4;  // fp32 staging [32 q][D]
  static constexpr int OFF_BAR = OFF_DQ + 32 * D * 4;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr int THREADS = 512;
  // TMEM: dK, dV (d columns each), two S^T buffers, dP^T, dQ^T (BQ = 64 columns each)
  static constexpr uint32_t TM_DK = 0, TM_DV = D, TM_S = 2 * D, TM_DP = 2 * D + 2 * BQ,
                            TM_DQ = 2 * D + 3 * BQ;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BQ, false, false);   // S^T, dP^T
  static constexpr uint32_t IDESC_ACC = idesc_bf16_f32(128, D, false, true);   // dV, dK
  // dQ^T = K^T dS^T with M = 128: at d = 64 the upper 64 rows are padding
  static constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, BQ, true, true);
  // TMEM column of the packed P^T of buffer b for MMA K-step kk (16 queries = 8 columns)
  __host__ __device__ static constexpr uint32_t p_col(int b, int kk) {
    return TM_S + (uint32_t)b * BQ + 8u * kk;
  }
};

// Every barrier is waited on by parity, so no waiter may fall two phases
// behind: each one below can only complete its next phase after its waiters
// have consumed the current one.  That is why P_FULL has one barrier per S^T
// buffer (the P warpgroup runs up to a step ahead of the MMA warp) and why the
// epilogue waits for MMA_DONE, which completes once.
enum {
  B_KV = 0,
  B_S_FULL = 1,      // [2] MMA -> P warpgroup: S^T buffer ready
  B_P_FULL = 3,      // [2] P warpgroup -> MMA, dS warpgroup: P^T of a buffer in TMEM,
                     //     fp32 P in shared memory
  B_DP_FULL = 5,     // MMA -> dS warpgroup: dP^T ready
  B_DP_FREE = 6,     // dS warpgroup -> MMA: dP^T read
  B_DS_FULL = 7,     // dS warpgroup -> MMA: dS^T in shared memory
  B_DS_FREE = 8,     // MMA -> dS warpgroup: dK and dQ have read dS^T
  B_MMA_DONE = 9,    // MMA -> drain of the MMA warp and the epilogue: every MMA finished
  B_DQ_FULL = 10,    // MMA -> drain: dQ^T ready
  B_DQ_FREE = 11,    // drain -> MMA: dQ^T read
  B_Q_FULL = 12,     // [QST]
  B_Q_EMPTY = 15,    // [QST]
  B_PBUF_FREE = 18,  // dS warpgroup -> P warpgroup: fp32 P buffer read
  B_COUNT = 19,
};

template <int D>
__global__ void __launch_bounds__(Bwd<D>::THREADS, 1)
    fattn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dk,
                     const __grid_constant__ CUtensorMap tm_dv,
                     const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = Bwd<D>;
  constexpr int BQ = C::BQ, QST = C::QST;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N;
  const int kb = (int)(blockIdx.x / (unsigned)p.BH);  // key block; causal: heaviest first
  const int bh = (int)(blockIdx.x % (unsigned)p.BH);
  const int k0 = kb * C::BK;
  const int n_qb = (N + BQ - 1) / BQ;
  const int i_start = p.causal ? k0 / BQ : 0;
  const int n_it = n_qb - i_start;

  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * B_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wctx{abort_flag, p.err};

  if (threadIdx.x == 0) {
    mbar_init(bar(B_KV), 1);
    mbar_init(bar(B_S_FULL + 0), 1);
    mbar_init(bar(B_S_FULL + 1), 1);
    mbar_init(bar(B_P_FULL + 0), 128);
    mbar_init(bar(B_P_FULL + 1), 128);
    mbar_init(bar(B_PBUF_FREE), 128);
    mbar_init(bar(B_DP_FULL), 1);
    mbar_init(bar(B_DP_FREE), 128);
    mbar_init(bar(B_DS_FULL), 128);
    mbar_init(bar(B_DS_FREE), 1);
    mbar_init(bar(B_MMA_DONE), 1);
    mbar_init(bar(B_DQ_FULL), 1);
    mbar_init(bar(B_DQ_FREE), 128);
    for (int s = 0; s < QST; ++s) {
      mbar_init(bar(B_Q_FULL + s), 1 + 32);
      mbar_init(bar(B_Q_EMPTY + s), 1 + 256);
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 13) {
    // ---------------------------------------------------------------- loads
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar(B_KV), 2 * C::TILE_K);
      for (int h = 0; h < D / 64; ++h) {
        tma_load_3d(sbase + C::OFF_K + h * C::KHALF, &tm_k, bar(B_KV), h * 64, k0, bh);
        tma_load_3d(sbase + C::OFF_V + h * C::KHALF, &tm_v, bar(B_KV), h * 64, k0, bh);
      }
    }
    const float kLog2e = 1.4426950408889634f;
    int issued = 0;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % QST, use = it / QST;
      const int q0 = (i_start + it) * BQ;
      // a stage is refilled only after its readers are done; when the CTA is
      // aborting nothing more is issued (the decision is uniform over the warp)
      bool ok = use == 0 || mbar_wait(bar(B_Q_EMPTY + st), (use - 1) & 1, wctx, ERR_SITE_BWD | 0x01);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_Q_FULL + st), 2 * C::TILE_Q);
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(sbase + C::OFF_Q + st * C::TILE_Q + h * C::QHALF, &tm_q, bar(B_Q_FULL + st),
                      h * 64, q0, bh);
          tma_load_3d(sbase + C::OFF_DO + st * C::TILE_Q + h * C::QHALF, &tm_do,
                      bar(B_Q_FULL + st), h * 64, q0, bh);
        }
      }
      float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT + st * 2 * BQ * 4);
      for (int c = lane; c < BQ; c += 32) {
        const int q = q0 + c;
        const bool ok = q < N;
        // a query past N gets LSE = +inf, so its P column is exactly zero
        stat[c] = ok ? p.lse[(size_t)bh * N + q] * kLog2e : INFINITY;
        stat[BQ + c] = ok ? p.delta[(size_t)bh * N + q] : 0.f;
      }
      mbar_arrive(bar(B_Q_FULL + st));
      issued = it + 1;
    }
    if (lane == 0) {  // drain: at most one load per stage can still be landing
      mbar_drain(bar(B_KV), 0, wctx, ERR_SITE_BWD | 0x02);
      for (int it = max(0, issued - QST); it < issued; ++it)
        mbar_drain(bar(B_Q_FULL + it % QST), (it / QST) & 1, wctx, ERR_SITE_BWD | 0x03);
    }
    __syncwarp();
  } else if (warp == 12) {
    // ---------------------------------------------------------------- MMA issuer (whole warp)
    {
      const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sDS = sbase + C::OFF_DS;
      // D[128 x BQ] = X[128 keys x D] * Y[BQ x D]^T, both K-major
      auto mma_xyT = [&](uint32_t d_col, uint32_t x, uint32_t y) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t xo = (kk >> 2) * C::KHALF + (kk & 3) * 32;
          const uint32_t yo = (kk >> 2) * C::QHALF + (kk & 3) * 32;
          mma_bf16_ss_w(tmem + d_col, sdesc_sw128(x + xo, 16, 1024), sdesc_sw128(y + yo, 16, 1024),
                      C::IDESC_S, kk > 0);
        }
      };
      // dV += P^T (TMEM) * dO (MN-major)
      auto mma_dv = [&](int b, uint32_t sdo, bool acc) {
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_bf16_ts_w(tmem + C::TM_DV, tmem + C::p_col(b, kk),
                      sdesc_sw128(sdo + kk * 16 * 128, C::QHALF, 1024), C::IDESC_ACC,
                      (acc || kk > 0));
      };
      // dK += dS^T (K-major) * Q (MN-major)
      auto mma_dk = [&](uint32_t sq, bool acc) {
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * C::KHALF + (kk & 3) * 32;
          mma_bf16_ss_w(tmem + C::TM_DK, sdesc_sw128(sDS + ao, 16, 1024),
                      sdesc_sw128(sq + kk * 16 * 128, C::QHALF, 1024), C::IDESC_ACC,
                      (acc || kk > 0));
        }
      };
      // dQ^T[128 x BQ] = K^T[d x keys] * dS^T[keys x BQ], both MN-major; at d = 64 the
      // second 64-row block of A is read from the next tile (V) and is padding
      auto mma_dq = [&]() {
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          const uint32_t o = kk * 16 * 128;
          mma_bf16_ss_w(tmem + C::TM_DQ, sdesc_sw128(sK + o, C::KHALF, 1024),
                        sdesc_sw128(sDS + o, C::KHALF, 1024), C::IDESC_DQ, kk > 0);
        }
      };
      auto q_wait = [&](int it) {
        return __all_sync(0xffffffffu,
                          mbar_wait(bar(B_Q_FULL + it % QST), (it / QST) & 1, wctx, ERR_SITE_BWD | 0x11));
      };
      auto sQ = [&](int it) { return sbase + C::OFF_Q + (it % QST) * C::TILE_Q; };
      auto sDO = [&](int it) { return sbase + C::OFF_DO + (it % QST) * C::TILE_Q; };

      // any failed wait means the CTA is aborting: issue nothing more
      bool ok = __all_sync(0xffffffffu, mbar_wait(bar(B_KV), 0, wctx, ERR_SITE_BWD | 0x12));
      ok = ok && q_wait(0);
      if (ok) {
        tc_fence_after();
        mma_xyT(C::TM_S, sK, sQ(0));
        mma_commit_w(bar(B_S_FULL + 0));
        mma_xyT(C::TM_DP, sV, sDO(0));
        mma_commit_w(bar(B_DP_FULL));
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const bool next = it + 1 < n_it;
        const int b = it & 1;
        if (next) {  // S^T of the next step into the other buffer, ahead of P of this one;
                     // that buffer was last read by dV two steps back (earlier in pipe order)
          if (!(ok = q_wait(it + 1))) break;
          tc_fence_after();
          mma_xyT(C::TM_S + (b ^ 1) * BQ, sK, sQ(it + 1));
          mma_commit_w(bar(B_S_FULL + (b ^ 1)));
        }
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_P_FULL + b), (it >> 1) & 1, wctx,
                                                      ERR_SITE_BWD | 0x13))))
          break;
        tc_fence_after();
        mma_dv(b, sDO(it), it > 0);
        if (next) {  // dP^T of the next step as soon as this one is in registers
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_DP_FREE), it & 1, wctx, ERR_SITE_BWD | 0x16)))) break;
          tc_fence_after();
          mma_xyT(C::TM_DP, sV, sDO(it + 1));
          mma_commit_w(bar(B_DP_FULL));
        }
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_DS_FULL), it & 1, wctx, ERR_SITE_BWD | 0x15)))) break;
        tc_fence_after();
        mma_dk(sQ(it), it > 0);
        if (it >= 1) {
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_DQ_FREE), (it - 1) & 1, wctx,
                                                        ERR_SITE_BWD | 0x17))))
            break;
          tc_fence_after();
        }
        mma_dq();
        mma_commit_w(bar(B_DQ_FULL));
        mma_commit_w(bar(B_DS_FREE));
        mma_commit_w(bar(B_Q_EMPTY + it % QST));
      }
      // drain: every MMA issued by this thread has finished before TMEM is freed
      mma_commit_w(bar(B_MMA_DONE));
      mbar_drain(bar(B_MMA_DONE), 0, wctx, ERR_SITE_BWD | 0x18);
    }
    __syncwarp();
  } else if (warp >= 8 && warp < 12) {
    // ---------------------------------------------------------------- dQ drain
    const int t = threadIdx.x & 127;  // TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    for (int it = 0; it < n_it; ++it) {
      const int q0 = (i_start + it) * BQ;
      mbar_wait(bar(B_DQ_FULL), it & 1, wctx, ERR_SITE_BWD | 0x31);
      tc_fence_after();
      uint32_t r[2][32];
      tmem_ld32(tmem + lane_off + C::TM_DQ, r[0]);
      tmem_ld32(tmem + lane_off + C::TM_DQ + 32, r[1]);
      tmem_wait_ld();
      reg_fence32(r[0]);
      reg_fence32(r[1]);
      tc_fence_before();
      mbar_arrive(bar(B_DQ_FREE));
      // lanes are d (lanes >= d are padding), columns are queries: stage 32 query
      // rows at a time in shared memory and add them with one bulk tensor reduce
      const uint32_t sdq = sbase + C::OFF_DQ;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (t == 0) bulk_wait_read_all();  // the previous reduce has read the staging
        named_bar_sync(2, 128);
        if (t < D) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(sdq + (uint32_t)(c * D + t) * 4u),
                         "r"(r[h][c])
                         : "memory");
        }
        fence_proxy_async_smem();
        named_bar_sync(2, 128);
        if (t == 0) {
          tma_reduce_add_3d(&tm_dq, sdq, 0, q0 + 32 * h, bh);
          bulk_commit();
        }
      }
    }
    if (t == 0) bulk_wait_all();
    __syncwarp();
  } else if (warp < 8) {
    // ---------------------------------------------------------------- compute (warps 0-7)
    // Warpgroup 0 forms P^T for a step, warpgroup 1 forms dS^T from it, so the
    // two run one step apart.  Thread t owns key row t (TMEM lane t) and all
    // BQ query columns of the step.
    const int w = warp >> 2;
    const int t = threadIdx.x & 127;
    const int ctid = threadIdx.x;        // 0..255
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int kr = k0 + t;
    const float sl2 = p.scale_log2;
    constexpr int NCH = C::NCH;
    const uint32_t tS = tmem + lane_off + C::TM_S;
    const uint32_t tDP = tmem + lane_off + C::TM_DP;
    const uint32_t pbuf = sbase + C::OFF_P + t * 16;  // chunk c of row t at pbuf + c * 128 * 16

    if (w == 0) {
      // ---- P^T = exp2(S^T * scale * log2e - LSE2), masked: bf16 into TMEM, fp32 into smem
      for (int it = 0; it < n_it; ++it) {
        const int st = it % QST;
        const int q0 = (i_start + it) * BQ;
        mbar_wait(bar(B_Q_FULL + st), (it / QST) & 1, wctx, ERR_SITE_BWD | 0x21);
        const float4* lse2 = reinterpret_cast<const float4*>(smem + C::OFF_STAT + st * 2 * BQ * 4);
        // key kr sees query q iff kr < N and (not causal or kr <= q); queries
        // past N already have LSE2 = +inf.  Only blocks that cross the diagonal
        // or hold keys past N need the element mask.
        const bool need_mask = (p.causal && k0 + C::BK - 1 > q0) || (k0 + C::BK > N);
        int lo = 0;
        if (kr >= N) lo = BQ;
        else if (p.causal) lo = min(max(kr - q0, 0), BQ);
        const int b = it & 1;
        mbar_wait(bar(B_S_FULL + b), (it >> 1) & 1, wctx, ERR_SITE_BWD | 0x22);
        tc_fence_after();
        if (it > 0) mbar_wait(bar(B_PBUF_FREE), (it - 1) & 1, wctx, ERR_SITE_BWD | 0x23);
#pragma unroll
        for (int h = 0; h < NCH; h += 2) {  // 64 queries at a time
          uint32_t u[2][32];
          const int nc = min(2, NCH - h);
#pragma unroll
          for (int c = 0; c < 2; ++c)
            if (c < nc) tmem_ld32(tS + b * BQ + (h + c) * 32, u[c]);
          tmem_wait_ld();
          reg_fence32(u[0]);
          reg_fence32(u[1]);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (c >= nc) break;
            float pv[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const int col = (h + c) * 32 + i;
              const float4 l4 = lse2[col / 4];
              pv[i] = ex2(fmaf(__uint_as_float(u[c][i]), sl2, -l4.x));
              pv[i + 1] = ex2(fmaf(__uint_as_float(u[c][i + 1]), sl2, -l4.y));
              pv[i + 2] = ex2(fmaf(__uint_as_float(u[c][i + 2]), sl2, -l4.z));
              pv[i + 3] = ex2(fmaf(__uint_as_float(u[c][i + 3]), sl2, -l4.w));
            }
            if (need_mask) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if ((h + c) * 32 + i < lo) pv[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              st_shared_v4(pbuf + (((h + c) * 32 + i) / 4) * 128 * 16, __float_as_uint(pv[i]),
                           __float_as_uint(pv[i + 1]), __float_as_uint(pv[i + 2]),
                           __float_as_uint(pv[i + 3]));
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(pv[2 * e], pv[2 * e + 1]);
            // columns [0, BQ/2) of S^T hold P^T: chunk h+c goes to 16 columns
            // that this thread has already read
            tmem_st16(tS + b * BQ + (h + c) * 16, pk);
          }
        }
        mbar_arrive(bar(B_Q_EMPTY + st));  // LSE2 of this stage is no longer read
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_P_FULL + b));
      }
    } else {
      // ---- dS^T = P^T o (dP^T - D) -> bf16 -> shared memory (K-major for dK, MN-major for dQ)
      for (int it = 0; it < n_it; ++it) {
        const int st = it % QST;
        mbar_wait(bar(B_Q_FULL + st), (it / QST) & 1, wctx, ERR_SITE_BWD | 0x24);
        const float4* dlt =
            reinterpret_cast<const float4*>(smem + C::OFF_STAT + st * 2 * BQ * 4 + BQ * 4);
        // all of dP^T into registers first, so the next dP^T can be computed meanwhile
        mbar_wait(bar(B_DP_FULL), it & 1, wctx, ERR_SITE_BWD | 0x26);
        tc_fence_after();
        uint32_t u[NCH][32];
#pragma unroll
        for (int c = 0; c < NCH; ++c) tmem_ld32(tDP + c * 32, u[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < NCH; ++c) reg_fence32(u[c]);
        tc_fence_before();
        mbar_arrive(bar(B_DP_FREE));
        mbar_wait(bar(B_P_FULL + (it & 1)), (it >> 1) & 1, wctx, ERR_SITE_BWD | 0x25);
        if (it > 0) {  // the previous dK / dQ MMAs have read the dS^T buffer
          mbar_wait(bar(B_DS_FREE), (it - 1) & 1, wctx, ERR_SITE_BWD | 0x27);
          tc_fence_after();
        }
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float ds[32];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 pf = *reinterpret_cast<const float4*>(
                smem + C::OFF_P + (size_t)((c * 32 + i) / 4) * 128 * 16 + t * 16);
            const float4 d4 = dlt[(c * 32 + i) / 4];
            ds[i] = pf.x * (__uint_as_float(u[c][i]) - d4.x);
            ds[i + 1] = pf.y * (__uint_as_float(u[c][i + 1]) - d4.y);
            ds[i + 2] = pf.z * (__uint_as_float(u[c][i + 2]) - d4.z);
            ds[i + 3] = pf.w * (__uint_as_float(u[c][i + 3]) - d4.w);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {  // four 16-byte chunks of 8 queries
            const int col = c * 32 + e * 8;
            const int half = col >> 6, chunk = (col & 63) >> 3;
            st_shared_v4(sbase + C::OFF_DS + half * C::KHALF + t * 128 + ((chunk ^ (t & 7)) << 4),
                         pack_bf16x2(ds[e * 8], ds[e * 8 + 1]),
                         pack_bf16x2(ds[e * 8 + 2], ds[e * 8 + 3]),
                         pack_bf16x2(ds[e * 8 + 4], ds[e * 8 + 5]),
                         pack_bf16x2(ds[e * 8 + 6], ds[e * 8 + 7]));
          }
        }
        mbar_arrive(bar(B_PBUF_FREE));
        mbar_arrive(bar(B_Q_EMPTY + st));  // D of this stage is no longer read
        fence_proxy_async_smem();
        mbar_arrive(bar(B_DS_FULL));
      }
    }

    // ---- epilogue (both warpgroups): dK = scale * acc, dV = acc -> bf16 -> smem
    // (K/V tiles are free) -> TMA
    // MMA_DONE completes once, after every MMA of the CTA (K, V, dK, dV are final)
    mbar_wait(bar(B_MMA_DONE), 0, wctx, ERR_SITE_BWD | 0x28);
    tc_fence_after();
    constexpr int EW = D / 2;  // d columns per warpgroup
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t col0 = which == 0 ? C::TM_DK : C::TM_DV;
      const uint32_t dst = sbase + (which == 0 ? C::OFF_K : C::OFF_V);
      const float mul = which == 0 ? p.scale : 1.f;
#pragma unroll
      for (int c = 0; c < EW / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + col0 + w * EW + c * 32, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int col = w * EW + c * 32 + q4 * 8;
          const int half = col >> 6, chunk = (col & 63) >> 3;
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(r[q4 * 8 + e]) * mul;
          st_shared_v4(dst + half * C::KHALF + t * 128 + ((chunk ^ (t & 7)) << 4),
                       pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                       pack_bf16x2(f[6], f[7]));
        }
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 256);
    if (ctid == 0) {
      for (int h = 0; h < D / 64; ++h) {
        tma_store_3d(&tm_dk, sbase + C::OFF_K + h * C::KHALF, h * 64, k0, bh);
        tma_store_3d(&tm_dv, sbase + C::OFF_V + h * C::KHALF, h * 64, k0, bh);
      }
      bulk_commit();
      bulk_wait_all();
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                   const CUtensorMap& tdq, const BwdParams& p, cudaStream_t stream) {
  using C = Bwd<D>;
  static_assert(C::SMEM <= 232448, "shared memory budget");
  static_assert(C::TM_DQ + C::BQ <= 512, "TMEM budget");
  cudaError_t e = cudaFuncSetAttribute(fattn_bwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const long long n_kb = (p.N + C::BK - 1) / C::BK;
  const long long blocks = n_kb * p.BH;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fattn_bwd_kernel<D><<<(unsigned)blocks, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tdo, tdk,
                                                                          tdv, tdq, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const CUtensorMap& tdq_acc, const BwdParams& p, cudaStream_t stream) {
  if (d == 128) return launch<128>(tq, tk, tv, tdo, tdk, tdv, tdq_acc, p, stream);
  if (d == 64) return launch<64>(tq, tk, tv, tdo, tdk, tdv, tdq_acc, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fattn
