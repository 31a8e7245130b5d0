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
// dV_j accumulate in TMEM while 128-query blocks Q_i, dO_i stream through TMA
// rings.  With causal masking only query blocks i with queries >= the block's
// first key are visited.
//
// Every MMA has M = 128 and, but for dQ at d = 64, N = 128 (an SS MMA with a
// 64-wide N reads a full A operand from shared memory for half the work):
// TMEM holds dK and dV (d columns each), a region X for S^T whose first half is
// overwritten in place by the bf16 P^T, and a region Y that holds dP^T, then
// (over dP^T's first half) the bf16 dS^T that dK takes as its TMEM operand.
// The MMA warp issues, per step i,
//
//   dP(i) -> Y  dV(i)  S(i+1) -> X  dK(i) (first half)  dK(i) (second half)  dQ(i)
//
// dP(i) does not wait for P(i), so dS(i) starts as soon as it lands; dV(i) and
// S(i+1) execute while dS(i) is formed, and so does the half of dK(i) over the
// queries of the compute warps' first pass.  P(i+1) is formed while the rest
// of dK(i), dQ(i) and the next dP execute.  Each compute warpgroup keeps the
// bf16 P^T of its 64 queries in registers from P to dS, so X can take S(i+1)
// right after dV(i).  The MMA pipe runs in issue order, so dP(i + 1)'s commit
// also tells the compute warps that dK(i) and dQ(i) have read dS^T(i).
//
// d = 128: dQ^T = K^T dS^T (M = d) goes over dP^T in Y.  A drain warpgroup reads
// it out of TMEM (freeing Y for dP(i+1)) and adds it into an fp32 accumulator
// with bulk tensor reduces of 16 query rows, staged round-robin through four
// shared-memory buffers so that filling one overlaps the reduces reading the
// others (two buffers were 11 % faster than one, three 1.2 % faster than two,
// four 3.8 % faster than three).  Each SM's bulk-copy unit adds at most about
// 25 bytes per cycle, and a step hands it 64 KB; together with the MMA
// operands, TMA loads, dS stores and the staging they share shared-memory
// bandwidth, and these two bound the kernel.
//
// d = 64: dQ^T would be an M = 128 MMA half of which is padding, so dQ = dS K
// (M = 128 queries, N = 64) is computed instead, into a TMEM region Z of its
// own: only the next dQ waits for the drain.  Each drain warp holds 32 query
// rows and adds them by itself, with reduces of 32 rows x 32 columns through
// two buffers of its own (16 % faster than dQ^T over Y for the whole non-causal
// backward at B 4, H 16, N 2048, 12 % causal).
//
// The alternative to the dQ reduces, a second pass parallel over query blocks,
// would recompute S and dP (seven matmuls per tile instead of five).
//
// Warp roles (512 threads): warps 0-7 form P and dS, warpgroup w for queries
// [64w, 64w + 64) of each step (thread t of a warpgroup owns key row t = TMEM
// lane t), warps 8-11 drain dQ (or dQ^T), warp 12 issues MMAs (the whole warp runs the
// loop, elect.sync picks the issuing lane), warp 13 issues TMA loads and stages
// LSE and D, warps 14-15 idle.  Registers move from the last warpgroup to the
// drain warpgroup (setmaxnreg).
#define FATTN_INLINE_WAIT_SLOW_PATH
#include "common.cuh"
#include "ptx.cuh"

namespace fattn {
namespace {

// Shape of the dQ staging (compile-time, for A/B builds): query rows per bulk
// reduce, staging buffers, and whether the layout keeps 1 KB of slack to align
// the dynamic shared memory (0: the kernel requires an aligned base and
// reports a misaligned one through the error word).
#ifndef FATTN_DQ_ROWS
#define FATTN_DQ_ROWS 16
#endif
#ifndef FATTN_DQ_BUFS
#define FATTN_DQ_BUFS 4
#endif
#ifndef FATTN_SMEM_SLACK
#define FATTN_SMEM_SLACK 0
#endif

template <int D>
struct Bwd {
  static constexpr int BK = 128;                 // keys per CTA
  static constexpr int BQ = 128;                 // queries per step
  static constexpr int QST = D == 128 ? 2 : 3;   // Q (+ LSE, D) ring stages
  static constexpr int OST = D == 128 ? 1 : 2;   // dO ring stages
  static constexpr int HALF = 128 * 128;         // 64-column (128-byte) half of a 128-row tile
  static constexpr int TILE = 128 * D * 2;       // 128 rows of K, V, Q or dO (bf16)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;                   // [QST]
  static constexpr int OFF_DO = OFF_Q + QST * TILE;            // [OST]
  static constexpr int OFF_DS = OFF_DO + OST * TILE;           // dS^T [128 keys][128 q] bf16
  static constexpr int OFF_STAT = OFF_DS + 2 * HALF;           // [QST] x {-lse2[BQ], delta[BQ]}
  // dQ staging: NDQ buffers of RPC query rows (fp32), filled round-robin, so that
  // NDQ - 1 bulk reduces are in flight while the next buffer is filled
  static constexpr int RPC = FATTN_DQ_ROWS;
  static constexpr int NDQ = FATTN_DQ_BUFS;
  // at d = 64 dQ = dS K is an N = 64 MMA with queries on the TMEM lanes (dQ^T would
  // need M = 128, half of it padding): each drain warp adds its own 32 query rows
  // with reduces of 32 rows x 32 columns (128-byte swizzled), through two buffers
  // of its own
  static constexpr bool DQ_QL = D == 64;
  static constexpr int DQ_WBUF = 32 * D * 4;  // one drain warp's 32 rows (fp32)
  static constexpr int OFF_DQ = OFF_STAT + QST * 2 * BQ * 4;  // fp32 staging
  static constexpr int DQ_BYTES = DQ_QL ? 4 * 2 * DQ_WBUF : NDQ * RPC * D * 4;
  static constexpr int OFF_BAR = OFF_DQ + DQ_BYTES;
  static constexpr int SLACK = FATTN_SMEM_SLACK;
  static constexpr int SMEM = OFF_BAR + 256 + SLACK;
  static constexpr int THREADS = 512;
  static constexpr uint32_t TM_DK = 0, TM_DV = D, TM_X = 2 * D, TM_Y = 2 * D + 128;
  // where dQ (or dQ^T) goes: d = 64, a region Z of its own, so dP(i + 1) need not
  // wait for the drain to read dQ(i); d = 128, over dP^T in Y (TMEM is full)
  static constexpr bool DQ_OWN = 2 * D + 384 <= 512;
  static constexpr uint32_t TM_Z = DQ_OWN ? 2 * D + 256 : TM_Y;
  static_assert(!DQ_QL || DQ_OWN, "dQ with queries on the lanes needs its own region");
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BQ, false, false);   // S^T, dP^T
  static constexpr uint32_t IDESC_ACC = idesc_bf16_f32(128, D, false, true);   // dV, dK
  // d = 64: dQ = dS K (M = 128 queries, N = 64); d = 128: dQ^T = K^T dS^T
  static constexpr uint32_t IDESC_DQ =
      DQ_QL ? idesc_bf16_f32(BQ, D, true, true) : idesc_bf16_f32(128, BQ, true, true);
  // registers per thread after the split (sum x 128 threads = the launch's 65536)
  // (64 for the MMA and loader warps: at 56 the MMA warp spilled, and its local
  // loads sat in the issue loop that feeds the tensor pipe)
  static constexpr int REG_COMPUTE = 128, REG_DRAIN = 192, REG_CTRL = 64;
  static_assert(2 * REG_COMPUTE + REG_DRAIN + REG_CTRL == 4 * 128, "register split");
  // TMEM column of the packed P^T for dV's K-step kk (16 queries = 8 columns); the
  // warpgroup of queries [64w, 64w + 64) keeps its P^T at X + 64w
  __host__ __device__ static constexpr uint32_t p_col(int kk) {
    return TM_X + 64u * (uint32_t)(kk >> 2) + 8u * (uint32_t)(kk & 3);
  }
  // the same for the packed dS^T that dK reads: each warpgroup writes it over the
  // first half of the dP^T columns it has read, Y + 64w
  __host__ __device__ static constexpr uint32_t ds_col(int kk) {
    return TM_Y + 64u * (uint32_t)(kk >> 2) + 8u * (uint32_t)(kk & 3);
  }
};

// Every barrier is waited on by parity, so no waiter may fall two phases
// behind: each one below can only complete its next phase after its waiters
// have consumed the current one (the MMA warp's issue order chains them).
//
// S_FULL has one slot per Q stage: the phase of step j's slot completes with the
// loader's 32 arrivals (LSE2 and D of step j stored) and the commit of S(j).  The
// loader arrives for step j + QST only after Q_EMPTY(j), which the compute warps
// reach after their wait on step j's phase, and S(j + QST) is issued only after
// that load, so no phase collects arrivals of two steps.
enum {
  B_KV = 0,
  B_P_FULL = 1,     // compute warps -> MMA: P^T (bf16) in X, S^T read
  B_DS_HALF = 2,    // compute warps -> MMA: the first 32 queries of each half of dS^T in TMEM
  B_DP_FULL = 3,    // MMA -> compute warps: dP^T in Y
  B_DS_FULL = 4,    // compute warps -> MMA: dS^T in TMEM and shared memory, dP^T read
  B_DQ_FULL = 5,    // MMA -> drain: dQ (d = 64, in Z) or dQ^T (d = 128, in Y)
  B_DQ_FREE = 6,    // drain -> MMA: dQ read, its region may be overwritten
  B_MMA_DONE = 7,   // MMA -> epilogue and the MMA warp's drain: every MMA finished
  B_S_FULL = 8,     // [QST] MMA + loader -> compute warps: S^T(i) in X, LSE2 and D of step i
  B_Q_FULL = 11,    // [QST] Q tile of a step (TMA)
  B_Q_EMPTY = 14,   // [QST] Q tile, LSE2 and D of a step no longer read
  B_O_FULL = 17,    // [OST] dO tile
  B_O_EMPTY = 19,   // [OST]
  B_COUNT = 21,
};
static_assert(Bwd<128>::QST <= 3 && Bwd<64>::QST <= 3 && Bwd<64>::OST <= 2, "barrier slots");

// Two-lane fp32 arithmetic (one instruction for a pair of queries; each lane
// rounds exactly as the scalar instruction would).
// r = a * b + c with b shared by both lanes
__device__ __forceinline__ void fma_x2(float a0, float a1, float b, float c0, float c1, float& r0,
                                       float& r1) {
  asm("{\n\t.reg .b64 a, b, c, r;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %4};\n\t"
      "mov.b64 c, {%5, %6};\n\t"
      "fma.rn.f32x2 r, a, b, c;\n\t"
      "mov.b64 {%0, %1}, r;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c0), "f"(c1));
}
// r = p * (x - y)
__device__ __forceinline__ void mul_sub_x2(float p0, float p1, float x0, float x1, float y0,
                                           float y1, float& r0, float& r1) {
  asm("{\n\t.reg .b64 p, x, y, r;\n\t"
      "mov.b64 p, {%2, %3};\n\t"
      "mov.b64 x, {%4, %5};\n\t"
      "mov.b64 y, {%6, %7};\n\t"
      "sub.rn.f32x2 x, x, y;\n\t"
      "mul.rn.f32x2 r, p, x;\n\t"
      "mov.b64 {%0, %1}, r;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(p0), "f"(p1), "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}

template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// VARLEN: the CTA's sequence comes from p.vl.cu_seqlens (packed head-major
// rows); otherwise the dense [B, H, N, d] layout.
template <int D, bool VARLEN>
__global__ void __launch_bounds__(Bwd<D>::THREADS, 1)
    fattn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dk,
                     const __grid_constant__ CUtensorMap tm_dv,
                     const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = Bwd<D>;
  constexpr int BQ = C::BQ, QST = C::QST, OST = C::OST;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  if (C::SLACK < 1023 && (raw & 1023u)) {  // no room to align: report and leave
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0u, (unsigned)(ERR_SITE_BWD | 0x41));
    return;
  }
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // key block kb (causal: heaviest first).  Dense: key-block-major within groups
  // of heads; varlen: one
  // (sequence, head) unit after another, so the CTAs in flight share their
  // unit's Q, dO and dQ accumulator in L2
  const int units = VARLEN ? p.vl.B * p.vl.H : p.BH;
  const int n_kb_grid = (p.N + C::BK - 1) / C::BK;
  int kb, unit;
  if (VARLEN) {
    kb = (int)(blockIdx.x % (unsigned)n_kb_grid);
    unit = (int)(blockIdx.x / (unsigned)n_kb_grid);
  } else {  // heads in groups whose Q, dO and dQ accumulator stay in L2 (p.group)
    grouped_order(blockIdx.x, units, n_kb_grid, p.group, &kb, &unit);
  }
  SeqView seq;
  if constexpr (VARLEN) {
    if (!seq_view(p.vl, p.N, unit / p.vl.H, unit % p.vl.H, unit, p.N, &seq)) {
      if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0u, (unsigned)(ERR_SITE_BWD | 0x40));
      return;
    }
    if (kb * C::BK >= seq.N) return;  // this sequence is shorter: nothing to do
  } else {
    seq = SeqView{p.N, 0, unit, (long long)unit * p.N};
  }
  const int N = seq.N;
  const int bh = seq.z;        // TMA z coordinate
  const int row0 = seq.row0;   // first row of the sequence in the tensor
  const int k0 = kb * C::BK;
  const int n_qb = (N + BQ - 1) / BQ;
  const int i_start = p.causal ? k0 / BQ : 0;
  const int n_it = n_qb - i_start;

  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * B_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wctx{abort_flag, p.err};

  // The loader thread initialises the barriers and issues the K and V loads
  // before the CTA-wide sync, so their latency overlaps the TMEM allocation.
  if (warp == 13 && lane == 0) {
    mbar_init(bar(B_KV), 1);
    mbar_init(bar(B_P_FULL), 256);
    mbar_init(bar(B_DP_FULL), 1);
    mbar_init(bar(B_DS_HALF), 256);
    mbar_init(bar(B_DS_FULL), 256);
    mbar_init(bar(B_DQ_FULL), 1);
    mbar_init(bar(B_DQ_FREE), 128);
    mbar_init(bar(B_MMA_DONE), 1);
    for (int s = 0; s < QST; ++s) {
      mbar_init(bar(B_S_FULL + s), 1 + 32);
      mbar_init(bar(B_Q_FULL + s), 1);
      mbar_init(bar(B_Q_EMPTY + s), 1 + 256);
    }
    for (int s = 0; s < OST; ++s) {
      mbar_init(bar(B_O_FULL + s), 1);
      mbar_init(bar(B_O_EMPTY + s), 1);
    }
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    mbar_arrive_expect_tx(bar(B_KV), 2 * C::TILE);
    for (int h = 0; h < D / 64; ++h) {
      tma_load_3d(sbase + C::OFF_K + h * C::HALF, &tm_k, bar(B_KV), h * 64, row0 + k0, bh);
      tma_load_3d(sbase + C::OFF_V + h * C::HALF, &tm_v, bar(B_KV), h * 64, row0 + k0, bh);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 12) {
    regs_dec<C::REG_CTRL>();
    if (warp == 13) {
      // ---------------------------------------------------------------- loads
      // (K and V went out before the sync)
      const float kLog2e = 1.4426950408889634f;
      int q_issued = 0, o_issued = 0;
      // Q(i) is released by dK(i), dO(i) by dV(i); in the MMA order dV(i) precedes
      // dK(i) precedes dV(i + 1), so loading Q(i), dO(i) alternately never waits
      // on a later release before an earlier one.
      for (int it = 0; it < n_it; ++it) {
        const int q0 = (i_start + it) * BQ;
        {
          const int st = it % QST, use = it / QST;
          const bool ok = use == 0 ||
                          mbar_wait(bar(B_Q_EMPTY + st), (use - 1) & 1, wctx, ERR_SITE_BWD | 0x01);
          if (!__all_sync(0xffffffffu, ok)) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(B_Q_FULL + st), C::TILE);
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d(sbase + C::OFF_Q + st * C::TILE + h * C::HALF, &tm_q,
                          bar(B_Q_FULL + st), h * 64, row0 + q0, bh);
          }
          q_issued = it + 1;
          float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT + st * 2 * BQ * 4);
          float l[BQ / 32], dl[BQ / 32];
#pragma unroll
          for (int j = 0; j < BQ / 32; ++j) {
            const int q = q0 + lane + 32 * j;
            // -LSE2; a query past N gets -inf, so its P column is exactly zero
            l[j] = q < N ? -p.lse[seq.stat0 + q] * kLog2e : -INFINITY;
            dl[j] = q < N ? p.delta[seq.stat0 + q] : 0.f;
          }
#pragma unroll
          for (int j = 0; j < BQ / 32; ++j) {
            stat[lane + 32 * j] = l[j];
            stat[BQ + lane + 32 * j] = dl[j];
          }
          mbar_arrive(bar(B_S_FULL + st));
        }
        {
          const int so = it % OST, use = it / OST;
          const bool ok = use == 0 ||
                          mbar_wait(bar(B_O_EMPTY + so), (use - 1) & 1, wctx, ERR_SITE_BWD | 0x04);
          if (!__all_sync(0xffffffffu, ok)) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(B_O_FULL + so), C::TILE);
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d(sbase + C::OFF_DO + so * C::TILE + h * C::HALF, &tm_do,
                          bar(B_O_FULL + so), h * 64, row0 + q0, bh);
          }
          o_issued = it + 1;
        }
      }
      if (lane == 0) {  // drain: at most one load per stage can still be landing
        mbar_drain(bar(B_KV), 0, wctx, ERR_SITE_BWD | 0x02);
        for (int it = max(0, q_issued - QST); it < q_issued; ++it)
          mbar_drain(bar(B_Q_FULL + it % QST), (it / QST) & 1, wctx, ERR_SITE_BWD | 0x03);
        for (int it = max(0, o_issued - OST); it < o_issued; ++it)
          mbar_drain(bar(B_O_FULL + it % OST), (it / OST) & 1, wctx, ERR_SITE_BWD | 0x05);
      }
      __syncwarp();
    } else if (warp == 12) {
      // ---------------------------------------------------------------- MMA issuer (whole warp)
      const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sDS = sbase + C::OFF_DS;
      // D[128 x 128] = X[128 rows x D] * Y[128 rows x D]^T, both K-major
      auto mma_xyT = [&](uint32_t d_col, uint32_t x, uint32_t y) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = (kk >> 2) * C::HALF + (kk & 3) * 32;
          mma_bf16_ss_w(tmem + d_col, sdesc_sw128(x + o, 16, 1024), sdesc_sw128(y + o, 16, 1024),
                        C::IDESC_S, kk > 0);
        }
      };
      // dV += P^T (TMEM, 16 queries = 8 packed columns per step) * dO (MN-major)
      auto mma_dv = [&](uint32_t sdo, bool acc) {
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_bf16_ts_w(tmem + C::TM_DV, tmem + C::p_col(kk),
                        sdesc_sw128(sdo + kk * 16 * 128, C::HALF, 1024), C::IDESC_ACC,
                        (acc || kk > 0));
      };
      // dK += dS^T (TMEM, over dP^T in Y) * Q (MN-major), over the 16-query steps kk
      // of one pass: pass 0 takes queries 0-31 of each 64-query half (kk = 0, 1, 4,
      // 5), pass 1 queries 32-63 (kk = 2, 3, 6, 7), as the compute warps store them.
      // With A in TMEM the MMA reads only Q from shared memory, whose bandwidth the
      // step's MMAs, TMA loads, dS stores and dQ reduces share
      auto mma_dk = [&](uint32_t sq, bool acc, int pass) {
#pragma unroll
        for (int j = 0; j < BQ / 32; ++j) {
          const int kk = (j >> 1) * 4 + pass * 2 + (j & 1);
          mma_bf16_ts_w(tmem + C::TM_DK, tmem + C::ds_col(kk),
                        sdesc_sw128(sq + kk * 16 * 128, C::HALF, 1024), C::IDESC_ACC,
                        (acc || kk > 0));
        }
      };
      // d = 64: dQ[BQ x D] = dS[BQ x keys] * K[keys x D]; d = 128: dQ^T[D x BQ] =
      // K^T[D x keys] * dS^T[keys x BQ]; all operands MN-major
      auto mma_dq = [&]() {
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          const uint32_t o = kk * 16 * 128;
          const uint64_t dk_ = sdesc_sw128(sK + o, C::HALF, 1024);
          const uint64_t ds_ = sdesc_sw128(sDS + o, C::HALF, 1024);
          mma_bf16_ss_w(tmem + C::TM_Z, C::DQ_QL ? ds_ : dk_, C::DQ_QL ? dk_ : ds_, C::IDESC_DQ,
                        kk > 0);
        }
      };
      auto wait_all = [&](int b, int parity, uint32_t site) {
        return __all_sync(0xffffffffu, mbar_wait(bar(b), parity & 1, wctx, ERR_SITE_BWD | site));
      };
      // A wait on a phase that has already completed still costs the warp a few hundred
      // cycles, and the pipe runs dry behind it (the warp cannot issue far ahead of
      // it). So at d = 64 phases that are usually complete are tested together with
      // the one the next MMA needs, in one overlapped test (2-3 % faster there; no
      // difference at d = 128); the bounded waits follow only for what is still open.
      auto all_done2 = [&](int b0, int p0, int b1, int p1) {
        return __all_sync(0xffffffffu, mbar_try_wait2(bar(b0), p0 & 1, bar(b1), p1 & 1));
      };
      auto all_done3 = [&](int b0, int p0, int b1, int p1, int b2, int p2) {
        return __all_sync(0xffffffffu,
                          mbar_try_wait3(bar(b0), p0 & 1, bar(b1), p1 & 1, bar(b2), p2 & 1));
      };
      auto sQ = [&](int it) { return sbase + C::OFF_Q + (it % QST) * C::TILE; };
      auto sDO = [&](int it) { return sbase + C::OFF_DO + (it % OST) * C::TILE; };

      // any failed wait means the CTA is aborting: issue nothing more
      bool ok = wait_all(B_KV, 0, 0x12) && wait_all(B_Q_FULL, 0, 0x11);
      if (ok) {
        tc_fence_after();
        mma_xyT(C::TM_X, sK, sQ(0));
        mma_commit_w(bar(B_S_FULL + 0));
      }
      bool o_in = false;  // dO(i) seen in the previous step's joint test
      for (int it = 0; ok && it < n_it; ++it) {
        const bool next = it + 1 < n_it;
        const int so = it % OST, uo = it / OST;
        // dP(i) into Y (d = 128: once the drain has read dQ^T(i - 1) there): it does
        // not wait for P(i), so dS(i) can start as soon as it lands
        if (!C::DQ_OWN) {
          if (!(ok = wait_all(B_O_FULL + so, uo, 0x14))) break;
          if (it > 0 && !(ok = wait_all(B_DQ_FREE, it - 1, 0x17))) break;
        } else if (!o_in && !(ok = wait_all(B_O_FULL + so, uo, 0x14))) {
          break;
        }
        tc_fence_after();
        mma_xyT(C::TM_Y, sV, sDO(it));
        mma_commit_w(bar(B_DP_FULL));
        // dV(i): P^T from X, dO(i); at d = 64 Q(i + 1) is tested with P(i) (at d = 128,
        // with two Q stages, it may still be landing, and that timed the same)
        const int sq1 = (it + 1) % QST, uq1 = (it + 1) / QST;
        const bool q_in = C::DQ_OWN && next && all_done2(B_P_FULL, it, B_Q_FULL + sq1, uq1);
        if (!q_in && !(ok = wait_all(B_P_FULL, it, 0x13))) break;
        tc_fence_after();
        mma_dv(sDO(it), it > 0);
        mma_commit_w(bar(B_O_EMPTY + so));  // dV is the last reader of dO(i)
        // S(i + 1) into X: dV(i), earlier in the pipe, was the last reader of P^T(i)
        if (next) {
          if (!q_in && !(ok = wait_all(B_Q_FULL + sq1, uq1, 0x11))) break;
          tc_fence_after();
          mma_xyT(C::TM_X, sK, sQ(it + 1));
          mma_commit_w(bar(B_S_FULL + sq1));
        }
        // dK(i) over the queries of the compute warps' first pass while they do
        // the second, then the rest of dK(i) and dQ(i) once dS^T(i) is complete
        if (!(ok = wait_all(B_DS_HALF, it, 0x19))) break;
        tc_fence_after();
        mma_dk(sQ(it), it > 0, 0);
        // d = 64: dS(i) complete and the drain has read dQ(i - 1) out of Z, tested
        // together with dO(i + 1) for the next dP
        const int so1 = (it + 1) % OST, uo1 = (it + 1) / OST;
        o_in = false;
        if (C::DQ_OWN && next && it > 0) {
          o_in = all_done3(B_DS_FULL, it, B_DQ_FREE, it - 1, B_O_FULL + so1, uo1);
          if (!o_in &&
              !(ok = wait_all(B_DS_FULL, it, 0x15) && wait_all(B_DQ_FREE, it - 1, 0x17)))
            break;
        } else if (C::DQ_OWN && next) {
          o_in = all_done2(B_DS_FULL, it, B_O_FULL + so1, uo1);
          if (!o_in && !(ok = wait_all(B_DS_FULL, it, 0x15))) break;
        } else {
          if (!(ok = wait_all(B_DS_FULL, it, 0x15))) break;
          if (C::DQ_OWN && it > 0 && !(ok = wait_all(B_DQ_FREE, it - 1, 0x17))) break;
        }
        tc_fence_after();
        mma_dk(sQ(it), true, 1);
        mma_commit_w(bar(B_Q_EMPTY + it % QST));  // dK is the last reader of Q(i)
        mma_dq();
        mma_commit_w(bar(B_DQ_FULL));
      }
      // drain: every MMA issued by this warp has finished before TMEM is freed
      mma_commit_w(bar(B_MMA_DONE));
      mbar_drain(bar(B_MMA_DONE), 0, wctx, ERR_SITE_BWD | 0x18);
      __syncwarp();
    }
  } else if (warp >= 8) {
    // ---------------------------------------------------------------- dQ drain
    regs_inc<C::REG_DRAIN>();
    const int t = threadIdx.x & 127;  // TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t sdq = sbase + C::OFF_DQ;
    if constexpr (C::DQ_QL) {
      // thread t holds query row t of dQ (TMEM lane t, D columns); warp wd adds rows
      // [32 wd, 32 wd + 32) on its own
      const int wd = warp & 3;
      for (int it = 0; it < n_it; ++it) {
        const int q0 = (i_start + it) * BQ;
        mbar_wait(bar(B_DQ_FULL), it & 1, wctx, ERR_SITE_BWD | 0x31);
        tc_fence_after();
        uint32_t r[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_off + C::TM_Z + 32 * c, r[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) reg_fence32(r[c]);
        tc_fence_before();
        mbar_arrive(bar(B_DQ_FREE));
        const uint32_t buf = sdq + (uint32_t)((2 * wd + (it & 1)) * C::DQ_WBUF);
        // this buffer's reduces, two steps ago, are done reading it
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < D / 32; ++c)  // 32 columns: one 128-byte-swizzled box
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(buf + c * 4096 + lane * 128 + ((j ^ (lane & 7)) << 4), r[c][4 * j],
                         r[c][4 * j + 1], r[c][4 * j + 2], r[c][4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // rows past the sequence end belong to the next one (or lie past the
          // tensor, where TMA clips them): their partial is exactly zero, since
          // their LSE is +inf, so adding it changes nothing
#pragma unroll
          for (int c = 0; c < D / 32; ++c)
            tma_reduce_add_3d(&tm_dq, buf + c * 4096, 32 * c, row0 + q0 + 32 * wd, bh);
          bulk_commit();
        }
      }
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
    } else {
      int nbuf = 0;  // chunks staged so far: the buffer of the next one is nbuf % NDQ
      for (int it = 0; it < n_it; ++it) {
        const int q0 = (i_start + it) * BQ;
        mbar_wait(bar(B_DQ_FULL), it & 1, wctx, ERR_SITE_BWD | 0x31);
        tc_fence_after();
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + C::TM_Z + 32 * c, r[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence32(r[c]);
        tc_fence_before();
        mbar_arrive(bar(B_DQ_FREE));
        // lanes are d (lanes >= d are padding), columns are queries: stage 16 query
        // rows at a time in shared memory and add them with one bulk tensor reduce
        constexpr int RPC = C::RPC, CPS = BQ / RPC;  // rows per reduce, reduces per step
#pragma unroll
        for (int h = 0; h < CPS; ++h, ++nbuf) {  // RPC query rows per reduce
          const uint32_t buf = sdq + (uint32_t)(nbuf % C::NDQ) * (RPC * D * 4);
          // the reduce that last read this buffer, NDQ chunks ago, is done reading it
          if (t == 0) bulk_wait_read<C::NDQ - 1>();
          named_bar_sync(2, 128);
          if (t < D) {
#pragma unroll
            for (int c = 0; c < RPC; ++c) {
              const int q = h * RPC + c;  // query column of the dQ^T tile
              asm volatile("st.shared.b32 [%0], %1;" ::"r"(buf + (uint32_t)(c * D + t) * 4u),
                           "r"(r[q >> 5][q & 31])
                           : "memory");
            }
          }
          fence_proxy_async_smem();
          named_bar_sync(2, 128);
          if (t == 0) {  // (rows past the sequence end add zero, as above)
            tma_reduce_add_3d(&tm_dq, buf, 0, row0 + q0 + RPC * h, bh);
            bulk_commit();
          }
        }
      }
      if (t == 0) bulk_wait_read_all();  // the CTA's exit needs only the shared-memory reads done
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------------- compute (warps 0-7)
    // Warpgroup w owns queries [64w, 64w + 64) of every step; thread t owns key
    // row t (TMEM lane t).  Per step i it forms dS^T(i) (as soon as dP^T(i) is
    // in Y) and then P^T(i + 1) (S^T(i + 1) is computed meanwhile), keeping the
    // bf16 P^T in registers for the next dS.
    const int w = warp >> 2;
    const int t = threadIdx.x & 127;
    const int ctid = threadIdx.x;  // 0..255
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int kr = k0 + t;
    const float sl2 = p.scale_log2;
    const uint32_t tX = tmem + lane_off + C::TM_X + 64u * w;  // S^T columns of this half
    const uint32_t tY = tmem + lane_off + C::TM_Y + 64u * w;  // dP^T columns of this half
    uint32_t pk[32];  // P^T of the current step: bf16 pairs of queries (2e, 2e + 1)

    // P^T = exp2(S^T * scale * log2e - LSE2), masked; bf16 into X (over the S^T
    // columns this thread has read) and into pk
    auto form_p = [&](int it) {
      const int st = it % QST;
      const int q0 = (i_start + it) * BQ;
      const float4* nlse2 =
          reinterpret_cast<const float4*>(smem + C::OFF_STAT + st * 2 * BQ * 4) + 16 * w;
      // key kr sees query q iff kr < N and (not causal or kr <= q); queries
      // past N already have LSE2 = +inf.  Only blocks that cross the diagonal
      // or hold keys past N need the element mask.
      const int qh = q0 + 64 * w;
      const bool need_mask = (p.causal && k0 + C::BK - 1 > qh) || (k0 + C::BK > N);
      int lo = 0;
      if (kr >= N) lo = 64;
      else if (p.causal) lo = min(max(kr - qh, 0), 64);
      // S^T(it) in X and this step's LSE2 in shared memory
      mbar_wait(bar(B_S_FULL + st), (it / QST) & 1, wctx, ERR_SITE_BWD | 0x22);
      tc_fence_after();
      uint32_t u[2][32];
      tmem_ld32(tX, u[0]);
      tmem_ld32(tX + 32, u[1]);
      tmem_wait_ld();
      reg_fence32(u[0]);
      reg_fence32(u[1]);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float pv[32];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 l4 = nlse2[(c * 32 + i) / 4];
          fma_x2(__uint_as_float(u[c][i]), __uint_as_float(u[c][i + 1]), sl2, l4.x, l4.y, pv[i],
                 pv[i + 1]);
          fma_x2(__uint_as_float(u[c][i + 2]), __uint_as_float(u[c][i + 3]), sl2, l4.z, l4.w,
                 pv[i + 2], pv[i + 3]);
#pragma unroll
          for (int j = 0; j < 4; ++j) pv[i + j] = ex2(pv[i + j]);
        }
        if (need_mask) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i < lo) pv[i] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[c * 16 + e] = pack_bf16x2(pv[2 * e], pv[2 * e + 1]);
      }
      tmem_st32(tX, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_P_FULL));
    };

    if (n_it > 0) form_p(0);
    for (int it = 0; it < n_it; ++it) {
      // ---- dS^T = P^T o (dP^T - D) -> bf16 -> shared memory (K-major for dK,
      // MN-major for dQ); this warpgroup writes the 64-query half w
      const int st = it % QST;
      const float4* dlt =
          reinterpret_cast<const float4*>(smem + C::OFF_STAT + st * 2 * BQ * 4 + BQ * 4) + 16 * w;
      mbar_wait(bar(B_DP_FULL), it & 1, wctx, ERR_SITE_BWD | 0x26);
      tc_fence_after();
      uint32_t u[2][32];
      tmem_ld32(tY, u[0]);
      tmem_ld32(tY + 32, u[1]);
      tmem_wait_ld();
      reg_fence32(u[0]);
      reg_fence32(u[1]);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float ds[32];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const uint32_t p01 = pk[c * 16 + i / 2], p23 = pk[c * 16 + i / 2 + 1];
          const float4 d4 = dlt[(c * 32 + i) / 4];
          mul_sub_x2(__uint_as_float(p01 << 16), __uint_as_float(p01 & 0xffff0000u),
                     __uint_as_float(u[c][i]), __uint_as_float(u[c][i + 1]), d4.x, d4.y, ds[i],
                     ds[i + 1]);
          mul_sub_x2(__uint_as_float(p23 << 16), __uint_as_float(p23 & 0xffff0000u),
                     __uint_as_float(u[c][i + 2]), __uint_as_float(u[c][i + 3]), d4.z, d4.w,
                     ds[i + 2], ds[i + 3]);
        }
        uint32_t dpk[16];  // bf16 pairs of queries (2e, 2e + 1)
#pragma unroll
        for (int e = 0; e < 16; ++e) dpk[e] = pack_bf16x2(ds[2 * e], ds[2 * e + 1]);
        // for dK: into TMEM over the dP^T columns already read (Y + 64w + 16c)
        tmem_st16(tY + 16 * c, dpk);
        // for dQ: into shared memory, MN-major
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // four 16-byte chunks of 8 queries
          const int chunk = c * 4 + e;
          st_shared_v4(sbase + C::OFF_DS + w * C::HALF + t * 128 + ((chunk ^ (t & 7)) << 4),
                       dpk[4 * e], dpk[4 * e + 1], dpk[4 * e + 2], dpk[4 * e + 3]);
        }
        if (c == 0) {  // the first pass's dS^T is in TMEM: dK can start on it
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(B_DS_HALF));
        }
      }
      mbar_arrive(bar(B_Q_EMPTY + st));  // LSE2 and D of this stage are no longer read
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();  // the dP^T reads and dS^T writes of Y precede dQ^T written into it
      mbar_arrive(bar(B_DS_FULL));
      if (it + 1 < n_it) form_p(it + 1);
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
          st_shared_v4(dst + half * C::HALF + t * 128 + ((chunk ^ (t & 7)) << 4),
                       pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                       pack_bf16x2(f[6], f[7]));
        }
      }
    }
    if (VARLEN && k0 + C::BK > N) {
      // the block runs past the end of the sequence, into the next one's rows:
      // thread (which, t) writes row t of dK or dV if it belongs to the sequence
      named_bar_sync(1, 256);
      const int which = ctid >> 7;
      if (k0 + t < N) {
        const uint32_t src = sbase + (which == 0 ? C::OFF_K : C::OFF_V);
        uint4* dst = reinterpret_cast<uint4*>((which == 0 ? p.dk : p.dv) +
                                              ((size_t)bh * p.vl.T + row0 + k0 + t) * D);
#pragma unroll
        for (int c16 = 0; c16 < D / 8; ++c16) {
          const int half = c16 >> 3, chunk = c16 & 7;
          uint4 v4;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(v4.x), "=r"(v4.y), "=r"(v4.z), "=r"(v4.w)
                       : "r"(src + half * C::HALF + t * 128 + ((chunk ^ (t & 7)) << 4)));
          dst[c16] = v4;
        }
      }
    } else {
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      if (ctid == 0) {
        for (int h = 0; h < D / 64; ++h) {
          tma_store_3d(&tm_dk, sbase + C::OFF_K + h * C::HALF, h * 64, row0 + k0, bh);
          tma_store_3d(&tm_dv, sbase + C::OFF_V + h * C::HALF, h * 64, row0 + k0, bh);
        }
        bulk_commit();
        bulk_wait_read_all();
      }
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

template <int D, bool VARLEN>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                   const CUtensorMap& tdq, const BwdParams& p, cudaStream_t stream) {
  using C = Bwd<D>;
  static_assert(C::SMEM <= 232448, "shared memory budget");
  static_assert(C::TM_Y + 128 <= 512 && C::TM_Z + 128 <= 512, "TMEM budget");
  static unsigned long long prepared[64];
  cudaError_t e = prepare_once(prepared, [] {
    cudaError_t r = cudaFuncSetAttribute(fattn_bwd_kernel<D, VARLEN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (r != cudaSuccess) return r;
    // the setmaxnreg split hands out exactly the launch's registers (128 per thread);
    // with fewer at launch an increase would never be granted
    cudaFuncAttributes fa;
    r = cudaFuncGetAttributes(&fa, fattn_bwd_kernel<D, VARLEN>);
    if (r != cudaSuccess) return r;
    return fa.numRegs == 128 ? cudaSuccess : cudaErrorInvalidConfiguration;
  });
  if (e != cudaSuccess) return e;
  const long long n_kb = (p.N + C::BK - 1) / C::BK;
  const long long blocks = n_kb * (VARLEN ? (long long)p.vl.B * p.vl.H : p.BH);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (blocks == 0) return cudaSuccess;
  fattn_bwd_kernel<D, VARLEN><<<(unsigned)blocks, C::THREADS, C::SMEM, stream>>>(
      tq, tk, tv, tdo, tdk, tdv, tdq, p);
  return cudaGetLastError();
}

}  // namespace

DqBox bwd_dq_box(int d) {
  if (Bwd<64>::DQ_QL && d == 64) return DqBox{32, 32, true};
  return DqBox{d, FATTN_DQ_ROWS, false};
}

cudaError_t launch_bwd_main(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const CUtensorMap& tdq_acc, const BwdParams& p, cudaStream_t stream) {
  const bool vl = p.vl.cu_seqlens != nullptr;
  if (d == 128) return vl ? launch<128, true>(tq, tk, tv, tdo, tdk, tdv, tdq_acc, p, stream)
                          : launch<128, false>(tq, tk, tv, tdo, tdk, tdv, tdq_acc, p, stream);
  if (d == 64) return vl ? launch<64, true>(tq, tk, tv, tdo, tdk, tdv, tdq_acc, p, stream)
                         : launch<64, false>(tq, tk, tv, tdo, tdk, tdv, tdq_acc, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fattn
