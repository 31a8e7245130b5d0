// fwd.cu -- FlashAttention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// One CTA owns 256 query rows of one (batch, head): two 128-row subtiles
// Q_0, Q_1 (SUB = 2; at d = 64 a CTA may own one, see below), each running
// the single-query recurrence of "tm_flash_attention_math"
// ("The block-wise update, and the full algorithm") for all of its rows at
// once.  K/V tiles of 128 keys stream through a ring of shared-memory slots
// filled by TMA; the score tile S = Q K^T lives only in TMEM ("A score tile is
// temporary state", page "FlashAttention tiles exact softmax without
// materializing the score matrix").
//
// Warp roles (384 threads):
//   warps 0-3  softmax for Q_0, warps 4-7 softmax for Q_1: thread t owns query
//              row t, which is TMEM lane t, so the row max and row sum need no
//              shuffles.  They also rescale their O accumulator by alpha when
//              the reference maximum moves, and run the epilogue O = o~ / l,
//              LSE = m + ln l.
//   warp 8     issues every tcgen05.mma and commit: the whole warp runs the
//              loop (so descriptor arithmetic stays warp-uniform) and
//              elect.sync picks the one lane that issues.
//   warp 9     one thread issues every TMA load.
//   warps 10-11 idle: with them the CTA is three whole warpgroups, so setmaxnreg
//              can move registers from the MMA/TMA warpgroup (48 each) to the
//              softmax warpgroups (224 each); with the compiler's 168 the
//              softmax's packed f32x2 arithmetic spilled.
//
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 after it.
// At d = 128, P_s (bf16, two per 32-bit column) overwrites the first 64 columns
// of S_s once the softmax has read S_s, and feeds O_s += P_s V as the TMEM A
// operand, so P never touches shared memory.  At d = 64, P_0 and P_1 have 64
// columns each after O_1, so S_s = Q_s K_{j+1}^T is issued as soon as the
// softmax has S_s(j) in registers (B_S_READ) and runs while it forms P_s(j).  The softmax releases P_s in two halves of
// 64 keys, and the MMA thread issues the half of O_s += P_s V_j over the first
// half while the softmax forms the second; per subtile it issues all of
// O_s += P_s V_j before S_s = Q_s K_{j+1}^T (the pipe runs them in order).
// Shared memory: Q_0, Q_1 | K/V ring.
//
// SUB = 1 (d = 64 only): one 128-row subtile per CTA, 256 threads (softmax
// warps 0-3, MMA warp 4, TMA warp 5, warps 6-7 idle), 256 TMEM columns (S, O,
// P) and a 5-slot ring, so that two CTAs share an SM.  Their barrier chains
// then run independently, and a short grid's last wave is split finer.  Each
// CTA streams its own K/V, twice the L2 traffic of SUB = 2, so the launcher
// takes it only for grids of a few waves.
// setmaxnreg regions may not call functions: inline the wait's slow path
#define FATTN_INLINE_WAIT_SLOW_PATH
#include "common.cuh"
#include "ptx.cuh"

// Built with FATTN_FWD_DEC64=0 the d = 64 kernel keeps P over S as at d = 128
// (kept buildable for A/B timing).
#ifndef FATTN_FWD_DEC64
#define FATTN_FWD_DEC64 1
#endif

namespace fattn {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
// Largest exp2 argument the softmax lets through before it moves its reference.
constexpr float kRescaleLog2 = 8.f;


template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Two-lane fp32 arithmetic: one instruction for a pair of elements, each lane
// rounded exactly as the scalar instruction would be.
// (r0, r1) = (a0, a1) * b + (c, c)
__device__ __forceinline__ void fma_x2(float a0, float a1, float b, float c, float& r0, float& r1) {
  asm("{\n\t.reg .b64 a, b, c, r;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %4};\n\t"
      "mov.b64 c, {%5, %5};\n\t"
      "fma.rn.f32x2 r, a, b, c;\n\t"
      "mov.b64 {%0, %1}, r;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (s0, s1) += (a0, a1)
__device__ __forceinline__ void add_x2(float& s0, float& s1, float a0, float a1) {
  asm("{\n\t.reg .b64 s, a;\n\t"
      "mov.b64 s, {%0, %1};\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "add.rn.f32x2 s, s, a;\n\t"
      "mov.b64 {%0, %1}, s;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}

template <int D, int SUB_>
struct Fwd {
  static constexpr int SUB = SUB_;                // 128-row Q subtiles per CTA
  static_assert(SUB == 2 || (SUB == 1 && D == 64), "one subtile per CTA at d = 64 only");
  static constexpr int ROWS = 128 * SUB;          // query rows per CTA
  static constexpr int MIN_CTAS = SUB == 1 ? 2 : 1;  // CTAs sharing an SM
  static constexpr int BM = 128;                  // rows per Q subtile
  static constexpr int BN = 128;                  // keys per K/V tile
  static constexpr int HALF = BM * 128;           // one 64-column, 128-row swizzled half (bytes)
  static constexpr int TILE = BM * D * 2;         // Q, K, V or O tile (bf16)
  static constexpr int STAGES = D == 128 ? 5 : (SUB == 1 ? 5 : 8);  // K/V ring slots
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + SUB * TILE;
  static constexpr int OFF_BAR = OFF_KV + STAGES * TILE;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // barriers + alignment slack
  // SUB softmax warpgroups and one control warpgroup (MMA warp, TMA warp, two idle)
  static constexpr int THREADS = 128 * (SUB + 1);
  static constexpr int W_MMA = 4 * SUB, W_TMA = 4 * SUB + 1;
  // registers per thread after setmaxnreg; the launch holds THREADS x REG_LAUNCH
  static constexpr int REG_LAUNCH = SUB == 1 ? 128 : 168;
  static constexpr int REG_SOFTMAX = SUB == 1 ? 208 : 224, REG_CTRL = 48;
  static_assert((SUB * REG_SOFTMAX + REG_CTRL) * 128 <= THREADS * REG_LAUNCH, "register split");
  static_assert(MIN_CTAS * (SMEM + 1024) <= 233472, "shared memory of the CTAs sharing an SM");
  // the registers admit at most MIN_CTAS CTAs per SM, so their TMEM allocations never wait
  static_assert((MIN_CTAS + 1) * THREADS * REG_LAUNCH > 65536, "a third CTA would wait for TMEM");
  static constexpr int TMEM_COLS = SUB == 1 ? 256 : 512;
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_O = 128 * SUB;
  // d = 64 leaves 128 TMEM columns free: P_s gets a region of its own there
  // (64 columns of bf16 pairs per subtile), so S_s = Q_s K_{j+1}^T can be
  // issued as soon as the softmax has read S_s(j) into registers, instead of
  // after O_s += P_s V_j; the softmax then never waits on its own subtile's MMAs
  static constexpr bool DEC = D == 64 && FATTN_FWD_DEC64 != 0;
  static constexpr uint32_t TM_P = DEC ? TM_O + SUB * D : TM_S;  // P_s at TM_P + (DEC ? 64 : 128) s
  static constexpr uint32_t P_STRIDE = DEC ? 64 : 128;
  static_assert(!DEC || TM_P + SUB * 64 <= TMEM_COLS, "TMEM budget");
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BN, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, false, true);
};

// Barrier slots (8 bytes each) inside the OFF_BAR block.
enum {
  B_Q = 0,
  B_S_FULL = 1,   // [2] MMA -> softmax: S_s ready in TMEM (and every earlier MMA done)
  B_P_FULL = 3,   // [2] softmax -> MMA: P_s in TMEM (both halves)
  B_PV_DONE = 5,  // [2] MMA -> epilogue: O_s += P_s V finished
  B_P_HALF = 7,   // [2] softmax -> MMA: keys 0-63 of P_s in TMEM and O_s rescaled
  B_MMA_DONE = 9,
  B_S_READ = 10,  // [2] softmax -> MMA (d = 64): S_s is in registers, its TMEM may be rewritten
  B_KV_FULL = 12,  // [STAGES], then kv_empty [STAGES]
};
// the barriers, the TMEM address slot and the abort flag share 256 bytes
static_assert(8 * (B_KV_FULL + 2 * Fwd<64, 2>::STAGES) + 8 <= 256, "barrier block");
static_assert(8 * (B_KV_FULL + 2 * Fwd<64, 1>::STAGES) + 8 <= 256, "barrier block");
static_assert(8 * (B_KV_FULL + 2 * Fwd<128, 2>::STAGES) + 8 <= 256, "barrier block");

// VARLEN: the CTA's sequence comes from p.vl.cu_seqlens (packed head-major
// rows); otherwise the dense [B, H, N, d] layout.  SPLIT (dense only): the CTA
// covers one range of key tiles and writes its normalised partial O and LSE
// (fp32) for the merge kernel; queries are the last p.Nq positions.
template <int D, int SUB, bool VARLEN, bool SPLIT>
__global__ void __launch_bounds__(Fwd<D, SUB>::THREADS, Fwd<D, SUB>::MIN_CTAS)
    fattn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  using C = Fwd<D, SUB>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // SPLIT: blockIdx = (query block, unit, split) with the split fastest
  const int split = SPLIT ? (int)(blockIdx.x % (unsigned)p.n_splits) : 0;
  const unsigned bidx = SPLIT ? blockIdx.x / (unsigned)p.n_splits : blockIdx.x;
  const int n_qb = ((SPLIT ? p.Nq : p.N) + C::ROWS - 1) / C::ROWS;  // p.N: the (longest) sequence length
  // heaviest (last) query blocks first
  // dense: query-block-major within groups of heads; varlen:
  // one (sequence, head) unit after another, so the CTAs in flight share their
  // unit's K/V in L2 (a unit-spread order streams each CTA's K/V from DRAM)
  const int units = VARLEN ? p.vl.B * p.vl.H : p.BH;
  int qb, unit;
  if (VARLEN) {
    qb = n_qb - 1 - (int)(bidx % (unsigned)n_qb);
    unit = (int)(bidx / (unsigned)n_qb);
  } else {  // heads in groups whose K/V stay in L2 (p.group)
    int blk;
    grouped_order(bidx, units, n_qb, p.group, &blk, &unit);
    qb = n_qb - 1 - blk;
  }
  SeqView seq;
  if constexpr (VARLEN) {
    if (!seq_view(p.vl, p.N, unit / p.vl.H, unit % p.vl.H, unit, p.N, &seq)) {
      if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0u, (unsigned)(ERR_SITE_FWD | 0x40));
      return;
    }
    if (qb * C::ROWS >= seq.N) return;  // this sequence is shorter: nothing to do
  } else {
    seq = SeqView{p.N, 0, unit, (long long)unit * p.N};
  }
  const int N = seq.N;         // keys
  const int Nq = SPLIT ? p.Nq : N;  // queries
  const int off = N - Nq;      // query i sits at key position i + off (0 unless SPLIT)
  const int bh = seq.z;        // TMA z coordinate
  const int row0 = seq.row0;   // first row of the sequence in the tensor
  const int n_kv_total = (N + C::BN - 1) / C::BN;
  // key tiles [jlo, jhi) belong to this CTA (all of them unless SPLIT)
  const int jlo = SPLIT ? split * p.tiles_per_split : 0;
  const int jhi = SPLIT ? jlo + p.tiles_per_split : 0x7fffffff;

  // rows [r0_s, r0_s + 128) of subtile s see key tiles [jlo, jlo + nt_s)
  auto tiles_for = [&](int r0) {
    if (r0 >= Nq) return 0;
    const int last_key = p.causal ? min(r0 + C::BM - 1 + off, N - 1) : N - 1;
    return max(0, min(last_key / C::BN + 1, jhi) - jlo);
  };
  // with one subtile, subtile 1 starts past every sequence and sees no tiles
  const int r0_0 = qb * C::ROWS, r0_1 = SUB == 2 ? r0_0 + 128 : (1 << 30);
  const int nt0 = tiles_for(r0_0), nt1 = tiles_for(r0_1);
  const int r0[2] = {r0_0, r0_1};
  const int nt[2] = {nt0, nt1};
  const int n_max = max(nt0, nt1);

  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  const uint32_t kv_full0 = bar(B_KV_FULL), kv_empty0 = bar(B_KV_FULL + ST);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * (B_KV_FULL + 2 * ST));
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wctx{abort_flag, p.err};

  // The TMA thread initialises the barriers and issues Q and the first ST K/V
  // loads (their slots are empty) before the CTA-wide sync, so that the load
  // latency overlaps the TMEM allocation and the sync.
  const bool tma_thread = warp == C::W_TMA && lane == 0;
  const int n_loads = 2 * n_max;
  const int n_pre = min(ST, n_loads);
  auto load_kv = [&](int i) {
    const int slot = i % ST;
    const uint32_t dst = sbase + C::OFF_KV + slot * C::TILE;
    const CUtensorMap* m = (i & 1) ? &tm_v : &tm_k;
    mbar_arrive_expect_tx(kv_full0 + 8u * slot, C::TILE);
    for (int h = 0; h < D / 64; ++h)
      tma_load_3d(dst + h * C::HALF, m, kv_full0 + 8u * slot, h * 64,
                  row0 + (jlo + (i >> 1)) * C::BN, bh);
  };
  if (tma_thread) {
    mbar_init(bar(B_Q), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_S_FULL + s), 1);
      mbar_init(bar(B_P_FULL + s), 128);
      mbar_init(bar(B_P_HALF + s), 128);
      mbar_init(bar(B_PV_DONE + s), 1);
      mbar_init(bar(B_S_READ + s), 128);
    }
    mbar_init(bar(B_MMA_DONE), 1);
    for (int i = 0; i < ST; ++i) {
      mbar_init(kv_full0 + 8u * i, 1);
      mbar_init(kv_empty0 + 8u * i, 1);
    }
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    const uint32_t q_bytes = (uint32_t)((nt0 > 0) + (nt1 > 0)) * C::TILE;
    mbar_arrive_expect_tx(bar(B_Q), q_bytes);
#pragma unroll
    for (int s = 0; s < 2; ++s)
      if (nt[s] > 0)
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(sbase + C::OFF_Q + s * C::TILE + h * C::HALF, &tm_q, bar(B_Q), h * 64,
                      row0 + r0[s], bh);
    for (int i = 0; i < n_pre; ++i) load_kv(i);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp > C::W_TMA) {
    regs_dec<C::REG_CTRL>();  // idle
  } else if (warp == C::W_TMA) {
    regs_dec<C::REG_CTRL>();
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int issued = n_pre;  // Q and loads [0, n_pre) went out before the sync
      for (int i = n_pre; i < n_loads; ++i) {
        const int slot = i % ST, use = i / ST;
        // a slot is refilled only after the MMAs that read it completed; when
        // the CTA is aborting nothing more is issued
        if (!mbar_wait(kv_empty0 + 8u * slot, (use - 1) & 1, wctx, ERR_SITE_FWD | 0x01)) break;
        load_kv(i);
        issued = i + 1;
      }
      // drain: at most one load per slot can still be landing, the latest one
      for (int i = max(0, issued - ST); i < issued; ++i)
        mbar_drain(kv_full0 + 8u * (i % ST), (i / ST) & 1, wctx, ERR_SITE_FWD | 0x02);
      mbar_drain(bar(B_Q), 0, wctx, ERR_SITE_FWD | 0x03);
    }
    __syncwarp();
  } else if (warp == C::W_MMA) {
    regs_dec<C::REG_CTRL>();
    // ---------------------------------------------------------------- MMA issuer (whole warp)
    {
      auto kv_wait = [&](int i) {
        return __all_sync(0xffffffffu, mbar_wait(kv_full0 + 8u * (i % ST), (i / ST) & 1, wctx, ERR_SITE_FWD | 0x11));
      };
      auto issue_s = [&](int s, int j) {  // S_s = Q_s K_j^T
        const uint32_t a = sbase + C::OFF_Q + s * C::TILE;
        const uint32_t b = sbase + C::OFF_KV + ((2 * j) % ST) * C::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::HALF + (kk & 3) * 32;
          mma_bf16_ss_w(tmem + C::TM_S + s * 128, sdesc_sw128(a + off, 16, 1024),
                      sdesc_sw128(b + off, 16, 1024), C::IDESC_S, kk > 0);
        }
        mma_commit_w(bar(B_S_FULL + s));
      };
      // O_s += P_s V_j over keys [64 half, 64 half + 64), P_s from TMEM
      auto issue_pv = [&](int s, int j, int half) {
        const uint32_t b = sbase + C::OFF_KV + ((2 * j + 1) % ST) * C::TILE;
#pragma unroll
        for (int k = 0; k < C::BN / 32; ++k) {  // 16 keys = 8 packed TMEM columns per step
          const int kk = half * (C::BN / 32) + k;
          mma_bf16_ts_w(tmem + C::TM_O + s * D, tmem + C::TM_P + s * C::P_STRIDE + kk * 8,
                      sdesc_sw128(b + kk * 16 * 128, C::HALF, 1024), C::IDESC_PV,
                      (j > 0 || kk > 0));
        }
        if (half == 1) mma_commit_w(bar(B_PV_DONE + s));
      };
      // any failed wait means the CTA is aborting: issue nothing more
      bool ok = __all_sync(0xffffffffu, mbar_wait(bar(B_Q), 0, wctx, ERR_SITE_FWD | 0x12));
      if (ok && n_max > 0) {
        ok = kv_wait(0);
        if (ok) {
          tc_fence_after();
          if (nt0 > 0) issue_s(0, 0);
          if (nt1 > 0) issue_s(1, 0);
          mma_commit_w(kv_empty0 + 8u * 0);
        }
      }
      for (int j = 0; C::DEC && ok && j < n_max; ++j) {
        // S_s(j + 1) once the softmax holds S_s(j) in registers; O_s += P_s V_j
        // once P_s(j) is in its own region.  The pipe runs them in issue order.
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (ok && j + 1 < nt[s]) {
            ok = kv_wait(2 * (j + 1)) &&
                 __all_sync(0xffffffffu, mbar_wait(bar(B_S_READ + s), j & 1, wctx, ERR_SITE_FWD | 0x19));
            if (ok) {
              tc_fence_after();
              issue_s(s, j + 1);
            }
          }
        }
        if (!ok) break;
        if (j + 1 < n_max) mma_commit_w(kv_empty0 + 8u * ((2 * (j + 1)) % ST));
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (ok && j < nt[s]) {
            ok = kv_wait(2 * j + 1) &&
                 __all_sync(0xffffffffu, mbar_wait(bar(B_P_HALF + s), j & 1, wctx, ERR_SITE_FWD | 0x18));
            if (ok) {
              tc_fence_after();
              issue_pv(s, j, 0);
              ok = __all_sync(0xffffffffu, mbar_wait(bar(B_P_FULL + s), j & 1, wctx, ERR_SITE_FWD | 0x14));
            }
            if (ok) {
              tc_fence_after();
              issue_pv(s, j, 1);
            }
          }
        }
        if (!ok) break;
        mma_commit_w(kv_empty0 + 8u * ((2 * j + 1) % ST));
      }
      // each K/V tile is waited for once per iteration, not once per subtile: a
      // satisfied wait still costs this warp tens of cycles, during which the
      // tensor pipe may run dry
      for (int j = 0; !C::DEC && ok && j < n_max; ++j) {
        const bool next = j + 1 < n_max;
        bool k_next = false;      // K_{j+1} waited for
        ok = kv_wait(2 * j + 1);  // V_j: some subtile has tile j
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const int nts = s ? nt1 : nt0;
          if (ok && j < nts) {
            // the first half of PV runs while the softmax forms the second half of P
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_P_HALF + s), j & 1, wctx, ERR_SITE_FWD | 0x18));
            if (ok) {
              tc_fence_after();
              issue_pv(s, j, 0);
              ok = __all_sync(0xffffffffu, mbar_wait(bar(B_P_FULL + s), j & 1, wctx, ERR_SITE_FWD | 0x14));
            }
            if (ok) {
              tc_fence_after();
              issue_pv(s, j, 1);
            }
          }
          if (ok && j + 1 < nts) {  // after the PV above: S_s is overwritten in pipe order
            if (!k_next) {
              ok = kv_wait(2 * (j + 1));
              k_next = true;
            }
            if (ok) issue_s(s, j + 1);
          }
        }
        if (!ok) break;
        if (next) mma_commit_w(kv_empty0 + 8u * ((2 * (j + 1)) % ST));
        mma_commit_w(kv_empty0 + 8u * ((2 * j + 1) % ST));
      }
      // drain: every MMA issued by this thread has finished before TMEM is freed
      mma_commit_w(bar(B_MMA_DONE));
      mbar_drain(bar(B_MMA_DONE), 0, wctx, ERR_SITE_FWD | 0x17);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax (warps 0-7)
    regs_inc<C::REG_SOFTMAX>();
    const int s = warp >> 2;
    const int t = threadIdx.x & 127;  // row in the subtile == TMEM lane
    const int my_r0 = s ? r0_1 : r0_0;
    const int my_nt = s ? nt1 : nt0;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S + s * 128;
    const uint32_t tO = tmem + lane_off + C::TM_O + s * D;
    const uint32_t tP = tmem + lane_off + C::TM_P + s * C::P_STRIDE;
    const int row = my_r0 + t;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    unsigned long long n_full = 0, n_masked = 0;

    for (int j = 0; j < my_nt; ++j) {
      // s_full also means every earlier MMA is done; at d = 128 that includes
      // O_s += P_s V_{j-1}, issued before S_s(j).  At d = 64 S_s(j) is issued
      // first, and the softmax waits for PV_DONE before it touches O_s or P_s.
      mbar_wait(bar(B_S_FULL + s), j & 1, wctx, ERR_SITE_FWD | 0x21);
      tc_fence_after();
      uint32_t u[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, u[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence32(u[c]);

      float sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(u[c][i]);
      if (C::DEC) {  // S_s is in registers: its TMEM may take S_s(j + 1)
        tc_fence_before();
        mbar_arrive(bar(B_S_READ + s));
      }

      // masks go in before the block maximum
      const int c0 = (jlo + j) * C::BN;
      const bool need_mask =
          (p.causal && min(c0 + C::BN - 1, N - 1) > my_r0 + off) || (c0 + C::BN > N);
      if (need_mask) {
        int lim = N - c0;
        if (p.causal) lim = min(lim, row + off - c0 + 1);
#pragma unroll
        for (int k = 0; k < 128; ++k)
          if (k >= lim) sv[k] = -INFINITY;
        ++n_masked;
      } else {
        ++n_full;
      }

      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = i == 0 ? m_run : -INFINITY;
#pragma unroll
      for (int k = 0; k < 128; k += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], sv[k + 2 * i], sv[k + 2 * i + 1]);
      const float m_blk = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                fmaxf(mx[6], mx[7]));  // max(m_old, block max)
      // The reference only moves when the block raises it by more than 2^8
      // (in base 2); until then p = exp2(s - m) <= 2^8 and O, l stay in the
      // old reference.  Any reference gives the same O and LSE (the shift
      // invariance of softmax), and skipping small moves skips most rescales
      // of O.  The first block always sets it (m_old = -inf).
      const float m_new = (m_run == -INFINITY || (m_blk - m_run) * sl2 > kRescaleLog2) ? m_blk : m_run;
      const float msc = (m_new == -INFINITY) ? 0.f : m_new * sl2;
      const bool rescale = m_new != m_run;
      // alpha = exp(m_old - m_new): 0 on the first block, exactly 1 when the reference stays
      const float alpha = rescale ? ex2(m_run * sl2 - msc) : 1.f;
      float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // 64 keys -> 32 packed bf16x2 TMEM columns
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 64; k += 4) {
          const int kk = h * 64 + k;
          float p0, p1, p2, p3;
          fma_x2(sv[kk], sv[kk + 1], sl2, -msc, p0, p1);
          fma_x2(sv[kk + 2], sv[kk + 3], sl2, -msc, p2, p3);
          p0 = ex2(p0);
          p1 = ex2(p1);
          p2 = ex2(p2);
          p3 = ex2(p3);
          add_x2(ls0, ls1, p0, p1);
          add_x2(ls2, ls3, p2, p3);
          pk[k / 2] = pack_bf16x2(p0, p1);
          pk[k / 2 + 1] = pack_bf16x2(p2, p3);
        }
        if (C::DEC && h == 0 && j > 0) {
          // O_s += P_s V_{j-1} has finished: P_s's region is free and O_s complete
          mbar_wait(bar(B_PV_DONE + s), (j - 1) & 1, wctx, ERR_SITE_FWD | 0x25);
          tc_fence_after();
        }
        tmem_st32(tP + h * 32, pk);
        if (h == 0) {
          // O_s is rescaled before the first half of PV adds into it (the scores of
          // the first half are no longer needed, which leaves the registers for it)
          if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_wait_ld(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(tO + c * 32, o);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(B_P_HALF + s));
        }
      }
      l_run = l_run * alpha + ((ls0 + ls1) + (ls2 + ls3));
      m_run = m_new;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_P_FULL + s));
    }

    if (SPLIT && my_r0 < Nq) {
      // ------------------------------------------------------------ split epilogue:
      // normalised partial O (fp32) and partial LSE of this key range; a row that
      // saw no key here gets O = 0 and LSE = -inf, which the merge weighs by zero
      const size_t prow = ((size_t)split * p.BH + bh) * Nq + row;
      const bool has = l_run > 0.f;
      const float inv_l = has ? 1.f / l_run : 0.f;
      if (my_nt > 0) {
        mbar_wait(bar(B_PV_DONE + s), (my_nt - 1) & 1, wctx, ERR_SITE_FWD | 0x24);
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);  // warp-wide: every lane loads, valid rows store
          tmem_wait_ld(o);
          if (row < Nq) {
            float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(o[4 * q4]) * inv_l,
                                    __uint_as_float(o[4 * q4 + 1]) * inv_l,
                                    __uint_as_float(o[4 * q4 + 2]) * inv_l,
                                    __uint_as_float(o[4 * q4 + 3]) * inv_l);
          }
        }
      } else if (row < Nq) {
        float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
        for (int q4 = 0; q4 < D / 4; ++q4) dst[q4] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (row < Nq) p.lse_part[prow] = has ? (m_run * sl2 + lg2(l_run)) * kLn2 : -INFINITY;
    } else if (!SPLIT && my_nt > 0) {
      // ------------------------------------------------------------ epilogue
      mbar_wait(bar(B_PV_DONE + s), (my_nt - 1) & 1, wctx, ERR_SITE_FWD | 0x23);
      tc_fence_after();
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const uint32_t o_base = sbase + C::OFF_Q + s * C::TILE;  // Q_s is no longer read
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld(o);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {  // four 16-byte chunks of 8 columns
          const int col = c * 32 + q4 * 8;
          const int half = col >> 6, chunk = (col & 63) >> 3;
          const uint32_t addr = o_base + half * C::HALF + t * 128 + ((chunk ^ (t & 7)) << 4);
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[q4 * 8 + e]) * inv_l;
          st_shared_v4(addr, pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                       pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
        }
      }
      if (VARLEN && my_r0 + C::BM > N) {
        // the tile runs past the end of the sequence, into the next one's rows:
        // each thread writes its own row if it belongs to the sequence
        if (row < N) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)bh * p.vl.T + row0 + row) * D);
#pragma unroll
          for (int c16 = 0; c16 < D / 8; ++c16) {
            const int half = c16 >> 3, chunk = c16 & 7;
            uint4 v4;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v4.x), "=r"(v4.y), "=r"(v4.z), "=r"(v4.w)
                         : "r"(o_base + half * C::HALF + t * 128 + ((chunk ^ (t & 7)) << 4)));
            dst[c16] = v4;
          }
        }
      } else {
        fence_proxy_async_smem();
        named_bar_sync(1 + s, 128);
        if (t == 0) {
          for (int h = 0; h < D / 64; ++h)
            tma_store_3d(&tm_o, o_base + h * C::HALF, h * 64, row0 + my_r0, bh);
          bulk_commit();
          bulk_wait_read_all();  // the CTA's exit needs only the shared-memory reads done
        }
      }
      if (row < N) p.lse[seq.stat0 + row] = (m_run * sl2 + lg2(l_run)) * kLn2;
      if (p.tiles && t == 0) {
        atomicAdd(p.tiles + 0, n_full);
        atomicAdd(p.tiles + 1, n_masked);
        atomicAdd(p.tiles + 2, (unsigned long long)(p.causal ? n_kv_total - my_nt : 0));
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Query blocks of ROWS rows the grid covers, times the units (and splits).
template <int ROWS, bool VARLEN, bool SPLIT>
long long fwd_blocks(const FwdParams& p) {
  const long long n_qb = ((SPLIT ? p.Nq : p.N) + ROWS - 1) / ROWS;
  return n_qb * (VARLEN ? (long long)p.vl.B * p.vl.H : p.BH) * (SPLIT ? p.n_splits : 1);
}

template <int D, int SUB, bool VARLEN, bool SPLIT>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   const CUtensorMap& to, const FwdParams& p, cudaStream_t stream) {
  using C = Fwd<D, SUB>;
  static_assert(C::SMEM <= 232448, "shared memory budget");
  static_assert(!(VARLEN && SPLIT), "split-KV is dense only");
  static unsigned long long prepared[64];
  cudaError_t e = prepare_once(prepared, [] {
    cudaError_t r = cudaFuncSetAttribute(fattn_fwd_kernel<D, SUB, VARLEN, SPLIT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (r != cudaSuccess) return r;
    // the setmaxnreg split hands out at most the launch's registers; with fewer
    // at launch an increase would never be granted
    cudaFuncAttributes fa;
    r = cudaFuncGetAttributes(&fa, fattn_fwd_kernel<D, SUB, VARLEN, SPLIT>);
    if (r != cudaSuccess) return r;
    return fa.numRegs >= C::REG_LAUNCH ? cudaSuccess : cudaErrorInvalidConfiguration;
  });
  if (e != cudaSuccess) return e;
  const long long blocks = fwd_blocks<C::ROWS, VARLEN, SPLIT>(p);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (blocks == 0) return cudaSuccess;
  fattn_fwd_kernel<D, SUB, VARLEN, SPLIT><<<(unsigned)blocks, C::THREADS, C::SMEM, stream>>>(
      tq, tk, tv, to, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, cudaStream_t stream) {
  const bool vl = p.vl.cu_seqlens != nullptr;
  if (d == 128) return vl ? launch<128, 2, true, false>(tq, tk, tv, to, p, stream)
                          : launch<128, 2, false, false>(tq, tk, tv, to, p, stream);
  if (d == 64) {
    // One subtile per CTA (two CTAs per SM) when the two-subtile grid would be
    // at most six waves.  Measured at B4 H16 N2048, B8 H16 N1024, B1 H16 N8192
    // and B2 H16 N6144: 4-13 % faster without a mask, 0-6 % with the causal
    // one; at 6.7 waves and more (B1 H16 N16384, B1 H64 N8192) the doubled K/V
    // traffic from L2 made it 0-3 % slower.
    const long long two = vl ? fwd_blocks<256, true, false>(p) : fwd_blocks<256, false, false>(p);
    const int n_sm = device_sm_count();
    if (n_sm > 0 && two <= 6LL * n_sm)
      return vl ? launch<64, 1, true, false>(tq, tk, tv, to, p, stream)
                : launch<64, 1, false, false>(tq, tk, tv, to, p, stream);
    return vl ? launch<64, 2, true, false>(tq, tk, tv, to, p, stream)
              : launch<64, 2, false, false>(tq, tk, tv, to, p, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_split(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                             const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p,
                             cudaStream_t stream) {
  if (d == 128) return launch<128, 2, false, true>(tq, tk, tv, to, p, stream);
  if (d == 64) return launch<64, 2, false, true>(tq, tk, tv, to, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fattn
