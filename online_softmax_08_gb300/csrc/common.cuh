// common.cuh -- launch parameters shared by the host API and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fattn {

// Codes written to the device error word by a wait that timed out.  The low
// byte names the waiting role, the next byte the barrier.
enum : uint32_t {
  ERR_SITE_FWD = 0x100,
  ERR_SITE_BWD = 0x200,
  ERR_SITE_CHECK = 0x300,  // fattn_check_wait_timeout
};

// Variable-length batches: B sequences packed head-major, [H, T, d] with
// sequence b at rows [cu_seqlens[b], cu_seqlens[b+1]) of every head (T =
// cu_seqlens[B]).  Null cu_seqlens means the dense [B, H, N, d] layout.
struct Varlen {
  const int* cu_seqlens;      // device, B + 1 entries, or null
  int B;                      // sequences
  int H;                      // heads
  int T;                      // total rows per head
};

struct FwdParams {
  int BH;                     // batch * heads
  int N;                      // sequence length (queries == keys); the longest one when varlen
  int causal;                 // key j visible to query i iff j <= i
  float scale_log2;           // scale * log2(e): scores are taken to base 2
  float* lse;                 // [BH, N] fp32, natural-log units
  unsigned long long* tiles;  // optional [3]: full, masked, skipped (may be null)
  unsigned int* err;          // device error word
  Varlen vl;
  uint16_t* o;                // O (bf16 bits); varlen writes the last tile of a sequence row by row
  // Split-KV (decode): N keys, Nq queries aligned to the END of the keys (query
  // i sits at position N - Nq + i); the key tiles are cut into n_splits ranges
  // of tiles_per_split tiles, one per CTA, whose normalised partial results go
  // to o_part [n_splits, BH, Nq, d] and lse_part [n_splits, BH, Nq] (fp32).
  int Nq;
  int n_splits;
  int tiles_per_split;
  float* o_part;
  float* lse_part;
  int group;                  // dense grid: heads per group of the CTA order (0: one group)
};

struct BwdParams {
  int BH;
  int N;
  int causal;
  float scale;                // softmax scale (dK and dQ are multiplied by it)
  float scale_log2;           // scale * log2(e)
  const float* lse;           // [BH, N] saved by the forward pass
  const float* delta;         // [BH, N] D_i = rowsum(dO o O)
  float* dq_acc;              // [BH, N, d] fp32 dQ accumulator (zeroed by the preprocess kernel)
  unsigned int* err;
  Varlen vl;
  uint16_t* dk;               // dK, dV (bf16 bits); varlen writes the last key block of a
  uint16_t* dv;               // sequence row by row
  int group;                  // dense grid: heads per group of the CTA order (0: one group)
};

// Dense grid order: the CTAs go through the heads in groups of `group` heads
// and, within a group, block by block (all of the group's heads for block 0,
// then block 1, ...), so the CTAs in flight read the tensors of one or two
// groups, which stay in L2.  group = 0 (or >= units) is one group: the order
// is block-major over all heads.  Returns the CTA's block index in that order
// and its (b, h) unit.
__device__ __forceinline__ void grouped_order(unsigned bidx, int units, int blocks, int group,
                                              int* blk, int* unit) {
  const int G = (group > 0 && group < units) ? group : units;
  const unsigned per_group = (unsigned)blocks * (unsigned)G;
  const int g = (int)(bidx / per_group);
  const int first = g * G;
  const int gs = min(G, units - first);  // only the last group may be smaller
  const unsigned r = bidx - (unsigned)g * per_group;
  *blk = (int)(r / (unsigned)gs);
  *unit = first + (int)(r % (unsigned)gs);
}

// Where a CTA's sequence lives: its length, its first row in the tensor's
// row dimension, the TMA z coordinate (b*H + h dense, h varlen), and the base
// row of its per-row statistics (LSE, D).  Returns false for a bad
// cu_seqlens entry (recorded in the error word by the caller).
struct SeqView {
  int N;
  int row0;
  int z;
  long long stat0;
};
__device__ __forceinline__ bool seq_view(const Varlen& vl, int dense_N, int seq, int head,
                                         int dense_bh, int max_len, SeqView* v) {
  if (vl.cu_seqlens == nullptr) {
    v->N = dense_N;
    v->row0 = 0;
    v->z = dense_bh;
    v->stat0 = (long long)dense_bh * dense_N;
    return true;
  }
  const int a = vl.cu_seqlens[seq], b = vl.cu_seqlens[seq + 1];
  if (a < 0 || b < a || b > vl.T || b - a > max_len) return false;
  v->N = b - a;
  v->row0 = a;
  v->z = head;
  v->stat0 = (long long)head * vl.T + a;
  return true;
}

// Identity of the calling thread's current CUDA context (the device's primary
// context under the runtime API): a process-unique id, 0 when no context is
// current yet.  Per-device caches remember the context they were filled in and
// fill themselves again when it changes, since cudaDeviceReset destroys the
// primary context and every attribute, address, stream and event made in it.
unsigned long long current_context_id();

// Per-device one-time preparation of a kernel (its shared-memory opt-in and
// register checks), so that later calls, including calls under stream capture
// into a CUDA graph, make no attribute calls.  ctx_ids: one entry per device,
// the context the preparation was made in (0: not prepared).
template <typename Prep>
cudaError_t prepare_once(unsigned long long (&ctx_ids)[64], Prep prep) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  if (ctx != 0 && __atomic_load_n(&ctx_ids[dev], __ATOMIC_ACQUIRE) == ctx) return cudaSuccess;
  const cudaError_t e = prep();  // idempotent: two threads may both run it
  if (e == cudaSuccess) __atomic_store_n(&ctx_ids[dev], current_context_id(), __ATOMIC_RELEASE);
  return e;
}

// Device facts the launchers size their grids and groups with.
int device_sm_count();             // streaming multiprocessors of the current device (0: error)
long long device_l2_bytes();       // L2 cache of the current device (0: error)

// When the environment variable FATTN_DEBUG is set to a non-zero value, an
// entry point that enqueued work successfully synchronises `stream` (unless it
// is being captured into a graph) and returns FATTN_ERR_TIMEOUT if the device
// error word is set; otherwise it returns `status` unchanged.
int debug_post_call(int status, cudaStream_t stream);

// Launchers (one per translation unit).  Return cudaSuccess or the launch error.
cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd_split(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                             const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p,
                             cudaStream_t stream);
// Row-wise softmax with the online normaliser (fp32 in and out, optional LSE per row).
cudaError_t launch_softmax_rows(const float* x, float* y, float* lse, long long rows, int cols,
                                int n_sm, cudaStream_t stream);
// Merge of split partials: lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s (bf16).
cudaError_t launch_merge(const float* o_part, const float* lse_part, int n_splits, long long rows,
                         int d, void* o, float* lse, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const void* o, const void* dout, float* delta, float* dq_acc,
                                  long long rows, int d, int n_sm, cudaStream_t stream);
cudaError_t launch_bwd_main(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const CUtensorMap& tdq_acc, const BwdParams& p, cudaStream_t stream);
// Query rows per bulk reduce of the backward's dQ partials (the box height of
// the accumulator's tensor map).
// box of the dQ accumulator's bulk reduces: columns x query rows, 128-byte swizzle or none
struct DqBox {
  int cols, rows;
  bool sw128;
};
DqBox bwd_dq_box(int d);
cudaError_t launch_bwd_convert(const float* dq_acc, void* dq, long long n, float scale,
                               int n_sm, cudaStream_t stream);

}  // namespace fattn
