/*
 * fattn.h -- C-ABI of libfattn: exact tiled scaled-dot-product attention
 * (FlashAttention forward and backward) for NVIDIA GB300 (sm_103a).
 *
 * The operation, for every (batch b, head h) independently
 * ("FlashAttention tiles exact softmax without materializing the score
 * matrix", opening equations; "tm_flash_attention_math", "What we must
 * compute, and why storage is the problem"):
 *
 *     S = scale * Q K^T            (N x N, never stored)
 *     P = softmax(S) row by row    (causal: key j visible to query i iff j <= i)
 *     O = P V
 *     LSE_i = m_i + ln l_i = ln sum_j exp(S_ij)
 *
 * LSE is the one per-row statistic the backward pass keeps ("Decoding flash
 * attention", "The backward pass"); the backward recomputes P = exp(S - LSE)
 * tile by tile and returns dQ, dK, dV of a loss whose gradient w.r.t. O is dO.
 *
 * Layout.  q, k, v, o, dout, dq, dk, dv are DEVICE pointers to contiguous
 * bf16 tensors [B, H, N, d] (row-major, d innermost).  lse is a DEVICE
 * pointer to fp32 [B, H, N].  Every pointer must be 16-byte aligned.
 * d must be 64 or 128.  N >= 1, B >= 1, H >= 1, B*H*N < 2^31.
 * scale must be finite and > 0 (every workload here uses 1/sqrt(d)).
 *
 * Ownership.  The caller allocates and owns every buffer; the library keeps
 * no per-call state and never frees caller memory.
 *
 * Streams and errors.  Calls are asynchronous on `stream` (a cudaStream_t;
 * NULL is the legacy default stream).  Arguments are validated before
 * anything is launched: a bad argument returns a non-zero status and
 * launches nothing.  A launch failure returns FATTN_ERR_CUDA.  Faults during
 * execution surface at the caller's next synchronisation, as usual in CUDA.
 * Every wait inside a kernel is bounded; a wait that runs out records a code
 * in a device error word and the kernel finishes without hanging.  The word is
 * read with fattn_device_error, which returns FATTN_ERR_TIMEOUT while it is
 * set.  With the environment variable FATTN_DEBUG set to a non-zero value
 * (read once per process), every entry point that launches work also
 * synchronises `stream` after enqueueing (not while the stream is being
 * captured into a graph) and returns FATTN_ERR_TIMEOUT if the word is set.
 *
 * The library remembers a few facts per device on first use (kernel
 * attributes, the SM count and L2 size, the error word's address); the
 * entries are tied to the device's current context and are set up again after
 * cudaDeviceReset.
 *
 * The device must be compute capability 10.3 (sm_103a), else
 * FATTN_ERR_UNSUPPORTED.
 */
#ifndef FATTN_H_
#define FATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FATTN_OK = 0,
  FATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, bad scale */
  FATTN_ERR_UNSUPPORTED = 2, /* d not in {64,128}, or the device is not sm_103 */
  FATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed */
  FATTN_ERR_WORKSPACE = 4,   /* workspace missing or too small */
  FATTN_ERR_TIMEOUT = 5      /* a bounded in-kernel wait ran out (fattn_device_error) */
} fattn_status;

/* Forward pass.  Writes o [B,H,N,d] bf16 and lse [B,H,N] fp32 (natural log,
 * in units of scaled scores).  The online-softmax state (running max m,
 * running sum l, unnormalised accumulator o~, rescale alpha = exp(m_old - m_new))
 * is carried across 128-key tiles ("tm_flash_attention_math", "The block-wise
 * update, and the full algorithm"); key tiles wholly above the causal
 * diagonal are skipped and only diagonal-crossing or ragged tiles are masked
 * element by element (page 1, "Causal masking fits inside the tiled
 * computation"). */
int fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int N, int d, float scale, int causal, void* stream);

/* fattn_fwd plus tile instrumentation: when tile_counts (DEVICE pointer to 3
 * unsigned 64-bit counters, 8-byte aligned) is not NULL, the kernel ADDS the
 * number of (128-row query tile, 128-key tile) pairs it processed without
 * masks [0], processed with element masks [1], and skipped as wholly above
 * the causal diagonal [2] (page 1, "Causal masking fits inside the tiled
 * computation": tiles beyond the permitted region are skipped, the ones on
 * the boundary masked).  The caller zeroes the counters.  The counters are an
 * argument of the call rather than library state set beforehand, so that
 * calls from several threads or streams, and calls captured into graphs,
 * each count into their own buffer. */
int fattn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, unsigned long long* tile_counts,
                 void* stream);

/* Bytes of device workspace fattn_bwd needs: an fp32 dQ accumulator
 * [B,H,N,d] and the fp32 row statistic D [B,H,N] (256-byte aligned parts).
 * No passage of the pages: it sizes the scratch of the backward formulas
 * below.  Returns 0 for B, H, N < 1 or d not in {64, 128}. */
size_t fattn_bwd_workspace_bytes(int B, int H, int N, int d);

/* Backward pass.  Inputs q, k, v, o, lse as produced by fattn_fwd and dout
 * = dL/dO; outputs dq, dk, dv [B,H,N,d] bf16.  The pages give no gradient
 * formulas; the calculus of the definition is used: D_i = sum_c dO_ic O_ic,
 * P = exp(S - LSE), dV = P^T dO, dP = dO V^T, dS = P o (dP - D),
 * dQ = scale dS K, dK = scale dS^T Q ("FlashAttention tiles exact softmax
 * without materializing the score matrix", "Backward computation can trade
 * recomputation for stored intermediates").
 * workspace: DEVICE memory of at least fattn_bwd_workspace_bytes(B,H,N,d)
 * bytes, 256-byte aligned, owned by the caller; its contents on entry do not
 * matter and are overwritten.  Too small or misaligned -> FATTN_ERR_WORKSPACE,
 * nothing launched.  NULL -> the call takes the scratch from the CUDA
 * stream-ordered allocator: cudaMallocAsync on `stream` before its kernels and
 * cudaFreeAsync on `stream` after them (workspace_bytes is then ignored); an
 * allocation failure returns FATTN_ERR_CUDA and launches nothing.  The
 * device's default memory pool keeps nothing across synchronisations unless
 * its release threshold is raised, so each such call maps its scratch anew;
 * a program that calls this repeatedly avoids that by passing a workspace. */
int fattn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
              const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
              float scale, int causal, void* workspace, size_t workspace_bytes, void* stream);

/* fattn_bwd plus phase timing: when phase_events is not NULL it points to 4
 * cudaEvent_t handles (created by the caller) that are recorded on `stream`
 * before the preprocess kernel, before the main kernel, after the main
 * kernel and after the dQ convert kernel. */
int fattn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, void* workspace, size_t workspace_bytes,
                 void* const* phase_events, void* stream);

/* Variable-length batches (padded attention without the padding: "Causal
 * masking fits inside the tiled computation" on page "FlashAttention tiles
 * exact softmax without materializing the score matrix" masks positions
 * inside a tile; here each sequence simply ends where its length says).
 * B sequences of lengths n_b = cu_seqlens[b+1] - cu_seqlens[b] are packed
 * head-major: q, k, v, o, dout, dq, dk, dv are DEVICE pointers to bf16
 * [H, total, d] (sequence b at rows [cu_seqlens[b], cu_seqlens[b+1]) of every
 * head) and lse is fp32 [H, total].  Each sequence is its own attention
 * problem: its queries see only its own keys (and, causal, only keys at or
 * before their own position in the sequence).
 * cu_seqlens: DEVICE int32 array of B+1 non-decreasing offsets, cu_seqlens[0]
 * = 0 and cu_seqlens[B] = total; max_seqlen >= every n_b (the grid is sized by
 * it); total is passed by the caller because the host cannot read device
 * memory without a synchronisation.  Entries are checked on the device: a
 * sequence that is out of range, decreasing or longer than max_seqlen is
 * skipped and reported through the device error word (code 0x140 forward,
 * 0x240 backward).  Empty sequences are allowed; total == 0 launches nothing.
 * Returns as fattn_fwd; tile counters are not available. */
int fattn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                     const int* cu_seqlens, int B, int H, int max_seqlen, int total, int d,
                     float scale, int causal, void* stream);

/* Backward of fattn_fwd_varlen ("Backward computation can trade recomputation
 * for stored intermediates" on page 1, per sequence): the layouts above;
 * workspace of at least fattn_bwd_workspace_bytes(1, H, total, d) bytes, or
 * NULL for stream-ordered scratch as in fattn_bwd.  Returns as fattn_bwd. */
int fattn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     const int* cu_seqlens, int B, int H, int max_seqlen, int total, int d,
                     float scale, int causal, void* workspace, size_t workspace_bytes,
                     void* stream);

/* Split-KV attention for a few queries against many keys (decoding).
 * q [B,H,Nq,d], k, v [B,H,Nkv,d] bf16, 1 <= Nq <= Nkv; outputs o [B,H,Nq,d]
 * bf16 and lse [B,H,Nq] fp32, all DEVICE pointers, 16-byte aligned.  The
 * queries are the LAST Nq positions of the sequence: with causal, query i
 * sees keys j <= Nkv - Nq + i (Nq == Nkv is fattn_fwd's causal mask).
 * The 128-key tiles are cut into key ranges, one per CTA of the forward
 * kernel, each leaving its range's normalised result and log-sum-exp in the
 * workspace; a merge kernel combines them (fattn_merge_partials).  This is
 * the block-wise recurrence of "tm_flash_attention_math" ("The block-wise
 * update, and the full algorithm"), with whole blocks' states merged, which
 * the page's "Proof of exactness" allows in any order.
 * n_splits: 0 = automatic (about ten waves of CTAs, at least four tiles per
 * range), else the requested number
 * of ranges (capped at one per tile; the count used is fattn_decode_splits).
 * workspace: DEVICE memory of fattn_decode_workspace_bytes(...) bytes,
 * 256-byte aligned, owned by the caller.  Returns FATTN_OK,
 * FATTN_ERR_INVALID_ARG, FATTN_ERR_UNSUPPORTED, FATTN_ERR_WORKSPACE or
 * FATTN_ERR_CUDA; launches nothing on an argument error. */
int fattn_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int Nq, int Nkv, int d, float scale, int causal, int n_splits, void* workspace,
                 size_t workspace_bytes, void* stream);

/* Number of key ranges fattn_decode uses for these arguments on the current
 * device (the automatic count follows its SM count); 0 if invalid.  A sizing
 * helper of fattn_decode; no passage of its own. */
int fattn_decode_splits(int B, int H, int Nq, int Nkv, int d, int n_splits);

/* Workspace bytes fattn_decode needs on the current device: S x B*H*Nq x
 * (d + 1) fp32 with S = fattn_decode_splits(...); 0 if invalid.  A sizing
 * helper of fattn_decode; no passage of its own. */
size_t fattn_decode_workspace_bytes(int B, int H, int Nq, int Nkv, int d, int n_splits);

/* Merge of partial results over disjoint key ranges ("tm_flash_attention_math",
 * "Proof of exactness": block states combine in any order): o_part [S, rows, d] and
 * lse_part [S, rows] fp32 (range s's normalised output and log-sum-exp; a
 * range in which a row saw no key has lse = -inf) -> lse = log sum_s
 * exp(lse_s), o = sum_s exp(lse_s - lse) o_s as bf16 [rows, d]; a row with
 * every lse_s = -inf gets o = 0 and lse = -inf.  DEVICE pointers, 16-byte
 * aligned; d in {64, 128}. */
int fattn_merge_partials(const float* o_part, const float* lse_part, int n_splits, long long rows,
                         int d, void* o, float* lse, void* stream);

/* Row-wise softmax with the online normaliser: y[r, :] = exp(x[r, :] - m_r) / l_r
 * with m_r the row maximum and l_r = sum exp(x[r, :] - m_r), formed in one
 * sweep by the (m, l) recurrence of "FlashAttention tiles exact softmax
 * without materializing the score matrix" ("The online softmax recurrence").
 * x, y: DEVICE fp32 [rows, cols], row-major, 16-byte aligned (y may equal x);
 * lse: DEVICE fp32 [rows] receiving m_r + ln l_r, or NULL.  A row whose values
 * are all -inf gets y = 0 and lse = -inf.  Rows of up to 49152 values are read
 * from HBM once; longer rows twice.  Returns FATTN_OK, FATTN_ERR_INVALID_ARG,
 * FATTN_ERR_UNSUPPORTED or FATTN_ERR_CUDA. */
int fattn_softmax_rows(const float* x, float* y, float* lse, long long rows, int cols,
                       void* stream);

/* Size of the device array that fattn_bwd_noalloc uses as its workspace. */
#define FATTN_NOALLOC_SCRATCH_BYTES (64u << 20)

/* fattn_bwd without a caller-provided workspace, for callers that cannot
 * allocate device memory where they run the backward (a plugin inside a host
 * program that owns the CUDA allocator, or a runtime that reserves its whole
 * memory budget up front).  The pages have no counterpart to this entry
 * point; it is a packaging variant of fattn_bwd.
 * The workspace is a fixed device array of FATTN_NOALLOC_SCRATCH_BYTES that
 * every GPU loading the library holds until exit; nothing is allocated or
 * freed.  Problems with fattn_bwd_workspace_bytes(B,H,N,d) larger than that
 * return FATTN_ERR_WORKSPACE and launch nothing.  All calls share the array:
 * calls that overlap on the GPU race on it.  The first call on a device looks
 * up the array's device address, so it should come before any stream capture.
 * Arguments, layouts, results and other errors are those of fattn_bwd. */
int fattn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                      int H, int N, int d, float scale, int causal, void* stream);

/* Sizing helper of fattn_fwd_bwd_host (no passage of its own).
 * Bytes of DEVICE workspace fattn_fwd_bwd_host needs: three staging slots,
 * each holding Q, K, V, dO, O, dQ, dK, dV and LSE of one chunk of heads plus
 * that chunk's backward workspace.  heads_per_chunk = 0 selects the library's
 * chunk size for the current device (the same one fattn_fwd_bwd_host picks
 * for 0).  Returns 0 for invalid sizes. */
size_t fattn_fwd_bwd_host_workspace_bytes(int B, int H, int N, int d, int heads_per_chunk);

/* Forward and backward of tensors in HOST memory: the same results as
 * fattn_fwd followed by fattn_bwd.  q, k, v, dout are HOST pointers to bf16
 * [B,H,N,d]; o, dq, dk, dv HOST pointers to bf16 [B,H,N,d] and lse to fp32
 * [B,H,N], all written by the call.  Every (b, h) slice is an independent
 * problem ("FlashAttention tiles exact softmax without materializing the score
 * matrix", opening equations), so the slices move through `workspace` (DEVICE,
 * 256-byte aligned, fattn_fwd_bwd_host_workspace_bytes large) in chunks of
 * heads_per_chunk consecutive slices (0 = the library's choice; the first
 * chunk is half as large so that the kernels start sooner), and the copy in of
 * one chunk, the kernels of the previous one and the copy out of the one
 * before run at the same time on three streams the library keeps per device.  Asynchronous on `stream` like the other entry points: the host
 * buffers must stay untouched until `stream` has reached this call's end.
 * The copies overlap only when the host buffers are page-locked
 * (cudaHostAlloc or cudaHostRegister); pageable memory gives the same results
 * with the copies serialised.  Calls from several host threads are
 * serialised while they enqueue.  Errors: those of fattn_fwd and fattn_bwd;
 * FATTN_ERR_WORKSPACE for a missing, misaligned or short workspace. */
int fattn_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dout, void* o,
                       float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                       float scale, int causal, int heads_per_chunk, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Tile shape used by a pass (0 = forward, 1 = backward) for head size d:
 * rows of Q per tile and keys per K/V tile; 128 x 128, the tile of "Decoding
 * flash attention" ("The idea: never build the matrix").  block_q and block_k may be NULL.
 * Returns FATTN_OK, FATTN_ERR_UNSUPPORTED (d) or FATTN_ERR_INVALID_ARG (pass). */
int fattn_tile_sizes(int d, int pass, int* block_q, int* block_k);

/* Read (and, if clear != 0, reset) the device error word of the current
 * device: *code = 0 if no in-kernel wait ran out since the last reset, else
 * the code of the first one (low byte: the waiting role; next byte: the
 * kernel).  Synchronises the device.  Returns FATTN_OK when the word was 0,
 * FATTN_ERR_TIMEOUT when it was set (with *code written, and cleared if
 * asked), FATTN_ERR_INVALID_ARG for a NULL code, FATTN_ERR_CUDA.  The pages
 * have no counterpart: it reports this library's bounded waits. */
int fattn_device_error(unsigned int* code, int clear);

/* Human-readable name of a status code (static storage).  No passage: a helper.
 * The library also exports two test and measurement hooks, declared apart in
 * fattn_testing.h; they are not part of this interface. */
const char* fattn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H_ */
