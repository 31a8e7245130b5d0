// staged.cu -- forward + backward of host-resident tensors, pipelined by head chunks.
//
// fattn_fwd_bwd_host takes Q, K, V, dO in host memory and returns O, LSE, dQ,
// dK, dV in host memory.  Every (batch, head) slice is independent in both
// passes ("FlashAttention tiles exact softmax without materializing the score
// matrix": each head is its own N x N problem), so the slices move through the
// device in chunks of consecutive heads, and three device slots let the copies
// of one chunk overlap the kernels of another:
//
//   copy-in stream   : Q, K, V of chunk c -> slot c % 3 (qkv_in); dO (do_in)
//   compute stream   : wait qkv_in; fattn_fwd (fwd_done); wait do_in; fattn_bwd (bwd_done)
//   copy-out stream  : wait fwd_done; O, LSE -> host; wait bwd_done; dQ, dK, dV -> host (out_done)
//
// The forward starts before dO has arrived and O, LSE leave while the
// backward runs.  The first chunk is half the size of the others, so the
// kernels start sooner.  Before a slot is filled again the copy-in stream
// waits for that slot's previous out_done.  The three streams first wait for
// the caller's stream, and the caller's stream finally waits for the last
// out_done, so the call is ordered like any other work on `stream`.  The
// kernels are the ones fattn_fwd and fattn_bwd launch, on B*H = (heads in the
// chunk).
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/fattn.h"
#include "common.cuh"

namespace {

constexpr int kSlots = 3;
constexpr int kMaxDevices = 64;

struct Pipeline {
  unsigned long long ctx = 0;  // context the streams and events were made in (0: none yet)
  int n_sm = 0;
  cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t qkv_in[kSlots] = {}, do_in[kSlots] = {}, fwd_done[kSlots] = {},
              bwd_done[kSlots] = {}, out_done[kSlots] = {};
  std::mutex mu;  // one call at a time enqueues on the shared streams
};
Pipeline g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

int pipeline_for_current_device(Pipeline** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  Pipeline& p = g_pipe[dev];
  const unsigned long long ctx = fattn::current_context_id();
  if (ctx == 0 || p.ctx != ctx) {
    // first use, or the context was reset: the old handles died with it
    const unsigned sf = cudaStreamNonBlocking;
    const unsigned ef = cudaEventDisableTiming;
    if (cudaDeviceGetAttribute(&p.n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.s_in, sf) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.s_comp, sf) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.s_out, sf) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, ef) != cudaSuccess)
      return FATTN_ERR_CUDA;
    for (int i = 0; i < kSlots; ++i)
      for (cudaEvent_t* e : {&p.qkv_in[i], &p.do_in[i], &p.fwd_done[i], &p.bwd_done[i],
                             &p.out_done[i]})
        if (cudaEventCreateWithFlags(e, ef) != cudaSuccess) return FATTN_ERR_CUDA;
    p.ctx = fattn::current_context_id();
  }
  *out = &p;
  return FATTN_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Byte offsets of one slot's buffers for chunks of `heads` slices.
struct SlotLayout {
  size_t tile;     // one bf16 [heads, N, d] tensor
  size_t lse;      // fp32 [heads, N]
  size_t bwd_ws;   // the backward's workspace
  size_t bytes;    // whole slot
  size_t off(int i) const { return tile * i; }  // q k v do o dq dk dv: i = 0..7
  size_t off_lse() const { return tile * 8; }
  size_t off_ws() const { return tile * 8 + lse; }
};

SlotLayout slot_layout(int heads, int N, int d) {
  SlotLayout L;
  const size_t rows = (size_t)heads * N;
  L.tile = align256(rows * d * 2);
  L.lse = align256(rows * 4);
  L.bwd_ws = fattn_bwd_workspace_bytes(1, heads, N, d);
  L.bytes = L.tile * 8 + L.lse + L.bwd_ws;
  return L;
}

// Heads per chunk when the caller leaves it to the library: enough backward
// CTAs (one per 128 keys and head) for about three waves over the SMs, and at
// least four chunks when there are enough heads for that.
int auto_heads(long long BH, int N, int n_sm) {
  const long long ctas_per_head = (N + 127) / 128;
  long long h = (3LL * n_sm + ctas_per_head - 1) / ctas_per_head;
  const long long quarter = (BH + 3) / 4;
  if (h > quarter) h = quarter;
  if (h < 1) h = 1;
  if (h > BH) h = BH;
  return (int)h;
}

int check_args(int B, int H, int N, int d, float scale, int heads_per_chunk) {
  if (B < 1 || H < 1 || N < 1 || heads_per_chunk < 0) return FATTN_ERR_INVALID_ARG;
  if ((long long)B * H * N >= (1LL << 31)) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || scale != scale || scale > 3.0e38f) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  return FATTN_OK;
}

int resolve_heads(int B, int H, int N, int heads_per_chunk, int* heads) {
  const long long BH = (long long)B * H;
  if (heads_per_chunk > 0) {
    *heads = (int)(heads_per_chunk < BH ? heads_per_chunk : BH);
    return FATTN_OK;
  }
  Pipeline* p = nullptr;
  const int st = pipeline_for_current_device(&p);
  if (st != FATTN_OK) return st;
  *heads = auto_heads(BH, N, p->n_sm);
  return FATTN_OK;
}

}  // namespace

extern "C" size_t fattn_fwd_bwd_host_workspace_bytes(int B, int H, int N, int d,
                                                      int heads_per_chunk) {
  if (check_args(B, H, N, d, 1.f, heads_per_chunk) != FATTN_OK) return 0;
  int heads = 0;
  if (resolve_heads(B, H, N, heads_per_chunk, &heads) != FATTN_OK) return 0;
  return kSlots * slot_layout(heads, N, d).bytes;
}

extern "C" int fattn_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dout,
                                  void* o, float* lse, void* dq, void* dk, void* dv, int B, int H,
                                  int N, int d, float scale, int causal, int heads_per_chunk,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_args(B, H, N, d, scale, heads_per_chunk);
  if (st != FATTN_OK) return st;
  if (!q || !k || !v || !dout || !o || !lse || !dq || !dk || !dv) return FATTN_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FATTN_ERR_WORKSPACE;
  int heads = 0;
  st = resolve_heads(B, H, N, heads_per_chunk, &heads);
  if (st != FATTN_OK) return st;
  const SlotLayout L = slot_layout(heads, N, d);
  if (workspace_bytes < kSlots * L.bytes) return FATTN_ERR_WORKSPACE;
  Pipeline* p = nullptr;
  st = pipeline_for_current_device(&p);
  if (st != FATTN_OK) return st;
  std::lock_guard<std::mutex> lock(p->mu);

  const cudaStream_t user = static_cast<cudaStream_t>(stream);
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (!ok(cudaEventRecord(p->start, user)) || !ok(cudaStreamWaitEvent(p->s_in, p->start, 0)) ||
      !ok(cudaStreamWaitEvent(p->s_comp, p->start, 0)) ||
      !ok(cudaStreamWaitEvent(p->s_out, p->start, 0)))
    return FATTN_ERR_CUDA;

  // every chunk's copies and kernels; returns the status of the first failure
  long long n_chunks = 0;
  auto enqueue_chunks = [&]() -> int {
    const long long BH = (long long)B * H;
    const size_t head_bytes = (size_t)N * d * 2;
    const void* in_host[4] = {q, k, v, dout};
    void* out_host[4] = {o, dq, dk, dv};
    const int first = (heads + 1) / 2;
    long long c = 0;
    for (long long h0 = 0; h0 < BH; ++c) {
      const int s = (int)(c % kSlots);
      const long long want = c == 0 ? first : heads;
      const int hc = (int)((BH - h0) < want ? (BH - h0) : want);
      char* slot = static_cast<char*>(workspace) + (size_t)s * L.bytes;
      char* dev[8];  // q k v do o dq dk dv
      for (int i = 0; i < 8; ++i) dev[i] = slot + L.off(i);
      float* dlse = reinterpret_cast<float*>(slot + L.off_lse());
      void* ws = slot + L.off_ws();
      const size_t bytes = (size_t)hc * head_bytes;
      const size_t host_off = (size_t)h0 * head_bytes;
      auto copy_in = [&](int i) {
        return ok(cudaMemcpyAsync(dev[i], static_cast<const char*>(in_host[i]) + host_off, bytes,
                                  cudaMemcpyHostToDevice, p->s_in));
      };
      auto copy_out = [&](int i) {  // i = 0..3: o dq dk dv
        return ok(cudaMemcpyAsync(static_cast<char*>(out_host[i]) + host_off, dev[4 + i], bytes,
                                  cudaMemcpyDeviceToHost, p->s_out));
      };

      // copy in (after the slot's previous contents have been copied out)
      if (c >= kSlots && !ok(cudaStreamWaitEvent(p->s_in, p->out_done[s], 0))) return FATTN_ERR_CUDA;
      if (!copy_in(0) || !copy_in(1) || !copy_in(2) || !ok(cudaEventRecord(p->qkv_in[s], p->s_in)) ||
          !copy_in(3) || !ok(cudaEventRecord(p->do_in[s], p->s_in)))
        return FATTN_ERR_CUDA;

      // forward once Q, K, V are in; backward once dO is in too
      if (!ok(cudaStreamWaitEvent(p->s_comp, p->qkv_in[s], 0))) return FATTN_ERR_CUDA;
      st = fattn_fwd(dev[0], dev[1], dev[2], dev[4], dlse, 1, hc, N, d, scale, causal, p->s_comp);
      if (st != FATTN_OK) return st;
      if (!ok(cudaEventRecord(p->fwd_done[s], p->s_comp)) ||
          !ok(cudaStreamWaitEvent(p->s_comp, p->do_in[s], 0)))
        return FATTN_ERR_CUDA;
      st = fattn_bwd(dev[0], dev[1], dev[2], dev[4], dlse, dev[3], dev[5], dev[6], dev[7], 1, hc, N,
                     d, scale, causal, ws, L.bwd_ws, p->s_comp);
      if (st != FATTN_OK) return st;
      if (!ok(cudaEventRecord(p->bwd_done[s], p->s_comp))) return FATTN_ERR_CUDA;

      // copy out: O and LSE while the backward runs, then the gradients
      if (!ok(cudaStreamWaitEvent(p->s_out, p->fwd_done[s], 0)) || !copy_out(0) ||
          !ok(cudaMemcpyAsync(lse + (size_t)h0 * N, dlse, (size_t)hc * N * sizeof(float),
                              cudaMemcpyDeviceToHost, p->s_out)) ||
          !ok(cudaStreamWaitEvent(p->s_out, p->bwd_done[s], 0)) || !copy_out(1) || !copy_out(2) ||
          !copy_out(3) || !ok(cudaEventRecord(p->out_done[s], p->s_out)))
        return FATTN_ERR_CUDA;
      h0 += hc;
    }
    n_chunks = c;
    return FATTN_OK;
  };
  st = enqueue_chunks();
  if (st != FATTN_OK) {
    // the caller's stream still waits for whatever was enqueued, so that the
    // host buffers stay in use until those copies have finished
    for (cudaStream_t q2 : {p->s_in, p->s_comp, p->s_out})
      if (cudaEventRecord(p->start, q2) == cudaSuccess) cudaStreamWaitEvent(user, p->start, 0);
    return st;
  }
  // the caller's stream continues once the last copy out is done (the copy-out
  // stream runs in order, and each of its chunks waited for that chunk's
  // kernels, which waited for that chunk's copies in)
  const int last = (int)((n_chunks - 1) % kSlots);
  if (!ok(cudaStreamWaitEvent(user, p->out_done[last], 0))) return FATTN_ERR_CUDA;
  return fattn::debug_post_call(FATTN_OK, user);
}
