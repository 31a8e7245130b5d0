// noalloc.cu -- fattn_bwd_noalloc: the backward pass with a built-in workspace.
//
// The backward pass needs device scratch memory (an fp32 dQ accumulator and
// the per-row statistic D).  fattn_bwd takes it from the caller.  Some callers
// cannot allocate device memory at the point where they run the backward:
// for example a plugin loaded into a host program that owns the CUDA
// allocator and does not expose it, or a runtime that reserves its whole
// memory budget up front and forbids allocation afterwards.  For them this
// file keeps the workspace in a fixed device array that is part of the
// library image, and fattn_bwd_noalloc hands that array to fattn_bwd.  No
// cudaMalloc, cudaFree or other allocating routine is called.
//
// Costs and limits:
//   * every GPU that loads the library holds FATTN_NOALLOC_SCRATCH_BYTES of
//     device memory for this array until the process exits;
//   * problems whose workspace (fattn_bwd_workspace_bytes) exceeds that size
//     are rejected with FATTN_ERR_WORKSPACE before anything is launched;
//   * all calls share the one array: calls whose kernels overlap on the GPU
//     (e.g. on two streams at once) race on it and give wrong results.  The
//     array keeps the previous call's contents; the parts that must start at
//     zero (the dQ accumulator) are cleared by the backward's own first kernel
//     on every call;
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it, so that
//     first call should come before any stream capture.  The cache remembers
//     the context it was filled in: after cudaDeviceReset the next call looks
//     the address up again.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/fattn.h"
#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchAddress {
  unsigned long long ctx = 0;  // context the address was looked up in (0: not yet)
  void* ptr = nullptr;
};
ScratchAddress g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set up once per
// device and context).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddress& e = g_scratch[dev];
  const unsigned long long ctx = fattn::current_context_id();
  if (ctx == 0 || e.ctx != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
      return FATTN_ERR_CUDA;
    e.ptr = ptr;
    e.ctx = fattn::current_context_id();  // the lookup made the context current
  }
  *out = e.ptr;
  return FATTN_OK;
}

}  // namespace

extern "C" int fattn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                 const float* lse, const void* dout, void* dq, void* dk,
                                 void* dv, int B, int H, int N, int d, float scale, int causal,
                                 void* stream) {
  // fattn_bwd's size checks, in its order, before the scratch-size check, so
  // that both entry points give the same status for the same bad arguments
  if (B < 1 || H < 1 || N < 1) return FATTN_ERR_INVALID_ARG;
  if ((long long)B * H * N >= (1LL << 31)) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  if (fattn_bwd_workspace_bytes(B, H, N, d) > (size_t)FATTN_NOALLOC_SCRATCH_BYTES)
    return FATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != FATTN_OK) return st;
  return fattn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, scratch,
                   (size_t)FATTN_NOALLOC_SCRATCH_BYTES, stream);
}
