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

struct FwdParams {
  int BH;                     // batch * heads
  int N;                      // sequence length (queries == keys)
  int causal;                 // key j visible to query i iff j <= i
  float scale_log2;           // scale * log2(e): scores are taken to base 2
  float* lse;                 // [BH, N] fp32, natural-log units
  unsigned long long* tiles;  // optional [3]: full, masked, skipped (may be null)
  unsigned int* err;          // device error word
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
};

// Launchers (one per translation unit).  Return cudaSuccess or the launch error.
cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const void* o, const void* dout, float* delta, float* dq_acc,
                                  long long rows, int d, cudaStream_t stream);
cudaError_t launch_bwd_main(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const CUtensorMap& tdq_acc, const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_convert(const float* dq_acc, void* dq, long long n, float scale,
                               cudaStream_t stream);

}  // namespace fattn
