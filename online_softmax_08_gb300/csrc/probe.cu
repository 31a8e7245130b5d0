// probe.cu -- measured throughput of the ex2 unit, the forward pass's second
// ceiling after the tensor cores.
//
// The online softmax takes one exponential per visible score
// ("tm_flash_attention_math", "The block-wise update, and the full
// algorithm"); the kernels evaluate it with ex2.approx on the multi-function
// unit.  This kernel keeps that unit busy with eight independent chains
// x <- ex2(-|x| / 2) per thread on every SM (the scaling runs on the FMA
// pipe), so that the measured rate is the one the forward's exponentials are
// compared with.
#include "../../include/fattn.h"
#include "common.cuh"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int kChains = 8;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) ex2_probe_kernel(float* out, int iters) {
  float x[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) x[c] = -1e-3f * (float)(threadIdx.x + c);
#pragma unroll 1
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = ex2(-0.5f * fabsf(x[c]));  // stays in (0, 1]
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += x[c];
  if (s == 12345.f) out[blockIdx.x] = s;  // keeps the loop; never true
}

}  // namespace
}  // namespace fattn

extern "C" int fattn_ex2_throughput(double* per_second, void* stream) {
  if (!per_second) return FATTN_ERR_INVALID_ARG;
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FATTN_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int blocks = n_sm * 8;  // 2048 threads per SM
  const int iters = 4096;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  int st = FATTN_OK;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    st = FATTN_ERR_CUDA;
  } else {
    fattn::ex2_probe_kernel<<<blocks, fattn::kThreads, 0, s>>>(nullptr, iters / 8);  // warm-up
    cudaEventRecord(e0, s);
    fattn::ex2_probe_kernel<<<blocks, fattn::kThreads, 0, s>>>(nullptr, iters);
    cudaEventRecord(e1, s);
    float ms = 0.f;
    if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess || !(ms > 0.f)) {
      st = FATTN_ERR_CUDA;
    } else {
      const double n = (double)blocks * fattn::kThreads * fattn::kChains * iters;
      *per_second = n / (ms * 1e-3);
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  return st;
}
