// bwd_aux.cu -- the two HBM-bound kernels around the backward main kernel.
//
//   preprocess: D_i = sum_c dO_ic * O_ic for every row (fp32), and zero the
//               fp32 dQ accumulator.  D_i equals sum_j P_ij dP_ij, the row term
//               of dS = P o (dP - D), because O = P V and dP = dO V^T.
//   convert:    dQ = bf16(scale * dQ_acc).
//
// Both stream their operands once with 16-byte accesses; the grid is a
// multiple of the SM count and loops over the rows.
#include <cuda_bf16.h>

#include "common.cuh"

namespace fattn {
namespace {

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// G threads per row, 8 elements (16 bytes of bf16) per thread.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const uint4* __restrict__ o,
                                                         const uint4* __restrict__ dout,
                                                         float* __restrict__ delta,
                                                         float4* __restrict__ dq_acc,
                                                         long long rows) {
  constexpr int G = D / 8;
  const long long total = rows * G;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int lane = threadIdx.x & 31, g = threadIdx.x % G;
  // warp-uniform trip count, so the group shuffles always see the full warp
  for (long long base = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < total;
       base += stride) {
    const long long t = base + lane;
    const bool valid = t < total;
    float acc = 0.f;
    if (valid) {
      const uint4 a = o[t], b = dout[t];
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = bf2_to_f2(av[i]), y = bf2_to_f2(bv[i]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, G);
    if (valid) {
      if (g == 0) delta[t / G] = acc;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      dq_acc[2 * t] = z;
      dq_acc[2 * t + 1] = z;
    }
  }
}

__global__ void __launch_bounds__(256) convert_kernel(const float4* __restrict__ acc,
                                                      uint4* __restrict__ out, long long n8,
                                                      float scale) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < n8; t += stride) {
    const float4 a = acc[2 * t], b = acc[2 * t + 1];
    __nv_bfloat162 r0 = __floats2bfloat162_rn(a.x * scale, a.y * scale);
    __nv_bfloat162 r1 = __floats2bfloat162_rn(a.z * scale, a.w * scale);
    __nv_bfloat162 r2 = __floats2bfloat162_rn(b.x * scale, b.y * scale);
    __nv_bfloat162 r3 = __floats2bfloat162_rn(b.z * scale, b.w * scale);
    uint4 u;
    u.x = *reinterpret_cast<uint32_t*>(&r0);
    u.y = *reinterpret_cast<uint32_t*>(&r1);
    u.z = *reinterpret_cast<uint32_t*>(&r2);
    u.w = *reinterpret_cast<uint32_t*>(&r3);
    out[t] = u;
  }
}

unsigned grid_for(long long work, int threads, int n_sm) {
  const long long want = (work + threads - 1) / threads;
  const long long cap = (long long)n_sm * 8;  // 8 resident 256-thread blocks per SM
  return (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void* o, const void* dout, float* delta, float* dq_acc,
                                  long long rows, int d, int n_sm, cudaStream_t stream) {
  const long long work = rows * (d / 8);
  const unsigned grid = grid_for(work, 256, n_sm);
  if (d == 128)
    preprocess_kernel<128><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(o),
                                                     static_cast<const uint4*>(dout), delta,
                                                     reinterpret_cast<float4*>(dq_acc), rows);
  else if (d == 64)
    preprocess_kernel<64><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(o),
                                                    static_cast<const uint4*>(dout), delta,
                                                    reinterpret_cast<float4*>(dq_acc), rows);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_bwd_convert(const float* dq_acc, void* dq, long long n, float scale,
                               int n_sm, cudaStream_t stream) {
  const long long n8 = n / 8;
  convert_kernel<<<grid_for(n8, 256, n_sm), 256, 0, stream>>>(reinterpret_cast<const float4*>(dq_acc),
                                                        static_cast<uint4*>(dq), n8, scale);
  return cudaGetLastError();
}

}  // namespace fattn
