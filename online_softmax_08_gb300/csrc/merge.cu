// merge.cu -- combine partial attention results computed over disjoint key ranges.
//
// A CTA of the split forward pass covers one range of keys and leaves, per
// query row, the result normalised over that range, o_s, and its log-sum-exp,
// lse_s.  Over all keys, lse = log sum_s exp(lse_s) and o = sum_s exp(lse_s -
// lse) o_s: the block-wise update of "tm_flash_attention_math" ("The
// block-wise update, and the full algorithm": a new block rescales the old
// state by exp(m_old - m_new) and adds its own terms), applied to whole
// blocks' states in any order ("Proof of exactness").  A range that gave a row
// no visible key carries lse_s = -inf and weight zero.
//
// One warp per row: lanes split the d columns; the weights are computed once
// per row from the S partial LSEs (maximum first, so no exponent is positive).
#include "common.cuh"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ o_part,
                                                    const float* __restrict__ lse_part, int S,
                                                    long long rows, uint16_t* __restrict__ o,
                                                    float* __restrict__ lse) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;  // warp-uniform
  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lse_part[(size_t)s * rows + row]);
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, w));
  float sum = 0.f;
  if (mx != -INFINITY)
    for (int s = lane; s < S; s += 32) sum += ex2((lse_part[(size_t)s * rows + row] - mx) * kLog2e);
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, w);
  const bool any = sum > 0.f;
  const float L = any ? mx + lg2(sum) * kLn2 : -INFINITY;  // log sum_s exp(lse_s)
  constexpr int PER = D / 32;  // columns per lane
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  if (any) {
    for (int s = 0; s < S; ++s) {
      const float ls = lse_part[(size_t)s * rows + row];
      if (ls == -INFINITY) continue;  // warp-uniform: no key of this range was visible
      const float w = ex2((ls - L) * kLog2e);
      const float* src = o_part + ((size_t)s * rows + row) * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
      }
    }
  }
  uint32_t* dst = reinterpret_cast<uint32_t*>(o + row * D + lane * PER);
#pragma unroll
  for (int i = 0; i < PER; i += 2) dst[i / 2] = pack_bf16x2(acc[i], acc[i + 1]);
  if (lane == 0) lse[row] = L;
}

}  // namespace

cudaError_t launch_merge(const float* o_part, const float* lse_part, int n_splits, long long rows,
                         int d, void* o, float* lse, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (d == 128)
    merge_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(o_part, lse_part, n_splits, rows,
                                                            static_cast<uint16_t*>(o), lse);
  else if (d == 64)
    merge_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(o_part, lse_part, n_splits, rows,
                                                           static_cast<uint16_t*>(o), lse);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace fattn
