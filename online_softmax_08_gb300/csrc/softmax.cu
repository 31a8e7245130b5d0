// softmax.cu -- row-wise softmax with the online normaliser, one CTA per row.
//
// The running pair (m, l) of "FlashAttention tiles exact softmax without
// materializing the score matrix" ("The online softmax recurrence"): m is the
// largest value seen so far and l the sum of exp(x - m) over the values seen;
// when a larger value arrives, l is rescaled by exp(m_old - m_new).  Each
// thread runs the recurrence over its own elements; the threads' pairs are
// then combined with the same rule (two states (m1, l1), (m2, l2) merge into
// m = max(m1, m2), l = l1 exp(m1 - m) + l2 exp(m2 - m)), and y = exp(x - m) / l.
//
// HBM-bound.  A row of up to kSmemCols fp32 values is staged in shared memory
// while the statistics are formed, so it is read from HBM once: 8 bytes of
// traffic per element.  A longer row is read twice (12 bytes per element).
// Loads and stores are 16-byte vectors when the row length allows.
#include "common.cuh"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int kThreads = 1024;
constexpr int kBatch = 4;  // 16-byte loads in flight per thread (64 KB per CTA)
constexpr int kSmemCols = 48 * 1024;  // 192 KB of fp32
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct MaxSum {
  float m, l;
};

// Online update of (m, l) by one value.
__device__ __forceinline__ void push(MaxSum& s, float x) {
  if (x > s.m) {
    s.l = s.l * ex2((s.m - x) * kLog2e) + 1.f;  // exp(-inf) = 0 on the first value
    s.m = x;
  } else {
    s.l += ex2((x - s.m) * kLog2e);  // callers skip x = -inf (exp2 of -inf - -inf is nan)
  }
}
__device__ __forceinline__ void push4(MaxSum& s, float4 v) {
  const float m4 = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
  if (m4 == -INFINITY) return;  // nothing visible in these four values
  if (m4 > s.m) {
    s.l = s.m == -INFINITY ? 0.f : s.l * ex2((s.m - m4) * kLog2e);
    s.m = m4;
  }
  const float mm = s.m * kLog2e;
  s.l += ex2(fmaf(v.x, kLog2e, -mm)) + ex2(fmaf(v.y, kLog2e, -mm)) +
         ex2(fmaf(v.z, kLog2e, -mm)) + ex2(fmaf(v.w, kLog2e, -mm));
}
__device__ __forceinline__ MaxSum merge(MaxSum a, MaxSum b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return MaxSum{m, 0.f};
  return MaxSum{m, a.l * ex2((a.m - m) * kLog2e) + b.l * ex2((b.m - m) * kLog2e)};
}

// (m, l) of the whole CTA, returned to every thread.
__device__ MaxSum block_merge(MaxSum s, MaxSum* red) {
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) {
    MaxSum o{__shfl_xor_sync(0xffffffffu, s.m, w), __shfl_xor_sync(0xffffffffu, s.l, w)};
    s = merge(s, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = s;
  __syncthreads();
  if (warp == 0) {
    s = lane < kThreads / 32 ? red[lane] : MaxSum{-INFINITY, 0.f};
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) {
      MaxSum o{__shfl_xor_sync(0xffffffffu, s.m, w), __shfl_xor_sync(0xffffffffu, s.l, w)};
      s = merge(s, o);
    }
    if (lane == 0) red[kThreads / 32] = s;
  }
  __syncthreads();
  const MaxSum r = red[kThreads / 32];
  __syncthreads();  // red is reused by the next row
  return r;
}

// x and y may be the same array: every element is read before the same thread
// writes it, so no __restrict__ on them.
//
// Staged rows with 16-byte elements (the common case) are software-pipelined
// over the CTA's rows: thread t owns the same shared slots in every row, so
// while it writes row r from its slots it loads row r + gridDim.x, overwrites
// the slots it has just consumed and starts that row's statistics, and the
// HBM reads of the next row overlap the writes of this one.
__global__ void __launch_bounds__(kThreads) softmax_rows_kernel(const float* x, float* y,
                                                                float* __restrict__ lse,
                                                                long long rows, int cols,
                                                                int staged) {
  extern __shared__ float4 srow[];  // the staged row (when staged != 0)
  __shared__ MaxSum red[kThreads / 32 + 1];
  const bool vec = (cols & 3) == 0;  // 16-byte rows (x, y are 16-byte aligned)
  const int n4 = cols >> 2;
  auto finish = [&](long long r, MaxSum t, float& inv_l, float& mm, bool& any) {
    any = t.l > 0.f;
    inv_l = any ? 1.f / t.l : 0.f;
    mm = t.m * kLog2e;
    if (lse && threadIdx.x == 0) lse[r] = any ? t.m + lg2(t.l) * kLn2 : -INFINITY;
  };
  auto out4 = [&](float4 v, float inv_l, float mm, bool any) {
    float4 o;
    o.x = any ? ex2(fmaf(v.x, kLog2e, -mm)) * inv_l : 0.f;
    o.y = any ? ex2(fmaf(v.y, kLog2e, -mm)) * inv_l : 0.f;
    o.z = any ? ex2(fmaf(v.z, kLog2e, -mm)) * inv_l : 0.f;
    o.w = any ? ex2(fmaf(v.w, kLog2e, -mm)) * inv_l : 0.f;
    return o;
  };

  if (vec && staged) {
    long long r = blockIdx.x;
    if (r >= rows) return;
    MaxSum s{-INFINITY, 0.f};
    {  // prologue: stage the first row, forming its statistics
      const float4* x4 = reinterpret_cast<const float4*>(x + (size_t)r * cols);
      for (int base = threadIdx.x; base < n4; base += kBatch * kThreads) {
        float4 v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int i = base + j * kThreads;
          v[j] = i < n4 ? __ldcs(x4 + i)
                        : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int i = base + j * kThreads;
          if (i < n4) srow[i] = v[j];
          push4(s, v[j]);  // the -inf padding changes nothing
        }
      }
    }
    for (; r < rows; r += gridDim.x) {
      const MaxSum t = block_merge(s, red);
      float inv_l, mm;
      bool any;
      finish(r, t, inv_l, mm, any);
      const long long rn = r + gridDim.x;
      const bool next = rn < rows;
      const float4* xn4 = reinterpret_cast<const float4*>(x + (size_t)(next ? rn : r) * cols);
      float4* y4 = reinterpret_cast<float4*>(y + (size_t)r * cols);
      s = MaxSum{-INFINITY, 0.f};
      for (int base = threadIdx.x; base < n4; base += kBatch * kThreads) {
        float4 v[kBatch];
        if (next) {
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int i = base + j * kThreads;
            v[j] = i < n4 ? __ldcs(xn4 + i)
                          : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int i = base + j * kThreads;
          if (i < n4) {
            __stcs(y4 + i, out4(srow[i], inv_l, mm, any));
            if (next) srow[i] = v[j];  // this thread's own slot, just consumed
          }
          if (next) push4(s, v[j]);
        }
      }
    }
    return;
  }

  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const float* xr = x + (size_t)r * cols;
    float* yr = y + (size_t)r * cols;
    MaxSum s{-INFINITY, 0.f};
    // pass 1: the online statistics (staging the row when it fits)
    if (vec) {
      // kBatch independent 16-byte loads per thread before they are consumed, so
      // about 64 KB per CTA is in flight (one load at a time left HBM at 44 %;
      // 1024 threads x 4 loads measured faster than 512 x 8)
      const float4* x4 = reinterpret_cast<const float4*>(xr);
      for (int base = threadIdx.x; base < n4; base += kBatch * kThreads) {
        float4 v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int i = base + j * kThreads;
          v[j] = i < n4 ? __ldcs(x4 + i)  // streamed: no reuse beyond this row
                        : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) push4(s, v[j]);  // the -inf padding changes nothing
      }
    } else {
      float* sr = reinterpret_cast<float*>(srow);
      for (int i = threadIdx.x; i < cols; i += kThreads) {
        const float v = __ldcs(xr + i);
        if (staged) sr[i] = v;
        if (v != -INFINITY) push(s, v);
      }
    }
    const MaxSum t = block_merge(s, red);
    float inv_l, mm;
    bool any;
    finish(r, t, inv_l, mm, any);
    // pass 2: y = exp(x - m) / l, from shared memory or a second read
    if (vec) {
      const float4* x4 = reinterpret_cast<const float4*>(xr);
      float4* y4 = reinterpret_cast<float4*>(yr);
      for (int base = threadIdx.x; base < n4; base += kBatch * kThreads) {
        float4 v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int i = base + j * kThreads;
          if (i < n4) v[j] = __ldcs(x4 + i);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int i = base + j * kThreads;
          if (i < n4) __stcs(y4 + i, out4(v[j], inv_l, mm, any));
        }
      }
    } else {
      const float* sr = reinterpret_cast<const float*>(srow);
      for (int i = threadIdx.x; i < cols; i += kThreads) {
        const float v = staged ? sr[i] : __ldcs(xr + i);
        __stcs(yr + i, any ? ex2(fmaf(v, kLog2e, -mm)) * inv_l : 0.f);
      }
    }
    __syncthreads();  // the staged row is overwritten by the next one
  }
}

}  // namespace

cudaError_t launch_softmax_rows(const float* x, float* y, float* lse, long long rows, int cols,
                                int n_sm, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int staged = cols <= kSmemCols ? 1 : 0;
  const size_t smem = staged ? (size_t)((cols + 3) & ~3) * sizeof(float) : 0;
  static unsigned long long prepared[64];
  cudaError_t e = prepare_once(prepared, [] {
    return cudaFuncSetAttribute(softmax_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(kSmemCols * sizeof(float)));
  });
  if (e != cudaSuccess) return e;
  // persistent: as many CTAs as fit (by shared memory) on every SM, rows strided
  const int per_sm = staged ? (int)max((size_t)1, (size_t)(220 * 1024) / (smem + 1024)) : 2;
  long long grid = (long long)n_sm * min(per_sm, 2048 / kThreads);
  if (grid > rows) grid = rows;
  softmax_rows_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(x, y, lse, rows, cols, staged);
  return cudaGetLastError();
}

}  // namespace fattn
