// api.cu -- the C-ABI of libfattn: argument checks, TMA descriptors, launches.
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "../../include/fattn.h"
#include "common.cuh"
#include "ptx.cuh"

namespace fattn {
namespace {

__device__ unsigned int g_error_word;  // first in-kernel wait that ran out (0 = none)

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  unsigned long long ctx = 0;   // context the entry was filled in (0: not yet)
  bool supported = false;
  unsigned int* err = nullptr;  // device address of g_error_word
  int n_sm = 0;                 // streaming multiprocessors
  long long l2_bytes = 0;       // L2 cache size
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& info = g_dev[dev];
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || info.ctx != ctx) {
    int major = 0, minor = 0, l2 = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FATTN_ERR_CUDA;
    info.supported = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&info.n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return FATTN_ERR_CUDA;
    info.l2_bytes = l2;
    // the symbol lookup also makes the device's primary context current
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_error_word) != cudaSuccess) return FATTN_ERR_CUDA;
    info.err = static_cast<unsigned int*>(addr);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return FATTN_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    info.ctx = current_context_id();
  }
  if (!info.supported) return FATTN_ERR_UNSUPPORTED;
  *out = &info;
  return FATTN_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D map over a [BH, N, inner] tensor (inner contiguous), box {box0, box1, 1}.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes,
              long long inner, long long N, long long BH, int box0, int box1,
              CUtensorMapSwizzle swz) {
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)(inner * elem_bytes), (cuuint64_t)(inner * N * elem_bytes)};
  cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_bf16_map(CUtensorMap* m, const void* base, int d, long long N, long long BH, int rows) {
  return make_map(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64, rows,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

int check_common(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FATTN_ERR_INVALID_ARG;
  if ((long long)B * H * N >= (1LL << 31)) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  return FATTN_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Heads per group of the dense grid order: as many as fit their tensors
// (bytes_per_head) in a quarter of L2, the share measured best for both
// kernels (an eighth and a half were slower), at least one.
int l2_group(const DeviceInfo& dev, long long bytes_per_head) {
  return (int)std::max<long long>(1, (dev.l2_bytes / 4) / bytes_per_head);
}

}  // namespace

unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static const GetCurrent get_current = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
                       cudaSuccess &&
                   q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<GetCurrent>(fn)
               : nullptr;
  }();
  static const GetId get_id = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                       cudaSuccess &&
                   q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<GetId>(fn)
               : nullptr;
  }();
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c ||
      get_id(c, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

int device_sm_count() {
  DeviceInfo* dev = nullptr;
  return current_device(&dev) == FATTN_OK ? dev->n_sm : 0;
}

long long device_l2_bytes() {
  DeviceInfo* dev = nullptr;
  return current_device(&dev) == FATTN_OK ? dev->l2_bytes : 0;
}

namespace {
bool debug_enabled() {
  static const bool on = [] {
    const char* v = getenv("FATTN_DEBUG");
    return v && *v && strcmp(v, "0") != 0;
  }();
  return on;
}
}  // namespace

int debug_post_call(int status, cudaStream_t stream) {
  if (status != FATTN_OK || !debug_enabled()) return status;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return FATTN_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return status;  // nothing has run yet
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FATTN_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess) return FATTN_ERR_CUDA;
  return word ? FATTN_ERR_TIMEOUT : FATTN_OK;
}

}  // namespace fattn

using namespace fattn;

namespace fattn {
namespace {

// Geometry of one call: the TMA maps span `map_rows` rows of `map_z` slices
// ([B*H, N, d] dense, [H, T, d] varlen); kernels see p.N = the (longest)
// sequence length and the varlen table, if any.
struct Geometry {
  long long map_rows;
  long long map_z;
  int BH;        // units the dense grid iterates over (B*H; H when varlen)
  int N;         // sequence length, or the longest one when varlen
  Varlen vl;
};

int run_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int d, float scale,
            int causal, const Geometry& g, unsigned long long* tile_counts, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FATTN_ERR_INVALID_ARG;
  if (tile_counts && (reinterpret_cast<uintptr_t>(tile_counts) & 7u)) return FATTN_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  const int st = current_device(&dev);
  if (st != FATTN_OK) return st;
  CUtensorMap tq, tk, tv, to;
  if (!make_bf16_map(&tq, q, d, g.map_rows, g.map_z, 128) ||
      !make_bf16_map(&tk, k, d, g.map_rows, g.map_z, 128) ||
      !make_bf16_map(&tv, v, d, g.map_rows, g.map_z, 128) ||
      !make_bf16_map(&to, o, d, g.map_rows, g.map_z, 128))
    return FATTN_ERR_CUDA;
  FwdParams p{};
  p.BH = g.BH;
  p.N = g.N;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.lse = lse;
  p.tiles = tile_counts;
  p.err = dev->err;
  p.vl = g.vl;
  p.o = static_cast<uint16_t*>(o);
  // dense: groups of heads whose K and V (4 N d bytes a head) fit in a quarter of L2
  p.group = l2_group(*dev, 4LL * g.N * d);
  cudaError_t e = launch_fwd(d, tq, tk, tv, to, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

size_t workspace_bytes_for_rows(long long rows, int d) {
  return align256((size_t)rows * d * sizeof(float)) + align256((size_t)rows * sizeof(float));
}

// The kernels of one backward call on a workspace that is already in place.
int launch_bwd_all(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, int d, float scale, int causal,
                   const Geometry& g, const DeviceInfo& dev, void* workspace,
                   void* const* phase_events, cudaStream_t s) {
  const long long rows = g.map_rows * g.map_z;
  float* dq_acc = static_cast<float*>(workspace);
  float* delta = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          align256((size_t)rows * d * sizeof(float)));
  int bq = 0, bk = 0;
  fattn_tile_sizes(d, 1, &bq, &bk);
  const long long R = g.map_rows, Z = g.map_z;
  CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
  if (!make_bf16_map(&tq, q, d, R, Z, bq) || !make_bf16_map(&tdo, dout, d, R, Z, bq) ||
      !make_bf16_map(&tk, k, d, R, Z, bk) || !make_bf16_map(&tv, v, d, R, Z, bk) ||
      !make_bf16_map(&tdk, dk, d, R, Z, bk) || !make_bf16_map(&tdv, dv, d, R, Z, bk))
    return FATTN_ERR_CUDA;
  // dQ accumulator: fp32, add-reduced one box of query rows at a time
  const DqBox qb = bwd_dq_box(d);
  if (!make_map(&tdq, dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, R, Z, qb.cols, qb.rows,
                qb.sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE))
    return FATTN_ERR_CUDA;
  auto mark = [&](int i) {
    return !phase_events ||
           cudaEventRecord(static_cast<cudaEvent_t>(phase_events[i]), s) == cudaSuccess;
  };
  if (!mark(0)) return FATTN_ERR_CUDA;
  if (launch_bwd_preprocess(o, dout, delta, dq_acc, rows, d, dev.n_sm, s) != cudaSuccess)
    return FATTN_ERR_CUDA;
  if (!mark(1)) return FATTN_ERR_CUDA;
  BwdParams p{};
  p.BH = g.BH;
  p.N = g.N;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.lse = lse;
  p.delta = delta;
  p.dq_acc = dq_acc;
  p.err = dev.err;
  p.vl = g.vl;
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  // dense: groups of heads whose Q, dO (bf16) and dQ accumulator (fp32), 8 N d
  // bytes a head, fit in a quarter of L2
  p.group = l2_group(dev, 8LL * g.N * d);
  cudaError_t e = launch_bwd_main(d, tq, tk, tv, tdo, tdk, tdv, tdq, p, s);
  if (e == cudaErrorNotSupported) return FATTN_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return FATTN_ERR_CUDA;
  if (!mark(2)) return FATTN_ERR_CUDA;
  if (launch_bwd_convert(dq_acc, dq, rows * d, scale, dev.n_sm, s) != cudaSuccess)
    return FATTN_ERR_CUDA;
  if (!mark(3)) return FATTN_ERR_CUDA;
  return FATTN_OK;
}

int run_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
            const void* dout, void* dq, void* dk, void* dv, int d, float scale, int causal,
            const Geometry& g, void* workspace, size_t workspace_bytes,
            void* const* phase_events, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FATTN_ERR_INVALID_ARG;
  const long long rows = g.map_rows * g.map_z;
  const size_t need = workspace_bytes_for_rows(rows, d);
  if (workspace && ((reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need))
    return FATTN_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  const int st = current_device(&dev);
  if (st != FATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (workspace)
    return launch_bwd_all(q, k, v, o, lse, dout, dq, dk, dv, d, scale, causal, g, *dev, workspace,
                          phase_events, s);
  // no workspace from the caller: stream-ordered scratch, allocated and freed
  // on `stream` around the kernels (256 spare bytes keep the 256-byte alignment)
  void* raw = nullptr;
  if (cudaMallocAsync(&raw, need + 256, s) != cudaSuccess) {
    cudaGetLastError();  // an allocation failure is not sticky: clear it
    return FATTN_ERR_CUDA;
  }
  void* ws = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(raw) + 255u) & ~(uintptr_t)255u);
  const int r = launch_bwd_all(q, k, v, o, lse, dout, dq, dk, dv, d, scale, causal, g, *dev, ws,
                               phase_events, s);
  if (cudaFreeAsync(raw, s) != cudaSuccess) return FATTN_ERR_CUDA;
  return r;
}

Geometry dense_geometry(int B, int H, int N) {
  return Geometry{N, (long long)B * H, B * H, N, Varlen{nullptr, 0, 0, 0}};
}

// Varlen arguments: B sequences, H heads, T total rows, the longest sequence
// max_seqlen; cu_seqlens is checked entry by entry on the device.
int check_varlen(const int* cu_seqlens, int B, int H, int max_seqlen, int T, int d, float scale) {
  if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return FATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || max_seqlen < 0 || T < 0 || max_seqlen > T) return FATTN_ERR_INVALID_ARG;
  if ((long long)H * T >= (1LL << 31)) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  return FATTN_OK;
}

}  // namespace
}  // namespace fattn

extern "C" int fattn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int N, int d, float scale, int causal,
                            unsigned long long* tile_counts, void* stream) {
  const int st = check_common(B, H, N, d, scale);
  if (st != FATTN_OK) return st;
  return debug_post_call(
      run_fwd(q, k, v, o, lse, d, scale, causal, dense_geometry(B, H, N), tile_counts, stream),
      static_cast<cudaStream_t>(stream));
}

extern "C" int fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, float scale, int causal, void* stream) {
  return fattn_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, nullptr, stream);
}

extern "C" int fattn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                const int* cu_seqlens, int B, int H, int max_seqlen, int total,
                                int d, float scale, int causal, void* stream) {
  const int st = check_varlen(cu_seqlens, B, H, max_seqlen, total, d, scale);
  if (st != FATTN_OK) return st;
  if (total == 0 || max_seqlen == 0) return FATTN_OK;  // no rows: nothing to compute
  const Geometry g{total, H, H, max_seqlen, Varlen{cu_seqlens, B, H, total}};
  return debug_post_call(run_fwd(q, k, v, o, lse, d, scale, causal, g, nullptr, stream),
                         static_cast<cudaStream_t>(stream));
}

namespace fattn {
namespace {

// Key ranges of a split call: n_tiles 128-key tiles cut into ranges of
// tiles_per_split tiles.  n_splits = 0 picks enough ranges for about ten
// waves of CTAs over the device's n_sm SMs (measured best at B4 H32 Nq1
// Nkv32768: 94 % of the copy bandwidth, against 90 % for one wave), keeping at
// least four tiles per range; a request is capped at one range per tile and
// empty ranges are dropped.
struct SplitPlan {
  int n_splits;
  int tiles_per_split;
};
SplitPlan plan_splits(long long units, int Nq, int Nkv, int n_splits, int n_sm) {
  const int n_tiles = (Nkv + 127) / 128;
  const long long n_qb = (Nq + 255) / 256;
  long long want = n_splits;
  if (want <= 0) {
    const long long ctas = units * n_qb;
    want = (10LL * n_sm + ctas - 1) / ctas;
    if (want > n_tiles / 4) want = n_tiles / 4;
  }
  if (want > n_tiles) want = n_tiles;
  if (want < 1) want = 1;
  const int tps = (int)((n_tiles + want - 1) / want);
  return SplitPlan{(n_tiles + tps - 1) / tps, tps};
}

int check_decode(int B, int H, int Nq, int Nkv, int d, float scale, int n_splits) {
  if (B < 1 || H < 1 || Nq < 1 || Nkv < Nq || n_splits < 0) return FATTN_ERR_INVALID_ARG;
  if ((long long)B * H * Nkv >= (1LL << 31)) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  return FATTN_OK;
}

size_t decode_ws_bytes(long long rows, int d, int S) {
  return align256((size_t)S * rows * d * sizeof(float)) + align256((size_t)S * rows * sizeof(float));
}

}  // namespace
}  // namespace fattn

extern "C" int fattn_decode_splits(int B, int H, int Nq, int Nkv, int d, int n_splits) {
  if (check_decode(B, H, Nq, Nkv, d, 1.f, n_splits) != FATTN_OK) return 0;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != FATTN_OK) return 0;
  return plan_splits((long long)B * H, Nq, Nkv, n_splits, dev->n_sm).n_splits;
}

extern "C" size_t fattn_decode_workspace_bytes(int B, int H, int Nq, int Nkv, int d,
                                               int n_splits) {
  if (check_decode(B, H, Nq, Nkv, d, 1.f, n_splits) != FATTN_OK) return 0;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != FATTN_OK) return 0;
  const SplitPlan sp = plan_splits((long long)B * H, Nq, Nkv, n_splits, dev->n_sm);
  return decode_ws_bytes((long long)B * H * Nq, d, sp.n_splits);
}

extern "C" int fattn_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int Nq, int Nkv, int d, float scale, int causal,
                            int n_splits, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_decode(B, H, Nq, Nkv, d, scale, n_splits);
  if (st != FATTN_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FATTN_ERR_INVALID_ARG;
  const long long BH = (long long)B * H, rows = BH * Nq;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FATTN_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  st = current_device(&dev);
  if (st != FATTN_OK) return st;
  const SplitPlan sp = plan_splits(BH, Nq, Nkv, n_splits, dev->n_sm);
  if (workspace_bytes < decode_ws_bytes(rows, d, sp.n_splits)) return FATTN_ERR_WORKSPACE;
  CUtensorMap tq, tk, tv;
  if (!make_bf16_map(&tq, q, d, Nq, BH, 128) || !make_bf16_map(&tk, k, d, Nkv, BH, 128) ||
      !make_bf16_map(&tv, v, d, Nkv, BH, 128))
    return FATTN_ERR_CUDA;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(
      static_cast<char*>(workspace) + align256((size_t)sp.n_splits * rows * d * sizeof(float)));
  FwdParams p{};
  p.BH = (int)BH;
  p.N = Nkv;
  p.Nq = Nq;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = dev->err;
  p.n_splits = sp.n_splits;
  p.tiles_per_split = sp.tiles_per_split;
  p.o_part = o_part;
  p.lse_part = lse_part;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_fwd_split(d, tq, tk, tv, tq, p, s) != cudaSuccess) return FATTN_ERR_CUDA;
  if (launch_merge(o_part, lse_part, sp.n_splits, rows, d, o, lse, s) != cudaSuccess)
    return FATTN_ERR_CUDA;
  return debug_post_call(FATTN_OK, s);
}

extern "C" int fattn_merge_partials(const float* o_part, const float* lse_part, int n_splits,
                                    long long rows, int d, void* o, float* lse, void* stream) {
  if (n_splits < 1 || rows < 1) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  if (!aligned16(o_part) || !aligned16(lse_part) || !aligned16(o) || !aligned16(lse))
    return FATTN_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  const int st = current_device(&dev);
  if (st != FATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return debug_post_call(
      launch_merge(o_part, lse_part, n_splits, rows, d, o, lse, s) == cudaSuccess ? FATTN_OK
                                                                                  : FATTN_ERR_CUDA,
      s);
}

extern "C" int fattn_softmax_rows(const float* x, float* y, float* lse, long long rows, int cols,
                                  void* stream) {
  if (rows < 1 || cols < 1) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FATTN_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  const int st = current_device(&dev);
  if (st != FATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return debug_post_call(
      launch_softmax_rows(x, y, lse, rows, cols, dev->n_sm, s) == cudaSuccess ? FATTN_OK
                                                                              : FATTN_ERR_CUDA,
      s);
}

extern "C" size_t fattn_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  return workspace_bytes_for_rows((long long)B * H * N, d);
}

extern "C" int fattn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv,
                            int B, int H, int N, int d, float scale, int causal, void* workspace,
                            size_t workspace_bytes, void* const* phase_events, void* stream) {
  const int st = check_common(B, H, N, d, scale);
  if (st != FATTN_OK) return st;
  return debug_post_call(run_bwd(q, k, v, o, lse, dout, dq, dk, dv, d, scale, causal,
                                 dense_geometry(B, H, N), workspace, workspace_bytes, phase_events,
                                 stream),
                         static_cast<cudaStream_t>(stream));
}

extern "C" int fattn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                const int* cu_seqlens, int B, int H, int max_seqlen, int total,
                                int d, float scale, int causal, void* workspace,
                                size_t workspace_bytes, void* stream) {
  const int st = check_varlen(cu_seqlens, B, H, max_seqlen, total, d, scale);
  if (st != FATTN_OK) return st;
  if (total == 0 || max_seqlen == 0) return FATTN_OK;  // no rows: nothing to compute
  const Geometry g{total, H, H, max_seqlen, Varlen{cu_seqlens, B, H, total}};
  return debug_post_call(run_bwd(q, k, v, o, lse, dout, dq, dk, dv, d, scale, causal, g, workspace,
                                 workspace_bytes, nullptr, stream),
                         static_cast<cudaStream_t>(stream));
}

extern "C" int fattn_bwd(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale, int causal, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return fattn_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                      workspace_bytes, nullptr, stream);
}

extern "C" int fattn_tile_sizes(int d, int pass, int* block_q, int* block_k) {
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  if (pass != 0 && pass != 1) return FATTN_ERR_INVALID_ARG;
  const int bq = 128, bk = 128;  // both passes, both head sizes
  if (block_q) *block_q = bq;
  if (block_k) *block_k = bk;
  return FATTN_OK;
}

namespace fattn {
namespace {
// One warp waits on an mbarrier that nothing ever completes, through the same
// bounded wait the attention kernels use, with a short limit (2^21 cycles,
// about 1 ms): the wait gives up, records ERR_SITE_CHECK | 1 in the error word
// and the kernel returns.
constexpr long long kCheckLimitCycles = 1ll << 21;
__global__ void wait_timeout_check_kernel(unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtx ctx{&abort_flag, err};
  mbar_wait<kCheckLimitCycles>(smem_u32(&bar), 0, ctx, ERR_SITE_CHECK | 0x01);
}
}  // namespace
}  // namespace fattn

extern "C" int fattn_check_wait_timeout(void* stream) {
  DeviceInfo* dev = nullptr;
  const int st = current_device(&dev);
  if (st != FATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fattn::wait_timeout_check_kernel<<<1, 32, 0, s>>>(dev->err);
  return debug_post_call(cudaGetLastError() == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA, s);
}

extern "C" int fattn_device_error(unsigned int* code, int clear) {
  if (!code) return FATTN_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return FATTN_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return FATTN_ERR_CUDA;
  *code = v;
  if (clear && v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess)
      return FATTN_ERR_CUDA;
  }
  return v ? FATTN_ERR_TIMEOUT : FATTN_OK;
}

extern "C" const char* fattn_status_string(int status) {
  switch (status) {
    case FATTN_OK: return "ok";
    case FATTN_ERR_INVALID_ARG: return "invalid argument";
    case FATTN_ERR_UNSUPPORTED: return "unsupported head size or device";
    case FATTN_ERR_CUDA: return "CUDA error";
    case FATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case FATTN_ERR_TIMEOUT: return "in-kernel wait timed out";
    default: return "unknown status";
  }
}
