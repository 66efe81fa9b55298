// Host side of the C ABI declared in include/attn_fwd.h: argument checks,
// TMA descriptors, the per-stream scheduling workspace, and the launches of
// the scheduler kernel (packed variable-length batches) and the persistent
// fused attention kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/attn_fwd.h"
#include "attn_fwd_kernel.cuh"
#include "attn_host.h"

namespace {

using attn::FwdCfg;
using attn::FwdParams;

thread_local int g_last_cuda_error = 0;
int g_last_error_site = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int major = 0, minor = 0;
  int* err = nullptr;  // [0] error bits, [1] site of an expired wait
};

struct StreamWorkspace {
  int* buf = nullptr;       // [0] entry count, [1] next-unit counter, [2] finished CTAs,
                            // [3] unused, [4..] (seq, q-block) pairs
  int64_t capacity = 0;     // entries
};

std::mutex g_mu;
std::map<int, DeviceState> g_dev;
std::map<std::pair<int, attn_stream_t>, StreamWorkspace> g_ws;

struct PartialWorkspace {
  float* buf = nullptr;  // split-KV partial O then LSE
  size_t capacity = 0;   // floats
};
std::map<std::pair<int, attn_stream_t>, PartialWorkspace> g_part;
EncodeTiledFn g_encode = nullptr;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return ATTN_ERR_CUDA;
}

int get_encode(EncodeTiledFn* out) {
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                      cudaEnableDefault, &q);
    if (e != cudaSuccess) return cuda_fail(e);
    if (q != cudaDriverEntryPointSuccess || !fn) return cuda_fail(cudaErrorSymbolNotFound);
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = g_encode;
  return ATTN_OK;
}

// Dynamic shared memory limits of every attention kernel instantiation.
cudaError_t set_smem_attributes() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_kernel<64, attn::kModePlain>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FwdCfg<64>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_kernel<128, attn::kModePlain>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FwdCfg<128>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_kernel<64, attn::kModeWindow>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FwdCfg<64>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_kernel<64, attn::kModeSplit>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FwdCfg<64>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_kernel<128, attn::kModeSplit>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FwdCfg<128>::kSmemBytes)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(attn::attn_fwd_kernel<128, attn::kModeWindow>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              FwdCfg<128>::kSmemBytes);
}

int device_state(int dev, DeviceState** out) {
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    cudaError_t e;
    if ((e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&st.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&st.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if (st.major != 10 || st.minor != 3) return ATTN_ERR_ARCH;
    if ((e = set_smem_attributes()) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMalloc(&st.err, 4 * sizeof(int))) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemset(st.err, 0, 4 * sizeof(int))) != cudaSuccess) return cuda_fail(e);
    st.ready = true;
  }
  *out = &st;
  return ATTN_OK;
}

int stream_workspace(int dev, attn_stream_t stream, int64_t entries, int** out) {
  StreamWorkspace& ws = g_ws[std::make_pair(dev, stream)];
  if (ws.capacity < entries || !ws.buf) {
    cudaError_t e;
    if (ws.buf) {
      // the old list may still be read by work queued on this stream
      if ((e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream))) != cudaSuccess)
        return cuda_fail(e);
      cudaFree(ws.buf);
      ws.buf = nullptr;
      ws.capacity = 0;
    }
    const int64_t cap = entries < 1024 ? 1024 : entries;
    if ((e = cudaMalloc(&ws.buf, (size_t)(4 + 2 * cap) * sizeof(int))) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaMemset(ws.buf, 0, 4 * sizeof(int))) != cudaSuccess) return cuda_fail(e);
    ws.capacity = cap;
  }
  *out = ws.buf;
  return ATTN_OK;
}

int partial_workspace(int dev, attn_stream_t stream, size_t floats, float** out) {
  PartialWorkspace& ws = g_part[std::make_pair(dev, stream)];
  if (ws.capacity < floats || !ws.buf) {
    cudaError_t e;
    if (ws.buf) {
      if ((e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream))) != cudaSuccess)
        return cuda_fail(e);
      cudaFree(ws.buf);
      ws.buf = nullptr;
      ws.capacity = 0;
    }
    if ((e = cudaMalloc(&ws.buf, floats * sizeof(float))) != cudaSuccess) return cuda_fail(e);
    ws.capacity = floats;
  }
  *out = ws.buf;
  return ATTN_OK;
}

// 3-D view [tokens, H, d] of a bf16 tensor; box = 128 tokens x 1 head x 64
// elements (128 bytes, the 128-byte swizzle span).
int make_map(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int64_t tokens, int H, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)attn::kBM};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

template <int D>
int launch_attn(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                const FwdParams& p, int grid, cudaStream_t s) {
  if (p.wl >= 0 || p.wr >= 0)
    attn::attn_fwd_kernel<D, attn::kModeWindow><<<grid, attn::kThreads, FwdCfg<D>::kSmemBytes, s>>>(mq, mk, mv, p);
  else
    attn::attn_fwd_kernel<D, attn::kModePlain><<<grid, attn::kThreads, FwdCfg<D>::kSmemBytes, s>>>(mq, mk, mv, p);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

}  // namespace

namespace {

int attn_fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int N, int d, float scale, int causal, int window_left, int window_right,
                  const int32_t* cu_seqlens, attn_stream_t stream, const attn_fwd_options* opts) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_SHAPE;
  if (window_left < -1 || window_right < -1) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
  if (!std::isfinite(scale)) return ATTN_ERR_SCALE;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_ALIGN;
  // token indices and the TMA outer extent stay within int32
  const int64_t tokens_bound = (int64_t)B * N;
  if (tokens_bound > INT32_MAX - 2 * attn::kBN || (int64_t)H * d > (1 << 20) || H > 65535)
    return ATTN_ERR_SHAPE;
  const int64_t nqb = (N + attn::kUnitRows - 1) / attn::kUnitRows;
  const int64_t units = (int64_t)B * nqb * H;
  if (units > INT32_MAX) return ATTN_ERR_SHAPE;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceState* ds = nullptr;
  int st = device_state(dev, &ds);
  if (st != ATTN_OK) return st;
  EncodeTiledFn enc = nullptr;
  if ((st = get_encode(&enc)) != ATTN_OK) return st;

  // The token extent of the TMA view is B*N.  Dense: exact.  Packed: an upper
  // bound of cu_seqlens[B] (every length <= N, checked on the device before
  // any load); the kernel never asks for a token at or past the end of its
  // sequence, so no copy reads beyond the caller's buffer.
  CUtensorMap mq, mk, mv;
  if ((st = make_map(enc, &mq, q, tokens_bound, H, d)) != ATTN_OK) return st;
  if ((st = make_map(enc, &mk, k, tokens_bound, H, d)) != ATTN_OK) return st;
  if ((st = make_map(enc, &mv, v, tokens_bound, H, d)) != ATTN_OK) return st;

  FwdParams p{};
  p.o = reinterpret_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.err = ds->err;
  p.B = B;
  p.H = H;
  p.N = N;
  p.causal = causal ? 1 : 0;
  p.wl = window_left;
  p.wr = window_right;
  p.scale = scale;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.timeout_ns = (opts && opts->wait_timeout_ns) ? opts->wait_timeout_ns : 2000000000ull;
  p.fault_inject = opts ? opts->fault_inject : 0;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int grid = ds->sms;
  int* ws = nullptr;
  const int64_t max_entries = cu_seqlens ? (int64_t)B * nqb : 0;
  if ((st = stream_workspace(dev, stream, max_entries, &ws)) != ATTN_OK) return st;
  p.sched = ws + 1;
  if (cu_seqlens) {
    p.num_entries = ws;
    p.work = ws + 4;
    const int ncost = (int)std::min<int64_t>((N + attn::kBN - 1) / attn::kBN,
                                             attn::kMaxCostBuckets - 1);
    attn::build_worklist_kernel<<<1, 1024, (ncost + 1) * sizeof(int), s>>>(
        cu_seqlens, B, N, p.causal, p.wl, p.wr, ws + 4, ws, ds->err, (int)max_entries, ws + 1);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
  } else if (units < grid) {
    grid = (int)units;
  }
  if (opts && opts->max_ctas > 0 && opts->max_ctas < grid) grid = opts->max_ctas;
  return d == 64 ? launch_attn<64>(mq, mk, mv, p, grid, s) : launch_attn<128>(mq, mk, mv, p, grid, s);
}

}  // namespace

extern "C" int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, float scale, int causal,
                           const int32_t* cu_seqlens, attn_stream_t stream,
                           const attn_fwd_options* opts) {
  return attn_fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, -1, -1, cu_seqlens, stream,
                       opts);
}

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int N, int d, float scale, int causal, const int32_t* cu_seqlens,
                        attn_stream_t stream) {
  return attn_fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, -1, -1, cu_seqlens, stream,
                       nullptr);
}

extern "C" int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int H, int N, int d, float scale, int causal,
                               int window_left, int window_right, const int32_t* cu_seqlens,
                               attn_stream_t stream) {
  return attn_fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, window_left, window_right,
                       cu_seqlens, stream, nullptr);
}

extern "C" int attn_last_device_error(attn_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
  auto it = g_dev.find(dev);
  if (it == g_dev.end() || !it->second.ready) {
    g_last_error_site = 0;
    return ATTN_OK;
  }
  int h[2] = {0, 0};
  if ((e = cudaMemcpy(h, it->second.err, sizeof h, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaMemset(it->second.err, 0, sizeof h)) != cudaSuccess) return cuda_fail(e);
  g_last_error_site = h[1];
  if (h[0] & attn::kErrTimeout) return ATTN_ERR_DEVICE_TIMEOUT;
  if (h[0] & attn::kErrSeqlens) return ATTN_ERR_SEQLENS;
  if (h[0] & attn::kErrWorklist) return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

extern "C" int attn_last_error_site(void) { return g_last_error_site; }

extern "C" int attn_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "null pointer";
    case ATTN_ERR_SHAPE: return "bad shape";
    case ATTN_ERR_HEADDIM: return "head dim must be 64 or 128";
    case ATTN_ERR_ALIGN: return "misaligned pointer";
    case ATTN_ERR_SCALE: return "scale is not finite";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case ATTN_ERR_SEQLENS: return "invalid cu_seqlens";
    case ATTN_ERR_ARCH: return "device is not sm_103";
    case ATTN_ERR_SCRATCH: return "problem larger than the fixed scratch of attn_fwd_noalloc";
    default: return "unknown status";
  }
}

// ---------------------------------------------------------------------------
// attn_fwd_noalloc: the same forward pass without any device allocation, for
// callers that cannot call cudaMalloc.  Its scratch is the file-scope array
// below: error bits, error site, entry count, then the (sequence, q-block)
// pairs of a packed batch.  Every call shares it.
namespace {

constexpr int kNoAllocMaxEntries = 1 << 16;
constexpr int kNoAllocHeader = 8;  // [0] error bits, [1] error site, [2] entry count,
                                   // [3] next-unit counter, [4] finished CTAs
constexpr int kNoAllocScratchInts = kNoAllocHeader + 2 * kNoAllocMaxEntries;

static __device__ __align__(256) int g_noalloc_scratch[kNoAllocScratchInts];

struct NoAllocDevice {
  bool ready = false;
  int sms = 0;
  int* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::map<int, NoAllocDevice> g_noalloc_dev;

// Once per device, with that device current: kernel attributes and the device
// address of the scratch array (the host-side name is only a stand-in).
int noalloc_setup(int dev, NoAllocDevice** out) {
  NoAllocDevice& st = g_noalloc_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    cudaError_t e;
    if ((e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if (major != 10 || minor != 3) return ATTN_ERR_ARCH;
    if ((e = set_smem_attributes()) != cudaSuccess) return cuda_fail(e);
    void* ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess) return cuda_fail(e);
    st.scratch = static_cast<int*>(ptr);
    st.ready = true;
  }
  *out = &st;
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int N, int d, float scale, int causal,
                                const int32_t* cu_seqlens, attn_stream_t stream) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
  if (!std::isfinite(scale)) return ATTN_ERR_SCALE;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_ALIGN;
  const int64_t tokens_bound = (int64_t)B * N;
  if (tokens_bound > INT32_MAX - 2 * attn::kBN || (int64_t)H * d > (1 << 20) || H > 65535)
    return ATTN_ERR_SHAPE;
  const int64_t nqb = (N + attn::kUnitRows - 1) / attn::kUnitRows;
  const int64_t entries = (int64_t)B * nqb;
  if (entries > kNoAllocMaxEntries) return ATTN_ERR_SCRATCH;
  const int64_t units = entries * H;
  if (units > INT32_MAX) return ATTN_ERR_SHAPE;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  NoAllocDevice* nd = nullptr;
  int st = noalloc_setup(dev, &nd);
  if (st != ATTN_OK) return st;
  EncodeTiledFn enc = nullptr;
  if ((st = get_encode(&enc)) != ATTN_OK) return st;
  CUtensorMap mq, mk, mv;
  if ((st = make_map(enc, &mq, q, tokens_bound, H, d)) != ATTN_OK) return st;
  if ((st = make_map(enc, &mk, k, tokens_bound, H, d)) != ATTN_OK) return st;
  if ((st = make_map(enc, &mv, v, tokens_bound, H, d)) != ATTN_OK) return st;

  int* scratch = nd->scratch;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the error word and the entry count must start at zero on every call
  if ((e = cudaMemsetAsync(scratch, 0, kNoAllocHeader * sizeof(int), s)) != cudaSuccess)
    return cuda_fail(e);

  FwdParams p{};
  p.o = reinterpret_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.err = scratch;
  p.sched = scratch + 3;
  p.B = B;
  p.H = H;
  p.N = N;
  p.causal = causal ? 1 : 0;
  p.wl = -1;
  p.wr = -1;
  p.scale = scale;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.timeout_ns = 2000000000ull;
  p.fault_inject = 0;

  int grid = nd->sms;
  if (cu_seqlens) {
    p.num_entries = scratch + 2;
    p.work = scratch + kNoAllocHeader;
    const int ncost = (int)std::min<int64_t>((N + attn::kBN - 1) / attn::kBN,
                                             attn::kMaxCostBuckets - 1);
    attn::build_worklist_kernel<<<1, 1024, (ncost + 1) * sizeof(int), s>>>(
        cu_seqlens, B, N, p.causal, p.wl, p.wr, scratch + kNoAllocHeader, scratch + 2, scratch,
        (int)entries, scratch + 3);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
  } else if (units < grid) {
    grid = (int)units;
  }
  return d == 64 ? launch_attn<64>(mq, mk, mv, p, grid, s) : launch_attn<128>(mq, mk, mv, p, grid, s);
}

// ---------------------------------------------------------------------------
// attn_fwd_kvsplit: queries and keys of different lengths (bottom-right
// causal alignment), the visible KV tiles of every query block cut into
// ranges processed by separate units, then merged by the combine kernel.
extern "C" int attn_fwd_kvsplit(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int Nq, int Nk, int d, float scale, int causal,
                                int num_splits, attn_stream_t stream) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || num_splits < 0 || num_splits > 256)
    return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
  if (!std::isfinite(scale)) return ATTN_ERR_SCALE;
  if (B == 0 || H == 0 || Nq == 0) return ATTN_OK;
  if (Nk == 0 || (causal && Nq > Nk)) return ATTN_ERR_SHAPE;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_ALIGN;
  const int64_t q_tokens = (int64_t)B * Nq, k_tokens = (int64_t)B * Nk;
  if (q_tokens > INT32_MAX - 2 * attn::kBN || k_tokens > INT32_MAX - 2 * attn::kBN ||
      (int64_t)H * d > (1 << 20) || H > 65535)
    return ATTN_ERR_SHAPE;
  const int64_t nqb = (Nq + attn::kUnitRows - 1) / attn::kUnitRows;
  const int64_t base_units = (int64_t)B * nqb * H;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceState* ds = nullptr;
  int st = device_state(dev, &ds);
  if (st != ATTN_OK) return st;
  EncodeTiledFn enc = nullptr;
  if ((st = get_encode(&enc)) != ATTN_OK) return st;

  int S = num_splits;
  if (S == 0) {
    // The number of ranges with the shortest estimated makespan: units of
    // equal cost run in ceil(units / SMs) rounds of ceil(tiles / S) KV tiles
    // each; every extra range adds about a quarter tile of partial-result
    // traffic and merge work.  At most one range per KV tile, at most 64.
    const int64_t tiles = (Nk + attn::kBN - 1) / attn::kBN;
    double best = 0.0;
    for (int64_t c = 1; c <= std::min<int64_t>(tiles, 64); ++c) {
      const int64_t rounds = (base_units * c + ds->sms - 1) / ds->sms;
      const double t = (double)rounds * (double)((tiles + c - 1) / c) + 0.25 * (double)(c - 1);
      if (c == 1 || t < best) {
        best = t;
        S = (int)c;
      }
    }
  }
  const int64_t units = base_units * S;
  const int64_t combine_blocks = (q_tokens * H * 32 + 255) / 256;
  if (units > INT32_MAX || combine_blocks > INT32_MAX) return ATTN_ERR_SHAPE;

  CUtensorMap mq, mk, mv;
  if ((st = make_map(enc, &mq, q, q_tokens, H, d)) != ATTN_OK) return st;
  if ((st = make_map(enc, &mk, k, k_tokens, H, d)) != ATTN_OK) return st;
  if ((st = make_map(enc, &mv, v, k_tokens, H, d)) != ATTN_OK) return st;

  int* ws = nullptr;
  if ((st = stream_workspace(dev, stream, 0, &ws)) != ATTN_OK) return st;
  float* part = nullptr;
  const size_t o_floats = (size_t)S * q_tokens * H * d;
  const size_t lse_floats = (size_t)S * B * H * Nq;
  if ((st = partial_workspace(dev, stream, o_floats + lse_floats, &part)) != ATTN_OK) return st;

  FwdParams p{};
  p.o = reinterpret_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.err = ds->err;
  p.sched = ws + 1;
  p.B = B;
  p.H = H;
  p.N = Nq;
  p.Nk = Nk;
  p.q_off = causal ? Nk - Nq : 0;
  p.num_splits = S;
  p.o_part = part;
  p.lse_part = part + o_floats;
  p.causal = causal ? 1 : 0;
  p.wl = -1;
  p.wr = -1;
  p.scale = scale;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.timeout_ns = 2000000000ull;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int grid = (int)std::min<int64_t>(units, ds->sms);
  if (d == 64)
    attn::attn_fwd_kernel<64, attn::kModeSplit><<<grid, attn::kThreads, FwdCfg<64>::kSmemBytes, s>>>(
        mq, mk, mv, p);
  else
    attn::attn_fwd_kernel<128, attn::kModeSplit><<<grid, attn::kThreads, FwdCfg<128>::kSmemBytes, s>>>(
        mq, mk, mv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
  const int blocks = (int)combine_blocks;
  if (d == 64)
    attn::attn_combine_kernel<64><<<blocks, 256, 0, s>>>(p.o_part, p.lse_part,
                                                         reinterpret_cast<__nv_bfloat16*>(o), lse, B, H,
                                                         Nq, S);
  else
    attn::attn_combine_kernel<128><<<blocks, 256, 0, s>>>(p.o_part, p.lse_part,
                                                          reinterpret_cast<__nv_bfloat16*>(o), lse, B, H,
                                                          Nq, S);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
  return ATTN_OK;
}

// ---------------------------------------------------------------------------
// Services shared with the backward's host code (attn_host.h).
namespace attn_host {

std::mutex& lib_mutex() { return g_mu; }

int lib_cuda_fail(cudaError_t e) { return cuda_fail(e); }

int lib_device(int* dev, int* sms, int** err) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceState* ds = nullptr;
  const int st = device_state(*dev, &ds);
  if (st != ATTN_OK) return st;
  *sms = ds->sms;
  *err = ds->err;
  return ATTN_OK;
}

int lib_make_map(CUtensorMap* map, const void* ptr, int64_t tokens, int H, int d) {
  EncodeTiledFn enc = nullptr;
  const int st = get_encode(&enc);
  if (st != ATTN_OK) return st;
  return make_map(enc, map, ptr, tokens, H, d);
}

}  // namespace attn_host
