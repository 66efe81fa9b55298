// Host side of the C ABI declared in include/attn_fwd.h: argument checks,
// TMA descriptors, the per-stream scheduling workspace, and the launches of
// the scheduler kernel (packed variable-length batches) and the persistent
// fused attention kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/attn_fp8.h"
#include "../../include/attn_fwd.h"
#include "attn_decode_kernel.cuh"
#include "attn_fp8_kernel.cuh"
#include "attn_fwd_kernel.cuh"
#include "attn_fwd_pair_kernel.cuh"
#include "attn_fwd_row_kernel.cuh"
#include "attn_fp8_row_kernel.cuh"
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
  int pair_clusters = 0;  // co-resident clusters of the pair kernel
  int major = 0, minor = 0;
  int* err = nullptr;  // [0] error bits, [1] site of an expired wait
};

struct StreamWorkspace {
  int* buf = nullptr;       // [0] entry count, [1] next-unit counter, [2] finished CTAs,
                            // [3] attn_fwd_decode's cu_seqlens_k check, [4..] (seq, q-block) pairs
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
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_kernel<64, attn::kModeSplitPair>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FwdCfg<64>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_kernel<128, attn::kModeSplitPair>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FwdCfg<128>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fp8_row_kernel<64>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::kFp8SmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fp8_row_kernel<128>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::kFp8SmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::fp8_quant_stage1_kernel<64>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::QuantCfg<64>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::fp8_quant_stage1_kernel<128>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::QuantCfg<128>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_row_kernel<64, attn::kModePlain>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::RowCfg<64>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_row_kernel<128, attn::kModePlain>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::RowCfg<128>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_row_kernel<64, attn::kModeWindow>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::RowCfg<64>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_row_kernel<128, attn::kModeWindow>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::RowCfg<128>::kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn::attn_fwd_pair_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::kPairSmemBytes)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(attn::attn_fwd_kernel<128, attn::kModeWindow>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              FwdCfg<128>::kSmemBytes);
}

// Clusters of the pair kernel that fit on the device at once (its persistent
// grid is twice this).
cudaError_t pair_cluster_count(int sms, int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sms & ~1), 1, 1);
  cfg.blockDim = dim3(attn::kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = attn::kPairSmemBytes;
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&n, attn::attn_fwd_pair_kernel, &cfg);
  if (e != cudaSuccess) return e;
  *out = n;
  return cudaSuccess;
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
    if ((e = pair_cluster_count(st.sms, &st.pair_clusters)) != cudaSuccess) return cuda_fail(e);
    if ((e = attn_host::lib_malloc(&st.err, 4 * sizeof(int))) != cudaSuccess) return cuda_fail(e);
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
      attn_host::lib_free(ws.buf);
      ws.buf = nullptr;
      ws.capacity = 0;
    }
    const int64_t cap = entries < 1024 ? 1024 : entries;
    if ((e = attn_host::lib_malloc(&ws.buf, (size_t)(4 + 2 * cap) * sizeof(int))) != cudaSuccess)
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
      attn_host::lib_free(ws.buf);
      ws.buf = nullptr;
      ws.capacity = 0;
    }
    if ((e = attn_host::lib_malloc(&ws.buf, floats * sizeof(float))) != cudaSuccess) return cuda_fail(e);
    ws.capacity = floats;
  }
  *out = ws.buf;
  return ATTN_OK;
}

// 3-D view [tokens, H, d] of a bf16 tensor; box = box_rows tokens (128 unless
// given) x 1 head x 64 elements (128 bytes, the 128-byte swizzle span).
int make_map(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int64_t tokens, int H, int d,
             int box_rows = attn::kBM) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The forward kernels' exponent scale c = scale * log2 e, at least the
// smallest normal float.  They form 2^(c s - c m) with masked logits s = -inf,
// and c = 0 (scale 0, or a scale whose product underflows) would make that
// NaN.  With c = 2^-126 every visible key gets 2^(c s - c m) = 1 within the
// ex2 approximation's error for |s| < 2^100: the uniform average scale 0
// defines; the LSE takes the caller's scale itself.
float exp2_scale(float scale) {
  return (float)std::max((double)scale * 1.4426950408889634, (double)FLT_MIN);
}

// (Batch, head) pairs per group of the dense unit order (0: one group): as
// many pairs as have their keys and values in about 32 MB, a quarter of the
// L2 cache, so that the units running at one time (at most two groups) find
// them there.  Causal units differ in cost, and a group order runs the long
// units of the last group at the end: on the long causal workload (1024
// units, 152 SMs) groups of 16, 8 and 4 pairs measured 3.7, 6.7 and 15 %
// slower than one group, for 2.2x fewer DRAM bytes at 8.  So causal calls
// keep one group unless they have at least 64 units per SM.
int pair_group(int N, int d, bool causal, int64_t units, int sms) {
  if (causal && units < 64 * (int64_t)sms) return 0;
  const int64_t kv = 2 * (int64_t)N * d * 2;
  return (int)std::max<int64_t>(1, std::min<int64_t>(1 << 20, (int64_t(32) << 20) / kv));
}

// Heads per group of the packed unit order (0: one group): as many heads as
// have the keys and values of all sequences (at most B N tokens) in about
// 32 MB, under the same rule as pair_group.
int head_group(int B, int N, int d, int H, bool causal, int64_t units, int sms) {
  if (causal && units < 64 * (int64_t)sms) return 0;
  const int64_t kv = 2 * (int64_t)B * N * d * 2;
  return (int)std::max<int64_t>(1, std::min<int64_t>(H, (int64_t(32) << 20) / kv));
}

// The library's choice of softmax layout for the one-CTA kernels (attn_fwd_options.kernel
// 0): one thread per query row, which measured faster at both head dims (same-process,
// TFLOP/s: GPT-2 shaped causal 377 against 347, long causal 1457 against 1327, long
// non-causal 1520 against 1408, stress 1525 against 1363); kernel 1 keeps two.
bool one_thread_per_row(int d, int kernel) {
  (void)d;
  return kernel != 1;
}

// rows: one softmax thread per query row (attn_fwd_row_kernel) instead of two
// Launch with programmatic stream serialisation: the kernel may start on the
// SMs the previous kernel of the stream has left (its set-up overlapping that
// kernel's last CTAs); it waits for that kernel's completion (griddepcontrol)
// before its first global access, so the order of the stream holds.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), int grid, int threads, size_t smem,
                             cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// mo: O through 32-row x 64-column boxes, for the one-thread-per-row kernel's
// TMA stores (unused by the other kernels).
template <int D>
int launch_attn(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                const CUtensorMap& mo, const FwdParams& p, int grid, cudaStream_t s,
                bool rows = false) {
  const bool window = p.wl >= 0 || p.wr >= 0;
  if (rows) {
    cudaError_t e = window ? launch_dependent(attn::attn_fwd_row_kernel<D, attn::kModeWindow>, grid,
                                              attn::kRowThreads, attn::RowCfg<D>::kSmemBytes, s, mq, mk, mv, mo, p)
                           : launch_dependent(attn::attn_fwd_row_kernel<D, attn::kModePlain>, grid,
                                              attn::kRowThreads, attn::RowCfg<D>::kSmemBytes, s, mq, mk, mv, mo, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
  }
  if (window)
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
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_ERR_SCALE;
  // the pair-of-SMs kernel takes d = 128 without a window only
  const bool use_pair = opts && opts->kernel == 2;
  if (use_pair && (d != 128 || window_left >= 0 || window_right >= 0)) return ATTN_ERR_SHAPE;
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
  // asked for, the pair kernel runs or the call fails (no other kernel instead)
  if (use_pair && ds->pair_clusters <= 0) return cuda_fail(cudaErrorLaunchOutOfResources);
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
  p.scale_log2 = exp2_scale(scale);
  p.timeout_ns = (opts && opts->wait_timeout_ns) ? opts->wait_timeout_ns : 2000000000ull;
  p.fault_inject = opts ? opts->fault_inject : 0;
  p.pair_group = cu_seqlens ? head_group(B, N, d, H, p.causal, units, ds->sms)
                            : pair_group(N, d, p.causal, units, ds->sms);

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
  // d = 128 without a window: the pair-of-SMs kernel when asked for; clusters
  // take the units round robin.  Asked for where it cannot run, the call fails
  // instead of running another kernel.
  if (use_pair) {
    CUtensorMap mk64;
    if ((st = make_map(enc, &mk64, k, tokens_bound, H, d, 64)) != ATTN_OK) return st;
    int64_t clusters = ds->pair_clusters;
    if (!cu_seqlens) clusters = std::min<int64_t>(clusters, units);
    if (opts && opts->max_ctas > 0) clusters = std::min<int64_t>(clusters, std::max(1, opts->max_ctas / 2));
    attn::attn_fwd_pair_kernel<<<(unsigned)(2 * clusters), attn::kPairThreads, attn::kPairSmemBytes, s>>>(
        mq, mk64, mv, p);
    e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
  }
  if (opts && opts->max_ctas > 0 && opts->max_ctas < grid) grid = opts->max_ctas;
  const bool rows = one_thread_per_row(d, opts ? opts->kernel : 0);
  CUtensorMap mo = mq;
  if (rows && (st = make_map(enc, &mo, o, tokens_bound, H, d, 32)) != ATTN_OK)
    return st;
  return d == 64 ? launch_attn<64>(mq, mk, mv, mo, p, grid, s, rows)
                 : launch_attn<128>(mq, mk, mv, mo, p, grid, s, rows);
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

namespace {

// attn_fwd_host's pipeline state for one (device, stream): two copy streams,
// the events that order them against the caller's stream, and a device
// workspace of two slots, each holding one head group's Q, K, V, O tiles and
// LSE block.
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_done[2] = {}, comp_done[2] = {}, out_done[2] = {};
  uint8_t* slot[2] = {nullptr, nullptr};
  size_t slot_bytes = 0;
};

std::mutex g_host_mu;  // attn_fwd_host's state; attn_fwd_impl takes g_mu itself
std::map<std::pair<int, attn_stream_t>, HostPipe> g_host;

size_t round_up_256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int host_pipe(int dev, attn_stream_t stream, size_t slot_bytes, HostPipe** out) {
  HostPipe& hp = g_host[std::make_pair(dev, stream)];
  cudaError_t e;
  if (!hp.in) {
    if ((e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e);
    cudaEvent_t* evs[] = {&hp.start, &hp.done, &hp.in_done[0], &hp.in_done[1], &hp.comp_done[0],
                          &hp.comp_done[1], &hp.out_done[0], &hp.out_done[1]};
    for (cudaEvent_t* ev : evs)
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e);
  }
  if (hp.slot_bytes < slot_bytes) {
    // the slots may still be read or written by the previous call's work
    if ((e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream))) != cudaSuccess)
      return cuda_fail(e);
    for (auto& p : hp.slot) {
      attn_host::lib_free(p);
      p = nullptr;
    }
    hp.slot_bytes = 0;
    for (auto& p : hp.slot)
      if ((e = attn_host::lib_malloc(&p, slot_bytes)) != cudaSuccess) return cuda_fail(e);
    hp.slot_bytes = slot_bytes;
  }
  *out = &hp;
  return ATTN_OK;
}

// Heads per group: about 32 MB of Q, K, V per group but at least two heads
// (groups of one head measured 1.3-1.9x slower end to end on the long causal,
// stress and packed workloads: a launch of one head holds too few work units
// for the SMs, and every group adds launches and hand-offs), and at least two
// groups when there are two heads (so that copies and attention overlap);
// groups as even as the head count allows.
int host_head_group(int64_t tokens, int H, int d) {
  const size_t head_bytes = 3 * (size_t)tokens * d * 2;
  int64_t hg = std::max<int64_t>(2, (int64_t)((32ull << 20) / std::max<size_t>(head_bytes, 1)));
  if (H >= 2) hg = std::min<int64_t>(hg, (H + 1) / 2);
  hg = std::min<int64_t>(hg, H);
  const int64_t groups = (H + hg - 1) / hg;
  return (int)((H + groups - 1) / groups);
}

}  // namespace

extern "C" int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int N, int d, float scale, int causal,
                             const int32_t* cu_seqlens, attn_stream_t stream) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_ERR_SCALE;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if ((int64_t)B * N > INT32_MAX - 2 * attn::kBN || (int64_t)H * d > (1 << 20) || H > 65535)
    return ATTN_ERR_SHAPE;
  // packed batches: the offsets are host memory, so they are checked here,
  // before any copy reads cu_seqlens[B] tokens of the caller's buffers
  int64_t tokens = (int64_t)B * N;
  if (cu_seqlens) {
    if (cu_seqlens[0] != 0) return ATTN_ERR_SEQLENS;
    for (int b = 0; b < B; ++b) {
      const int64_t len = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
      if (len < 0 || len > N) return ATTN_ERR_SEQLENS;
    }
    tokens = cu_seqlens[B];
    if (tokens == 0) return ATTN_OK;
  }
  const int hg = host_head_group(tokens, H, d);
  const size_t tile = round_up_256((size_t)tokens * hg * d * 2);  // [tokens, hg, d] bf16
  const size_t lse_bytes = round_up_256((size_t)tokens * hg * sizeof(float));
  const size_t cu_bytes = cu_seqlens ? round_up_256((size_t)(B + 1) * sizeof(int32_t)) : 0;

  std::lock_guard<std::mutex> lock(g_host_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  HostPipe* hp = nullptr;
  int st = host_pipe(dev, stream, 4 * tile + lse_bytes + cu_bytes, &hp);
  if (st != ATTN_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t row = (size_t)H * d * 2;  // bytes of one token's heads
  const auto* qh = static_cast<const uint8_t*>(q);
  const auto* kh = static_cast<const uint8_t*>(k);
  const auto* vh = static_cast<const uint8_t*>(v);
  auto* oh = static_cast<uint8_t*>(o);
  // the copies start after the caller's earlier work (and this stream's
  // previous call, which used the same slots)
  if ((e = cudaEventRecord(hp->start, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaStreamWaitEvent(hp->in, hp->start, 0)) != cudaSuccess) return cuda_fail(e);
  // On an error past this point, later work on the caller's stream still
  // waits for every copy already queued, so that the caller may release its
  // buffers once the stream is idle; the error is returned.
  auto fail_joined = [&](int status) {
    if (cudaEventRecord(hp->done, hp->in) == cudaSuccess) cudaStreamWaitEvent(s, hp->done, 0);
    if (cudaEventRecord(hp->done, hp->out) == cudaSuccess) cudaStreamWaitEvent(s, hp->done, 0);
    return status;
  };
  const int groups = (H + hg - 1) / hg;
  for (int g = 0; g < groups; ++g) {
    const int j = g & 1;
    const int h0 = g * hg, hn = std::min(hg, H - h0);
    const size_t w = (size_t)hn * d * 2;  // bytes of one token's heads of this group
    uint8_t* base = hp->slot[j];
    uint8_t *dq = base, *dk = base + tile, *dv = base + 2 * tile, *dout = base + 3 * tile;
    float* dlse = reinterpret_cast<float*>(base + 4 * tile);
    int32_t* dcu = cu_seqlens ? reinterpret_cast<int32_t*>(base + 4 * tile + lse_bytes) : nullptr;
    // Q, K, V of the group into slot j, once group g - 2's attention has read it
    if (g >= 2 && (e = cudaStreamWaitEvent(hp->in, hp->comp_done[j], 0)) != cudaSuccess)
      return fail_joined(cuda_fail(e));
    const uint8_t* srcs[3] = {qh, kh, vh};
    uint8_t* dsts[3] = {dq, dk, dv};
    for (int t = 0; t < 3; ++t)
      if ((e = cudaMemcpy2DAsync(dsts[t], w, srcs[t] + (size_t)h0 * d * 2, row, w, (size_t)tokens,
                                 cudaMemcpyDefault, hp->in)) != cudaSuccess)
        return fail_joined(cuda_fail(e));
    if (dcu && (e = cudaMemcpyAsync(dcu, cu_seqlens, (size_t)(B + 1) * sizeof(int32_t),
                                    cudaMemcpyDefault, hp->in)) != cudaSuccess)
      return fail_joined(cuda_fail(e));
    if ((e = cudaEventRecord(hp->in_done[j], hp->in)) != cudaSuccess)
      return fail_joined(cuda_fail(e));
    // attention of the group on the caller's stream, once its inputs are in
    // and group g - 2's outputs have left slot j
    if ((e = cudaStreamWaitEvent(s, hp->in_done[j], 0)) != cudaSuccess)
      return fail_joined(cuda_fail(e));
    if (g >= 2 && (e = cudaStreamWaitEvent(s, hp->out_done[j], 0)) != cudaSuccess)
      return fail_joined(cuda_fail(e));
    st = attn_fwd_impl(dq, dk, dv, dout, dlse, B, hn, N, d, scale, causal, -1, -1, dcu, stream,
                       nullptr);
    if (st != ATTN_OK) return fail_joined(st);
    if ((e = cudaEventRecord(hp->comp_done[j], s)) != cudaSuccess)
      return fail_joined(cuda_fail(e));
    // O and the LSE of the group back to the host buffers (LSE: dense [B, H,
    // N], the group's [B, hn, N] block; packed [H, tokens], its rows h0 ..)
    if ((e = cudaStreamWaitEvent(hp->out, hp->comp_done[j], 0)) != cudaSuccess)
      return fail_joined(cuda_fail(e));
    if ((e = cudaMemcpy2DAsync(oh + (size_t)h0 * d * 2, row, dout, w, w, (size_t)tokens,
                               cudaMemcpyDefault, hp->out)) != cudaSuccess)
      return fail_joined(cuda_fail(e));
    if (cu_seqlens)
      e = cudaMemcpyAsync(lse + (size_t)h0 * tokens, dlse, (size_t)hn * tokens * sizeof(float),
                          cudaMemcpyDefault, hp->out);
    else
      e = cudaMemcpy2DAsync(lse + (size_t)h0 * N, (size_t)H * N * sizeof(float), dlse,
                            (size_t)hn * N * sizeof(float), (size_t)hn * N * sizeof(float), B,
                            cudaMemcpyDefault, hp->out);
    if (e != cudaSuccess) return fail_joined(cuda_fail(e));
    if ((e = cudaEventRecord(hp->out_done[j], hp->out)) != cudaSuccess)
      return fail_joined(cuda_fail(e));
  }
  // later work on the caller's stream sees O and the LSE in the host buffers
  if ((e = cudaEventRecord(hp->done, hp->out)) != cudaSuccess) return fail_joined(cuda_fail(e));
  if ((e = cudaStreamWaitEvent(s, hp->done, 0)) != cudaSuccess) return cuda_fail(e);
  return ATTN_OK;
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
    case ATTN_ERR_SCALE: return "scale is negative or not finite";
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

namespace {

int attn_fwd_noalloc_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int H, int N, int d, float scale, int causal, const int32_t* cu_seqlens,
                          attn_stream_t stream, const attn_fwd_options* opts) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_ERR_SCALE;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_ALIGN;
  const int64_t tokens_bound = (int64_t)B * N;
  if (tokens_bound > INT32_MAX - 2 * attn::kBN || (int64_t)H * d > (1 << 20) || H > 65535)
    return ATTN_ERR_SHAPE;
  const int64_t nqb = (N + attn::kUnitRows - 1) / attn::kUnitRows;
  const int64_t entries = (int64_t)B * nqb;
  // only packed batches keep a scheduling list in the scratch
  if (cu_seqlens && entries > kNoAllocMaxEntries) return ATTN_ERR_SCRATCH;
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
  p.scale_log2 = exp2_scale(scale);
  p.timeout_ns = (opts && opts->wait_timeout_ns) ? opts->wait_timeout_ns : 2000000000ull;
  p.fault_inject = opts ? opts->fault_inject : 0;
  p.pair_group = cu_seqlens ? head_group(B, N, d, H, p.causal, units, nd->sms)
                            : pair_group(N, d, p.causal, units, nd->sms);

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
  if (opts && opts->max_ctas > 0 && opts->max_ctas < grid) grid = opts->max_ctas;
  const bool rows = one_thread_per_row(d, opts ? opts->kernel : 0);
  CUtensorMap mo = mq;
  if (rows && (st = make_map(enc, &mo, o, tokens_bound, H, d, 32)) != ATTN_OK)
    return st;
  return d == 64 ? launch_attn<64>(mq, mk, mv, mo, p, grid, s, rows)
                 : launch_attn<128>(mq, mk, mv, mo, p, grid, s, rows);
}

}  // namespace

extern "C" int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int N, int d, float scale, int causal,
                                const int32_t* cu_seqlens, attn_stream_t stream) {
  return attn_fwd_noalloc_impl(q, k, v, o, lse, B, H, N, d, scale, causal, cu_seqlens, stream,
                               nullptr);
}

extern "C" int attn_fwd_noalloc_ex(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int B, int H, int N, int d, float scale,
                                   int causal, const int32_t* cu_seqlens, attn_stream_t stream,
                                   const attn_fwd_options* opts) {
  return attn_fwd_noalloc_impl(q, k, v, o, lse, B, H, N, d, scale, causal, cu_seqlens, stream,
                               opts);
}

// Reads the error words of attn_fwd_noalloc's scratch with plain copies
// (no allocation) and clears them.
extern "C" int attn_fwd_noalloc_last_device_error(attn_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
  auto it = g_noalloc_dev.find(dev);
  if (it == g_noalloc_dev.end() || !it->second.ready) {
    g_last_error_site = 0;
    return ATTN_OK;
  }
  int h[2] = {0, 0};
  if ((e = cudaMemcpy(h, it->second.scratch, sizeof h, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaMemset(it->second.scratch, 0, sizeof h)) != cudaSuccess) return cuda_fail(e);
  g_last_error_site = h[1];
  if (h[0] & attn::kErrTimeout) return ATTN_ERR_DEVICE_TIMEOUT;
  if (h[0] & attn::kErrSeqlens) return ATTN_ERR_SEQLENS;
  if (h[0] & attn::kErrWorklist) return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

extern "C" size_t attn_device_bytes(void) { return attn_host::lib_device_bytes(); }

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
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_ERR_SCALE;
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

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (Nq == 1) {
    // One query row: the CUDA-core kernel, one work item per (sequence, head,
    // key range); by default about 16 items per SM, ranges of at least 64 keys.
    int S = num_splits;
    if (S == 0) {
      const int64_t bh = (int64_t)B * H;
      const int64_t want = ((int64_t)ds->sms * 16 + bh - 1) / bh;
      S = (int)std::max<int64_t>(1, std::min<int64_t>({want, (Nk + 63) / 64, 256}));
    }
    const int chunk = (Nk + S - 1) / S;
    const int64_t items = (int64_t)B * H * S;
    const int64_t combine_blocks = (q_tokens * H * 32 + 255) / 256;
    if (items > INT32_MAX || combine_blocks > INT32_MAX) return ATTN_ERR_SHAPE;
    float* part = nullptr;
    const size_t o_floats = (size_t)S * q_tokens * H * d;
    const size_t lse_floats = (size_t)S * B * H;
    if ((st = partial_workspace(dev, stream, o_floats + lse_floats, &part)) != ATTN_OK) return st;
    float* lse_part = part + o_floats;
    const int grid = (int)std::min<int64_t>(items, (int64_t)ds->sms * 8);
    const float c = exp2_scale(scale);
    auto q16 = reinterpret_cast<const __nv_bfloat16*>(q);
    auto k16 = reinterpret_cast<const __nv_bfloat16*>(k);
    auto v16 = reinterpret_cast<const __nv_bfloat16*>(v);
    if (d == 64)
      attn::decode::attn_decode_kernel<64><<<grid, attn::decode::kThreads, 0, s>>>(
          q16, k16, v16, part, lse_part, B, H, Nk, S, chunk, scale, c, nullptr, nullptr);
    else
      attn::decode::attn_decode_kernel<128><<<grid, attn::decode::kThreads, 0, s>>>(
          q16, k16, v16, part, lse_part, B, H, Nk, S, chunk, scale, c, nullptr, nullptr);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    if (d == 64)
      attn::attn_combine_kernel<64><<<(int)combine_blocks, 256, 0, s>>>(
          part, lse_part, reinterpret_cast<__nv_bfloat16*>(o), lse, B, H, 1, S);
    else
      attn::attn_combine_kernel<128><<<(int)combine_blocks, 256, 0, s>>>(
          part, lse_part, reinterpret_cast<__nv_bfloat16*>(o), lse, B, H, 1, S);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
  }

  // At most 128 queries (one query tile per 256-row block): the two query
  // tiles of a unit would repeat one another, so the two softmax groups take
  // two different KV ranges of the same tile instead (an even range count).
  const bool paired = Nq <= attn::kBM;
  int S = num_splits;
  if (S == 0) {
    // The number of ranges with the shortest estimated makespan: units of
    // equal cost run in ceil(units / SMs) rounds of ceil(tiles / S) KV tiles
    // each (paired: two ranges per unit); every extra range adds about a
    // quarter tile of partial-result traffic and merge work.  At most one
    // range per KV tile (paired: two), at most 64.
    const int64_t tiles = (Nk + attn::kBN - 1) / attn::kBN;
    const int step = paired ? 2 : 1;
    double best = 0.0;
    for (int64_t c = step; c <= std::max<int64_t>(step, std::min<int64_t>(tiles, 64)); c += step) {
      const int64_t rounds = (base_units * (c / step) + ds->sms - 1) / ds->sms;
      const double t = (double)rounds * (double)((tiles + c - 1) / c) + 0.25 * (double)(c - 1);
      if (c == step || t < best) {
        best = t;
        S = (int)c;
      }
    }
  } else if (paired && (S & 1)) {
    ++S;  // paired ranges need an even count
  }
  const int64_t units = base_units * (paired ? S / 2 : S);
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
  p.scale_log2 = exp2_scale(scale);
  p.timeout_ns = 2000000000ull;

  const int grid = (int)std::min<int64_t>(units, ds->sms);
  if (paired) {
    if (d == 64)
      attn::attn_fwd_kernel<64, attn::kModeSplitPair>
          <<<grid, attn::kThreads, FwdCfg<64>::kSmemBytes, s>>>(mq, mk, mv, p);
    else
      attn::attn_fwd_kernel<128, attn::kModeSplitPair>
          <<<grid, attn::kThreads, FwdCfg<128>::kSmemBytes, s>>>(mq, mk, mv, p);
  } else if (d == 64) {
    attn::attn_fwd_kernel<64, attn::kModeSplit><<<grid, attn::kThreads, FwdCfg<64>::kSmemBytes, s>>>(
        mq, mk, mv, p);
  } else {
    attn::attn_fwd_kernel<128, attn::kModeSplit><<<grid, attn::kThreads, FwdCfg<128>::kSmemBytes, s>>>(
        mq, mk, mv, p);
  }
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
// attn_fwd_decode: one query per sequence against packed key sequences of
// different lengths (the CUDA-core decode kernel and the combine).
extern "C" int attn_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int H, int d, float scale, const int32_t* cu_seqlens_k,
                               int max_seqlen_k, int num_splits, attn_stream_t stream) {
  if (B < 0 || H < 0 || max_seqlen_k < 0 || num_splits < 0 || num_splits > 256)
    return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_ERR_SCALE;
  if (B == 0 || H == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse || !cu_seqlens_k) return ATTN_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(cu_seqlens_k, 4))
    return ATTN_ERR_ALIGN;
  // key token indices (at most B * max_seqlen_k) stay within int32
  if ((int64_t)B * max_seqlen_k > INT32_MAX - 256 || (int64_t)H * d > (1 << 20) || H > 65535)
    return ATTN_ERR_SHAPE;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceState* ds = nullptr;
  int st = device_state(dev, &ds);
  if (st != ATTN_OK) return st;
  // key ranges: by default about 16 (sequence, head, range) items per SM,
  // ranges of at least 64 keys of the longest sequence
  int S = num_splits;
  if (S == 0) {
    const int64_t bh = (int64_t)B * H;
    const int64_t want = ((int64_t)ds->sms * 16 + bh - 1) / bh;
    S = (int)std::max<int64_t>(1, std::min<int64_t>({want, ((int64_t)max_seqlen_k + 63) / 64, 256}));
  }
  const int64_t items = (int64_t)B * H * S;
  const int64_t combine_blocks = ((int64_t)B * H * 32 + 255) / 256;
  if (items > INT32_MAX || combine_blocks > INT32_MAX) return ATTN_ERR_SHAPE;
  int* ws = nullptr;  // [3]: the validity flag of cu_seqlens_k
  if ((st = stream_workspace(dev, stream, 0, &ws)) != ATTN_OK) return st;
  float* part = nullptr;
  const size_t o_floats = (size_t)S * B * H * d;
  if ((st = partial_workspace(dev, stream, o_floats + (size_t)S * B * H, &part)) != ATTN_OK)
    return st;
  float* lse_part = part + o_floats;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  attn::decode::decode_check_kernel<<<1, 256, 0, s>>>(cu_seqlens_k, B, max_seqlen_k, ws + 3,
                                                       ds->err);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
  const int grid = (int)std::min<int64_t>(items, (int64_t)ds->sms * 8);
  const float c = exp2_scale(scale);
  auto q16 = reinterpret_cast<const __nv_bfloat16*>(q);
  auto k16 = reinterpret_cast<const __nv_bfloat16*>(k);
  auto v16 = reinterpret_cast<const __nv_bfloat16*>(v);
  if (d == 64)
    attn::decode::attn_decode_kernel<64><<<grid, attn::decode::kThreads, 0, s>>>(
        q16, k16, v16, part, lse_part, B, H, 0, S, 0, scale, c, cu_seqlens_k, ws + 3);
  else
    attn::decode::attn_decode_kernel<128><<<grid, attn::decode::kThreads, 0, s>>>(
        q16, k16, v16, part, lse_part, B, H, 0, S, 0, scale, c, cu_seqlens_k, ws + 3);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
  if (d == 64)
    attn::attn_combine_kernel<64><<<(int)combine_blocks, 256, 0, s>>>(
        part, lse_part, reinterpret_cast<__nv_bfloat16*>(o), lse, B, H, 1, S, ws + 3);
  else
    attn::attn_combine_kernel<128><<<(int)combine_blocks, 256, 0, s>>>(
        part, lse_part, reinterpret_cast<__nv_bfloat16*>(o), lse, B, H, 1, S, ws + 3);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
  return ATTN_OK;
}

// ---------------------------------------------------------------------------
// Services shared with the backward's host code (attn_host.h).
namespace attn_host {

std::mutex& lib_mutex() { return g_mu; }

int lib_cuda_fail(cudaError_t e) { return cuda_fail(e); }

namespace {
std::mutex g_alloc_mu;                 // the allocation record (own lock: attn_fwd_host
std::map<void*, size_t> g_alloc;       // allocates under its own lock, not the library's)
size_t g_alloc_bytes = 0;
}  // namespace

cudaError_t lib_malloc_raw(void** p, size_t bytes) {
  cudaError_t e = cudaMalloc(p, bytes);
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> lock(g_alloc_mu);
    g_alloc[*p] = bytes;
    g_alloc_bytes += bytes;
  }
  return e;
}

size_t lib_device_bytes() {
  std::lock_guard<std::mutex> lock(g_alloc_mu);
  return g_alloc_bytes;
}

void lib_free(void* p) {
  if (!p) return;
  {
    std::lock_guard<std::mutex> lock(g_alloc_mu);
    auto it = g_alloc.find(p);
    if (it != g_alloc.end()) {
      g_alloc_bytes -= it->second;
      g_alloc.erase(it);
    }
  }
  cudaFree(p);
}

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

// ---------------------------------------------------------------------------
// FP8 path (include/attn_fp8.h).
namespace {

struct Fp8Workspace {
  void* buf = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, attn_stream_t>, Fp8Workspace> g_fp8_ws;

int fp8_workspace(int dev, attn_stream_t stream, size_t bytes, uint8_t** out) {
  Fp8Workspace& ws = g_fp8_ws[std::make_pair(dev, stream)];
  if (ws.bytes < bytes || !ws.buf) {
    cudaError_t e;
    if (ws.buf) {
      if ((e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream))) != cudaSuccess)
        return cuda_fail(e);
      attn_host::lib_free(ws.buf);
      ws.buf = nullptr;
      ws.bytes = 0;
    }
    if ((e = attn_host::lib_malloc(&ws.buf, bytes)) != cudaSuccess) return cuda_fail(e);
    ws.bytes = bytes;
  }
  *out = static_cast<uint8_t*>(ws.buf);
  return ATTN_OK;
}

// e4m3 rows [tokens, H, 128]: box 128 bytes x 1 head x 128 rows.
int make_map_fp8_rows(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int64_t tokens, int H) {
  cuuint64_t dims[3] = {(cuuint64_t)attn::kFp8D, (cuuint64_t)H, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)attn::kFp8D, (cuuint64_t)H * attn::kFp8D};
  cuuint32_t box[3] = {(cuuint32_t)attn::kFp8D, 1, (cuuint32_t)attn::kBM};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : cuda_fail(cudaErrorInvalidValue);
}

// transposed e4m3 V [B*H][d][Np]: box 128 keys x d channels x 1.
int make_map_fp8_vt(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int64_t bh, int64_t np,
                    int d) {
  cuuint64_t dims[3] = {(cuuint64_t)np, (cuuint64_t)d, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)np, (cuuint64_t)np * d};
  cuuint32_t box[3] = {(cuuint32_t)attn::kBN, (cuuint32_t)d, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : cuda_fail(cudaErrorInvalidValue);
}

int fp8_check(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
  const int64_t tokens = (int64_t)B * N;
  if (tokens > INT32_MAX - 2 * attn::kBN || H > 65535 ||
      (int64_t)B * H * ((N + attn::kBN - 1) / attn::kBN) > INT32_MAX / 2)
    return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

attn::Fp8Signs pack_signs(const int8_t* signs, int d) {
  attn::Fp8Signs sg{};
  if (signs)
    for (int c = 0; c < d; ++c)
      if (signs[c] < 0) sg.bits[c / 32] |= 1u << (c % 32);
  return sg;
}

// Packed batches: validates cu_seqlens and builds the longest-first (sequence,
// q-block) list in the stream workspace; the quantisers and the attention
// kernel that follow on the stream read its entry count (0 when cu_seqlens
// is invalid, with the error word set).  *ws_out: the stream workspace, [0]
// the entry count, [1, 3) the attention kernel's unit counters, [4, ...) the
// list.  Dense batches only get the workspace.
int fp8_worklist(int dev, attn_stream_t stream, DeviceState* ds, const int32_t* cu_seqlens, int B,
                 int N, int causal, int** ws_out) {
  const int64_t max_entries = (int64_t)B * ((N + attn::kUnitRows - 1) / attn::kUnitRows);
  int* ws = nullptr;
  int st = stream_workspace(dev, stream, cu_seqlens ? max_entries : 0, &ws);
  if (st != ATTN_OK) return st;
  if (cu_seqlens) {
    const int ncost = (int)std::min<int64_t>((N + attn::kBN - 1) / attn::kBN,
                                             attn::kMaxCostBuckets - 1);
    attn::build_worklist_kernel<<<1, 1024, (ncost + 1) * sizeof(int),
                                  reinterpret_cast<cudaStream_t>(stream)>>>(
        cu_seqlens, B, N, causal, -1, -1, ws + 4, ws, ds->err, (int)max_entries, ws + 1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  *ws_out = ws;
  return ATTN_OK;
}

// bf16 rows [tokens, H, d] for the first quantisation stage: box 64 channels
// x 1 head x 128 rows, 128-byte swizzle (one copy per 64-channel chunk).
int make_map_quant_rows(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int64_t tokens, int H,
                        int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)attn::kBM};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : cuda_fail(cudaErrorInvalidValue);
}

// First stage: Q and / or K codes and block scales, and / or max |V| per
// 128-row block of V (amax_v: B * H * T words).  Null inputs are skipped.
// Packed (cu_seqlens): num_entries is the worklist's entry count.  The token
// extent of the copies is B * N (packed: an upper bound of cu_seqlens[B]; no
// copy leaves its sequence).
int launch_quant_stage1(const void* q, const void* k, const void* v, uint8_t* q8, uint8_t* k8,
                        float* sq, float* sk, unsigned int* amax_v, int B, int H, int N, int d,
                        int code_stride, const int8_t* signs, const int32_t* cu_seqlens,
                        const int* num_entries, DeviceState* ds, cudaStream_t s) {
  const int T = (N + attn::kBM - 1) / attn::kBM;
  const int nb = B * H * T;
  const int64_t tokens = (int64_t)B * N;
  EncodeTiledFn enc = nullptr;
  int st = get_encode(&enc);
  if (st != ATTN_OK) return st;
  CUtensorMap maps[3];
  std::memset(maps, 0, sizeof(maps));
  const void* src[3] = {q, k, v};
  for (int i = 0; i < 3; ++i)
    if (src[i] && (st = make_map_quant_rows(enc, &maps[i], src[i], tokens, H, d)) != ATTN_OK) return st;
  // segments: Q, K, V (the blocks run from the first present one to the last)
  const int nseg = v ? 3 : (k ? 2 : 1);
  const int first = q ? 0 : (k ? 1 : 2);
  const int n_blocks = (nseg - first) * nb;
  const int grid = std::min(n_blocks, (d == 64 ? attn::QuantCfg<64>::kCtasPerSm
                                                : attn::QuantCfg<128>::kCtasPerSm) * ds->sms);
  // a programmatic dependent of the stream's previous kernel (the kernel
  // waits for it before its first global access)
  const attn::Fp8Signs sg = pack_signs(signs, d);
  const int rotate = signs ? 1 : 0, block0 = first * nb;
  cudaError_t e =
      d == 64 ? launch_dependent(attn::fp8_quant_stage1_kernel<64>, grid, attn::kQuantThreads,
                                 attn::QuantCfg<64>::kSmemBytes, s, maps[0], maps[1], maps[2], q8, k8,
                                 sq, sk, amax_v, B, H, N, T, sg, rotate, block0, n_blocks,
                                 cu_seqlens, num_entries, ds->err, code_stride)
              : launch_dependent(attn::fp8_quant_stage1_kernel<128>, grid, attn::kQuantThreads,
                                 attn::QuantCfg<128>::kSmemBytes, s, maps[0], maps[1], maps[2], q8, k8,
                                 sq, sk, amax_v, B, H, N, T, sg, rotate, block0, n_blocks,
                                 cu_seqlens, num_entries, ds->err, code_stride);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return ATTN_OK;
}

int launch_quant_v(const void* v, uint8_t* codes_t, float* scale, unsigned int* amax_bits, int B,
                   int H, int N, int d, const int32_t* cu_seqlens, const int* num_entries,
                   cudaStream_t s) {
  const int T = (N + attn::kBN - 1) / attn::kBN;
  auto v16 = reinterpret_cast<const __nv_bfloat16*>(v);
  // a programmatic dependent of the first stage (the kernel waits for it)
  const int Np = T * attn::kBN;
  cudaError_t e =
      d == 64 ? launch_dependent(attn::fp8_quant_v_kernel<64>, B * H * T, 256, 0, s, v16, amax_bits,
                                 scale, codes_t, B, H, N, Np, cu_seqlens, num_entries)
              : launch_dependent(attn::fp8_quant_v_kernel<128>, B * H * T, 256, 0, s, v16, amax_bits,
                                 scale, codes_t, B, H, N, Np, cu_seqlens, num_entries);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

}  // namespace

extern "C" int attn_fp8_quantize_qk(const void* x, uint8_t* codes, float* scales, int B, int H,
                                    int N, int d, const int32_t* cu_seqlens, const int8_t* signs,
                                    attn_stream_t stream) {
  int st = fp8_check(B, H, N, d);
  if (st != ATTN_OK) return st;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!x || !codes || !scales) return ATTN_ERR_NULL;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return ATTN_ERR_ALIGN;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds)) != ATTN_OK) return st;
  int* ws = nullptr;
  if ((st = fp8_worklist(dev, stream, ds, cu_seqlens, B, N, 0, &ws)) != ATTN_OK) return st;
  return launch_quant_stage1(x, nullptr, nullptr, codes, nullptr, scales, nullptr, nullptr, B, H, N,
                             d, d, signs, cu_seqlens, ws, ds, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int attn_fp8_quantize_v(const void* v, uint8_t* codes_t, float* scale, int B, int H,
                                   int N, int d, const int32_t* cu_seqlens, attn_stream_t stream) {
  int st = fp8_check(B, H, N, d);
  if (st != ATTN_OK) return st;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!v || !codes_t || !scale) return ATTN_ERR_NULL;
  if (!aligned(v, 16) || !aligned(codes_t, 16) || !aligned(scale, 4)) return ATTN_ERR_ALIGN;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds)) != ATTN_OK) return st;
  uint8_t* ws = nullptr;
  const size_t n_blk = (size_t)B * H * ((N + attn::kBM - 1) / attn::kBM);
  if ((st = fp8_workspace(dev, stream, n_blk * sizeof(unsigned int) + 256, &ws)) != ATTN_OK)
    return st;
  unsigned int* amax = reinterpret_cast<unsigned int*>(ws);  // max |V| per 128-row block
  int* list = nullptr;
  if ((st = fp8_worklist(dev, stream, ds, cu_seqlens, B, N, 0, &list)) != ATTN_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launch_quant_stage1(nullptr, nullptr, v, nullptr, nullptr, nullptr, nullptr, amax, B, H,
                                N, d, d, nullptr, cu_seqlens, list, ds, s)) != ATTN_OK)
    return st;
  return launch_quant_v(v, codes_t, scale, amax, B, H, N, d, cu_seqlens, list, s);
}

namespace {

// The FP8 attention kernel on codes and scales already in device memory: Q
// and K codes in rows of 128 bytes, V codes [B*H][d][Np]; list: the FP8
// worklist (packed batches) and unit counters.
int launch_fp8_attention(EncodeTiledFn enc, DeviceState* ds, int* list, const uint8_t* q8,
                         const float* sq, const uint8_t* k8, const float* sk, const uint8_t* vt,
                         const float* sv, void* o, float* lse, int B, int H, int N, int d,
                         float scale, int causal, bool rotated, const int32_t* cu_seqlens,
                         cudaStream_t s) {
  const int64_t tokens = (int64_t)B * N;
  const int64_t T = (N + attn::kBM - 1) / attn::kBM;
  const int64_t np = T * attn::kBN;
  const int64_t bh = (int64_t)B * H;
  int st;
  CUtensorMap mq, mk, mvt, mo;
  if ((st = make_map_fp8_rows(enc, &mq, q8, tokens, H)) != ATTN_OK) return st;
  if ((st = make_map_fp8_rows(enc, &mk, k8, tokens, H)) != ATTN_OK) return st;
  if ((st = make_map_fp8_vt(enc, &mvt, vt, bh, np, d)) != ATTN_OK) return st;
  // O (bf16 [tokens, H, d]) through 32-row x 64-channel boxes: the epilogue's TMA stores
  if ((st = make_map(enc, &mo, o, tokens, H, d, 32)) != ATTN_OK) return st;
  attn::Fp8Params p{};
  p.o = reinterpret_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.sq = sq;
  p.sk = sk;
  p.sv = sv;
  p.err = ds->err;
  p.sched = list + 1;
  p.cu_seqlens = cu_seqlens;
  p.work = list + 4;
  p.num_entries = list;
  p.B = B;
  p.H = H;
  p.N = N;
  p.T = (int)T;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  // the unnormalised rotation multiplies Q K^T by d
  p.logit_log2 = (float)((double)scale * 1.4426950408889634 / (rotated ? (double)d : 1.0));
  p.timeout_ns = 2000000000ull;
  const int64_t units = bh * ((N + attn::kUnitRows - 1) / attn::kUnitRows);
  // packed: heads in groups whose codes (one byte per channel) fit in about
  // 32 MB, as for the bf16 path
  p.head_group = cu_seqlens ? head_group(B, N, d / 2, H, causal != 0, units, ds->sms) : 0;
  const int grid = cu_seqlens ? ds->sms : (int)std::min<int64_t>(units, ds->sms);
  // a programmatic dependent of the stream's previous kernel (the V
  // quantiser in attn_fwd_fp8): its set-up overlaps that kernel's last CTAs
  cudaError_t e = d == 64 ? launch_dependent(attn::attn_fp8_row_kernel<64>, grid, attn::kRowThreads,
                                             attn::kFp8SmemBytes, s, mq, mk, mvt, mo, p)
                          : launch_dependent(attn::attn_fp8_row_kernel<128>, grid, attn::kRowThreads,
                                             attn::kFp8SmemBytes, s, mq, mk, mvt, mo, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

}  // namespace

extern "C" int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int N, int d, float scale, int causal,
                            const int32_t* cu_seqlens, const int8_t* signs,
                            attn_stream_t stream) {
  int st = fp8_check(B, H, N, d);
  if (st != ATTN_OK) return st;
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_ERR_SCALE;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_ALIGN;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds)) != ATTN_OK) return st;
  EncodeTiledFn enc = nullptr;
  if ((st = get_encode(&enc)) != ATTN_OK) return st;

  const int64_t tokens = (int64_t)B * N;
  const int64_t T = (N + attn::kBM - 1) / attn::kBM;
  const int64_t np = T * attn::kBN;
  const int64_t bh = (int64_t)B * H;
  // workspace: Q codes, K codes, V codes (transposed, padded), Q and K block
  // scales, V scales, V block maxima (bits); each part 256-byte aligned
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t b_q = up((size_t)tokens * H * attn::kFp8D), b_vt = up((size_t)bh * d * np);
  const size_t b_s = up((size_t)bh * T * sizeof(float)), b_v = up((size_t)bh * sizeof(float));
  uint8_t* ws = nullptr;
  if ((st = fp8_workspace(dev, stream, 2 * b_q + b_vt + 3 * b_s + b_v + 256, &ws)) != ATTN_OK)
    return st;
  uint8_t* q8 = ws;
  uint8_t* k8 = q8 + b_q;
  uint8_t* vt = k8 + b_q;
  float* sq = reinterpret_cast<float*>(vt + b_vt);
  float* sk = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sq) + b_s);
  float* sv = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sk) + b_s);
  unsigned int* amax = reinterpret_cast<unsigned int*>(reinterpret_cast<uint8_t*>(sv) + b_v);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* list = nullptr;  // [0] entries, [1, 3) unit counters, [4, ...) the packed worklist
  if ((st = fp8_worklist(dev, stream, ds, cu_seqlens, B, N, causal ? 1 : 0, &list)) != ATTN_OK)
    return st;
  // Q and K codes in rows of 128 bytes (d = 64: zero-padded), V codes [B*H][d][Np]
  if ((st = launch_quant_stage1(q, k, v, q8, k8, sq, sk, amax, B, H, N, d, attn::kFp8D, signs,
                                cu_seqlens, list, ds, s)) != ATTN_OK)
    return st;
  if ((st = launch_quant_v(v, vt, sv, amax, B, H, N, d, cu_seqlens, list, s)) != ATTN_OK) return st;

  return launch_fp8_attention(enc, ds, list, q8, sq, k8, sk, vt, sv, o, lse, B, H, N, d, scale,
                              causal, signs != nullptr, cu_seqlens, s);
}

extern "C" int attn_fwd_fp8_codes(const uint8_t* q8, const float* sq, const uint8_t* k8,
                                  const float* sk, const uint8_t* vt, const float* sv, void* o,
                                  float* lse, int B, int H, int N, int d, float scale, int causal,
                                  int rotated, const int32_t* cu_seqlens, attn_stream_t stream) {
  int st = fp8_check(B, H, N, d);
  if (st != ATTN_OK) return st;
  // (d = 64: the quantisers' code rows are 64 bytes, the kernel reads 128)
  if (d != attn::kFp8D) return ATTN_ERR_HEADDIM;
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_ERR_SCALE;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q8 || !sq || !k8 || !sk || !vt || !sv || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(vt, 16) || !aligned(o, 16) ||
      !aligned(sq, 4) || !aligned(sk, 4) || !aligned(sv, 4) || !aligned(lse, 4))
    return ATTN_ERR_ALIGN;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds)) != ATTN_OK) return st;
  EncodeTiledFn enc = nullptr;
  if ((st = get_encode(&enc)) != ATTN_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* list = nullptr;
  if ((st = fp8_worklist(dev, stream, ds, cu_seqlens, B, N, causal ? 1 : 0, &list)) != ATTN_OK)
    return st;
  return launch_fp8_attention(enc, ds, list, q8, sq, k8, sk, vt, sv, o, lse, B, H, N, d, scale,
                              causal, rotated != 0, cu_seqlens, s);
}
