// Host side of the C ABI declared in include/attn_bwd.h: argument checks, the
// per-stream workspace (per-row D and LSE * log2 e, unit counters), TMA
// descriptors and the three launches (row prologue, dK/dV kernel, dQ kernel).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <map>
#include <set>
#include <utility>

#include "../../include/attn_bwd.h"
#include "attn_bwd_kernel.cuh"
#include "attn_host.h"

namespace {

using bwd::BwdCfg;
using bwd::BwdParams;

struct BwdWorkspace {
  void* buf = nullptr;   // [0, 256): unit counters (int), then lse2 and D (float), then the
                         // packed-batch lists (int)
  size_t floats = 0;     // capacity of each of the two float arrays
  size_t ints = 0;       // capacity of the list area
};

std::map<std::pair<int, attn_stream_t>, BwdWorkspace> g_bwd_ws;
std::set<int> g_bwd_ready;

constexpr size_t kCounterBytes = 256;

cudaError_t set_bwd_attributes() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(bwd::bwd_tile_kernel<64, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                BwdCfg<64>::kKvSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(bwd::bwd_tile_kernel<128, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                BwdCfg<128>::kKvSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(bwd::bwd_tile_kernel<64, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                BwdCfg<64>::kQSmemBytes)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(bwd::bwd_tile_kernel<128, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              BwdCfg<128>::kQSmemBytes);
}

int bwd_workspace(int dev, attn_stream_t stream, size_t floats, size_t ints, int** counters,
                  float** lse2, float** dd, int** lists) {
  BwdWorkspace& ws = g_bwd_ws[std::make_pair(dev, stream)];
  if (ws.floats < floats || ws.ints < ints || !ws.buf) {
    cudaError_t e;
    if (ws.buf) {
      // the old buffers may still be read by work queued on this stream
      if ((e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream))) != cudaSuccess)
        return attn_host::lib_cuda_fail(e);
      attn_host::lib_free(ws.buf);
      ws.buf = nullptr;
      ws.floats = 0;
    }
    const size_t cap = std::max<size_t>(floats, 1 << 16);
    const size_t icap = std::max<size_t>(ints, 1024);
    if ((e = attn_host::lib_malloc(&ws.buf, kCounterBytes + 2 * cap * sizeof(float) + icap * sizeof(int))) !=
        cudaSuccess)
      return attn_host::lib_cuda_fail(e);
    if ((e = cudaMemset(ws.buf, 0, kCounterBytes)) != cudaSuccess) return attn_host::lib_cuda_fail(e);
    ws.floats = cap;
    ws.ints = icap;
  }
  *counters = static_cast<int*>(ws.buf);
  *lse2 = reinterpret_cast<float*>(static_cast<char*>(ws.buf) + kCounterBytes);
  *dd = *lse2 + ws.floats;
  *lists = reinterpret_cast<int*>(*dd + ws.floats);
  return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

template <int D>
int launch_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
               const CUtensorMap& mdo, const void* o, const void* dout, const float* lse,
               BwdParams p, int* counters, int64_t max_tiles, int grid, cudaStream_t s) {
  // every row slot of every tile and head (packed: an upper bound of the
  // tiles), PrepCfg<D>::kRowsPerWarp slots per warp
  const long long slots = (long long)p.H * max_tiles * bwd::kTile;
  const long long warps = slots / bwd::PrepCfg<D>::kRowsPerWarp;
  const long long blocks = (warps * 32 + 255) / 256;
  bwd::bwd_prep_kernel<D><<<(unsigned)blocks, 256, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(o), reinterpret_cast<const __nv_bfloat16*>(dout), lse,
      p, slots);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return attn_host::lib_cuda_fail(e);
  p.sched = counters;
  bwd::bwd_tile_kernel<D, true><<<grid, bwd::kThreads, BwdCfg<D>::kKvSmemBytes, s>>>(
      mq, mk, mv, mdo, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return attn_host::lib_cuda_fail(e);
  p.sched = counters + 4;
  // the dQ kernel as the dK/dV kernel's programmatic dependent (it may start
  // on the SMs that kernel leaves; see bwd_tile_kernel)
  {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(bwd::kThreads);
    cfg.dynamicSmemBytes = BwdCfg<D>::kQSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, bwd::bwd_tile_kernel<D, false>, mq, mk, mv, mdo, p);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return attn_host::lib_cuda_fail(e);
  return ATTN_OK;
}

}  // namespace

namespace {

int attn_bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  float scale, int causal, int window_left, int window_right,
                  const int32_t* cu_seqlens, attn_stream_t stream) {
  if (B < 0 || H < 0 || N < 0 || window_left < -1 || window_right < -1) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_ERR_SCALE;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_NULL;
  for (const void* ptr : {q, k, v, o, dout, (const void*)dq, (const void*)dk, (const void*)dv})
    if (!aligned(ptr, 16)) return ATTN_ERR_ALIGN;
  if (!aligned(lse, 4)) return ATTN_ERR_ALIGN;
  const int64_t tokens = (int64_t)B * N;
  if (tokens > INT32_MAX - 2 * bwd::kTile || (int64_t)H * d > (1 << 20) || H > 65535)
    return ATTN_ERR_SHAPE;
  const int64_t T = (N + bwd::kTile - 1) / bwd::kTile;
  const int64_t max_tiles = (int64_t)B * T;  // packed: every length <= N
  const int64_t units = max_tiles * H;
  if (units > INT32_MAX / bwd::kTile || (cu_seqlens && T > bwd::kMaxCostBuckets)) return ATTN_ERR_SHAPE;

  std::lock_guard<std::mutex> lock(attn_host::lib_mutex());
  int dev = 0, sms = 0;
  int* err = nullptr;
  int st = attn_host::lib_device(&dev, &sms, &err);
  if (st != ATTN_OK) return st;
  if (!g_bwd_ready.count(dev)) {
    cudaError_t e = set_bwd_attributes();
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd::bwd_worklist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               2 * (bwd::kMaxCostBuckets + 1) * (int)sizeof(int));
    if (e != cudaSuccess) return attn_host::lib_cuda_fail(e);
    g_bwd_ready.insert(dev);
  }
  CUtensorMap mq, mk, mv, mdo;
  if ((st = attn_host::lib_make_map(&mq, q, tokens, H, d)) != ATTN_OK) return st;
  if ((st = attn_host::lib_make_map(&mk, k, tokens, H, d)) != ATTN_OK) return st;
  if ((st = attn_host::lib_make_map(&mv, v, tokens, H, d)) != ATTN_OK) return st;
  if ((st = attn_host::lib_make_map(&mdo, dout, tokens, H, d)) != ATTN_OK) return st;
  int* counters = nullptr;
  float *lse2 = nullptr, *dd = nullptr;
  int* lists = nullptr;
  // lists: [0] tile count, tile_off [B + 1] (at 8), then three (sequence, tile) lists
  const size_t off_lists = 8 + (size_t)B + 1;
  const size_t ints = cu_seqlens ? off_lists + 6 * (size_t)max_tiles : 0;
  if ((st = bwd_workspace(dev, stream, (size_t)units * bwd::kTile, ints, &counters, &lse2, &dd,
                          &lists)) != ATTN_OK)
    return st;

  BwdParams p{};
  p.dq = reinterpret_cast<__nv_bfloat16*>(dq);
  p.dk = reinterpret_cast<__nv_bfloat16*>(dk);
  p.dv = reinterpret_cast<__nv_bfloat16*>(dv);
  p.lse2 = lse2;
  p.dd = dd;
  p.err = err;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cu_seqlens) {
    int* tile_list = lists + off_lists;
    int* kv_list = tile_list + 2 * max_tiles;
    int* q_list = kv_list + 2 * max_tiles;
    p.cu_seqlens = cu_seqlens;
    p.num_tiles = lists;
    p.tile_off = lists + 8;
    p.tile_list = tile_list;
    p.kv_list = kv_list;
    p.q_list = q_list;
    bwd::bwd_worklist_kernel<<<1, 1024, 2 * (T + 1) * sizeof(int), s>>>(
        cu_seqlens, B, N, causal ? 1 : 0, window_left, window_right, lists, lists + 8, tile_list,
        kv_list, q_list, err,
        (int)max_tiles, counters, counters + 4);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return attn_host::lib_cuda_fail(e);
  }
  p.B = B;
  p.H = H;
  p.N = N;
  p.T = (int)T;
  p.causal = causal ? 1 : 0;
  p.wl = window_left;
  p.wr = window_right;
  p.scale = scale;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.timeout_ns = 2000000000ull;
  // packed causal calls with at least 64 units per SM (units counted from the
  // length bound): heads in groups whose streamed operands (two [tokens, d]
  // bf16 tensors of all sequences, at most B N tokens) fit in about 32 MB of
  // L2, the forward's rule
  if (cu_seqlens && (!causal || units >= 64 * (int64_t)sms)) {
    const int64_t bytes = 2 * (int64_t)B * N * d * 2;
    p.head_group = (int)std::max<int64_t>(1, std::min<int64_t>(H, (int64_t(32) << 20) / bytes));
  }
  // dense calls: (sequence, head) pairs in groups whose streamed operands fit
  // in about 64 MB of L2 (long causal workload, 32 pairs: 955 TFLOP/s with
  // groups of 16, 950 with 8, 938 with 4 and 915 with one group)
  if (!cu_seqlens) {
    const int64_t bytes = 2 * (int64_t)N * d * 2;
    p.pair_group = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)B * H, (int64_t(64) << 20) / bytes));
  }
  const int grid = (int)std::min<int64_t>(units, sms);
  return d == 64 ? launch_bwd<64>(mq, mk, mv, mdo, o, dout, lse, p, counters, max_tiles, grid, s)
                 : launch_bwd<128>(mq, mk, mv, mdo, o, dout, lse, p, counters, max_tiles, grid, s);
}

}  // namespace

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                        int H, int N, int d, float scale, int causal, const int32_t* cu_seqlens,
                        attn_stream_t stream) {
  return attn_bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, -1, -1,
                       cu_seqlens, stream);
}

extern "C" int attn_bwd_window(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               int B, int H, int N, int d, float scale, int causal,
                               int window_left, int window_right, const int32_t* cu_seqlens,
                               attn_stream_t stream) {
  return attn_bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, window_left,
                       window_right, cu_seqlens, stream);
}
