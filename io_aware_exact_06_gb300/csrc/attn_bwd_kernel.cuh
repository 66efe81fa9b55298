// Fused exact attention backward for sm_103a (GB300): dQ, dK, dV of
// O = softmax(scale * Q K^T) V for an upstream gradient dO.
//
// The score and probability matrices are rebuilt tile by tile from Q, K, V and
// the forward's saved row statistic (the LSE) instead of being stored:
// "flash-attention-evolution" (letsgetai), FlashAttention "核心机制", the
// recomputation paragraph; "FlashAttention 1-4 演进速查" (argus-lessons),
// FlashAttention-1 items.  Per visible (query i, key j):
//   P_ij  = exp(scale q_i.k_j - LSE_i)          (= 2^(c s_ij - LSE_i log2 e))
//   dP_ij = dO_i . v_j,   D_i = dO_i . O_i,     dS_ij = P_ij (dP_ij - D_i)
//   dV_j += P_ij dO_i,    dK_j += scale dS_ij q_i,   dQ_i += scale dS_ij k_j
//
// Three kernels:
//   bwd_prep_kernel   D_i and LSE_i log2(e) per row, written per 128-row query
//                     tile (rows of a pulled-back tail tile that the previous
//                     tile already holds, and rows outside the sequence, get
//                     LSE = +inf, so their P is 0 wherever they are loaded);
//   bwd_kv_kernel     one 128-key tile per work unit: K_j, V_j resident in
//                     shared memory, dK_j and dV_j accumulated in TMEM over
//                     the query tiles that see the keys;
//   bwd_q_kernel      one 128-query tile per work unit: Q_i, dO_i resident,
//                     dQ_i accumulated in TMEM over the key tiles it sees.
// The dQ kernel repeats the S and dP products of the dK/dV kernel (3 MMAs per
// tile pair there, 4 here, against 5 without the repeat) in exchange for
// owning every output row: no atomics, no fp32 dQ buffer, deterministic.
//
// CTA layout of both tile kernels (640 threads, one CTA per SM, persistent):
//   warps 0-15  compute: warp w reads TMEM lanes 32*(w%4).. (32 rows) and
//               columns [32*(w/4), +32) of each 128-column product; no two
//               warps share a column, so they never synchronise with each
//               other, only with the MMA warp through mbarriers
//   warp  16    TMA producer (lane 0)
//   warp  17    MMA issuer (lane 0) and TMEM owner
//   warps 18-19 idle
// A compute warp writes the bf16 operand it produces (P or dS, 32 values per
// row) into the first 16 columns of its own 32 (two values per column); the
// TMEM-operand MMA then reads k-step kk (16 keys or queries) from column
// 32*(kk/2) + 8*(kk%2) of the region.
//
// Every wait is bounded; on a timeout the kernel records an error word, stops
// issuing work, lets copies in flight land, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "sm100_ptx.cuh"

namespace bwd {

using attn::bulk_load;
using attn::globaltimer_ns;
using attn::make_idesc_bf16;
using attn::make_sdesc;
using attn::mbar_arrive;
using attn::mbar_arrive_expect_tx;
using attn::mbar_init;
using attn::mbar_try_wait;
using attn::mbar_wait;
using attn::mma_commit;
using attn::mma_ss;
using attn::mma_ts;
using attn::smem_u32;
using attn::tc_fence_after;
using attn::tc_fence_before;
using attn::tma_load_3d;
using attn::tma_prefetch_desc;

constexpr int kTile = 128;                 // rows of a query tile and of a key tile
constexpr int kComputeWarps = 16;
constexpr int kProducerWarp = kComputeWarps;
constexpr int kMmaWarp = kComputeWarps + 1;
constexpr int kThreads = 32 * (kComputeWarps + 4);
constexpr int kLaunchRegs = 96;
constexpr int kComputeRegs = 104;
constexpr int kControlRegs = 64;
static_assert(kThreads == 640, "five warpgroups");
static_assert(kComputeWarps * 32 * kComputeRegs + 128 * kControlRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allotment");
constexpr int kChunkBytes = kTile * 128;   // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kUnitSlots = 2;

constexpr int kMaxCostBuckets = 8192;  // packed batches: at most this many tiles per sequence

constexpr int kErrTimeout = 1;
constexpr int kErrSeqlens = 2;
constexpr int kErrWorklist = 4;

struct BwdParams {
  __nv_bfloat16* dq;   // [tokens, H, D]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* lse2;   // [H][tiles][128]: LSE * log2(e) per row of each 128-row tile (+inf: none)
  const float* dd;     // [H][tiles][128]: D_i = <dO_i, O_i>
  int* err;            // [0] error bits, [1] where a wait gave up
  int* sched;          // [0] next-unit counter, [1] finished CTAs (zero at launch, reset at exit)
  // packed batches (cu_seqlens != null): the scheduler kernel's lists
  const int* cu_seqlens;
  const int* num_tiles;  // tiles of all sequences (one 128-row tile = one unit per head)
  const int* tile_off;   // [nseq + 1]: first tile of each sequence
  const int* tile_list;  // [tiles] (sequence, tile) in sequence order
  const int* kv_list;    // [tiles] (sequence, tile), longest dK/dV unit first
  const int* q_list;     // [tiles] (sequence, tile), longest dQ unit first
  int B, H, N, T;        // dense: B sequences of length N, T = ceil(N / 128) tiles each
  int causal;
  int wl, wr;            // sliding window: keys i - wl <= j <= i + wr visible (-1: unbounded)
  float scale;         // softmax scale on the logits
  float scale_log2;    // scale * log2(e)
  unsigned long long timeout_ns;
  int head_group;        // packed: heads per group of the unit order (0: one group)
  int pair_group;        // dense: (sequence, head) pairs per group of the unit order (0: one)
};

// Dense unit u in pair groups of p.pair_group: within a group, rank (the
// position in the longest-first tile order) first, then pair.
__device__ __forceinline__ void dense_grouped(const BwdParams& p, int u, int& rank, int& b, int& h) {
  const int P = p.B * p.H;
  const int G = p.pair_group;
  const int full = P / G;
  int gi, r, np_;
  if (u < full * G * p.T) {
    gi = u / (G * p.T);
    r = u - gi * G * p.T;
    np_ = G;
  } else {
    gi = full;
    r = u - full * G * p.T;
    np_ = P - full * G;
  }
  rank = r / np_;
  const int pair = gi * G + (r - rank * np_);
  b = pair / p.H;
  h = pair - b * p.H;
}

// Start (sequence-relative) of the 128-row tile t, pulled back so the tile
// ends at the sequence end at the latest; rows before 128 t are the previous
// tile's and are neither counted twice nor stored.
__host__ __device__ __forceinline__ int tile_start(int t, int N) { return min(t * kTile, N - kTile); }

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int kTileBytes = (D / 64) * kChunkBytes;  // one 128 x D bf16 tile
  // dK/dV kernel: K, V resident; one ring of stages (Q, dO, LSE*log2e, D).
  // (Q and dO in rings of their own, dO's slot refilled after the dV product,
  // measured 3.5 % slower: one more commit and wait per tile.)
  static constexpr int kKvStages = D == 128 ? 2 : 4;
  static constexpr int kKvStageBytes = 2 * kTileBytes + 1024;
  static constexpr int kKvSmemBytes = 2 * kTileBytes + kKvStages * kKvStageBytes + 1024;
  // dQ kernel: Q, dO staged for their copy into TMEM; ring A = K slots, last
  // read by dQ += dS K, ring B = V slots, last read by dP = dO V^T, each with
  // its own full / empty barriers.  K feeds the first product of a tile (S),
  // so it gets a third slot at D = 128 (225 KB in all, within the 227 KB a
  // CTA may have) and its slot is refilled a whole tile ahead.
  static constexpr int kQASlots = D == 128 ? 3 : 4;
  static constexpr int kQBSlots = D == 128 ? 2 : 4;
  static constexpr int kQSmemBytes = 2 * kTileBytes + (kQASlots + kQBSlots) * kTileBytes + 1024;
  static_assert(kKvStages <= 4 && kQASlots <= 4 && kQBSlots <= 4, "barrier slots");
  static_assert(kKvSmemBytes <= 232448 && kQSmemBytes <= 232448, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescS = make_idesc_bf16(kTile, kTile, false);
  static constexpr uint32_t kIdescAcc = make_idesc_bf16(kTile, D, true);
};

// ---------------------------------------------------------------- MMAs --
// D = A B^T over D/16 k-steps: A and B both 128 rows x D, K-major, 128-byte
// swizzle (64-element chunks 16 KB apart, 8-row groups 1024 bytes apart; a
// 16-element step inside a chunk advances the start address by 32 bytes).
template <int D>
__device__ __forceinline__ void mma_rows_rows(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
  const uint64_t a0 = make_sdesc(a_smem, 16, 1024, attn::kSwizzle128B);
  const uint64_t b0 = make_sdesc(b_smem, 16, 1024, attn::kSwizzle128B);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (uint64_t)(((kk / 4) * kChunkBytes + (kk % 4) * 32) >> 4);
    mma_ss(d_tmem, a0 + off, b0 + off, BwdCfg<D>::kIdescS, kk > 0 ? 1u : 0u);
  }
}

// D (+)= A B over 128/16 k-steps: A (128 x 128 bf16) in TMEM in the grouped
// column layout above, B (128 rows x D) in shared memory, MN-major (D
// contiguous), 128-byte swizzle: 64-element chunks 16 KB apart (leading
// offset), 8-row groups 1024 bytes apart (stride offset); 16 rows advance the
// start address by 2048 bytes.
template <int D>
__device__ __forceinline__ void mma_tmem_rows(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem,
                                              bool accumulate) {
  const uint64_t b0 = make_sdesc(b_smem, kChunkBytes, 1024, attn::kSwizzle128B);
  const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk)
    mma_ts(d_tmem, a_tmem + 32 * (kk / 2) + 8 * (kk % 2), b0 + (uint64_t)((kk * 2048) >> 4),
           BwdCfg<D>::kIdescAcc, kk > 0 ? 1u : acc0);
}

// D = A B^T over D/16 k-steps with A (128 rows x D bf16, two elements per
// column, k-step kk in columns 8 kk..) in TMEM and B (128 rows x D) K-major in
// shared memory as for mma_rows_rows: the dQ kernel's S and dP products with
// Q and dO kept in TMEM, so that only K and V are read from shared memory.
template <int D>
__device__ __forceinline__ void mma_cols_rows(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem) {
  const uint64_t b0 = make_sdesc(b_smem, 16, 1024, attn::kSwizzle128B);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (uint64_t)(((kk / 4) * kChunkBytes + (kk % 4) * 32) >> 4);
    mma_ts(d_tmem, a_tmem + 8 * kk, b0 + off, BwdCfg<D>::kIdescS, kk > 0 ? 1u : 0u);
  }
}

// Row r of a 128 x D bf16 tile in the 128-byte-swizzled layout of the TMA
// copies (64-element chunks 16 KB apart, row r's 16-byte unit u at
// (u ^ (r % 8)) * 16), elements [32 cg, 32 cg + 32), to 16 TMEM columns of
// this thread's lane (two elements per column).
template <int D>
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t* tile, uint32_t taddr, int r, int cg) {
  const uint8_t* row = tile + (cg / 2) * kChunkBytes + r * 128;
  uint32_t w[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int u = 4 * (cg % 2) + k;
    const uint4 v = *reinterpret_cast<const uint4*>(row + ((u ^ (r & 7)) << 4));
    w[4 * k + 0] = v.x;
    w[4 * k + 1] = v.y;
    w[4 * k + 2] = v.z;
    w[4 * k + 3] = v.w;
  }
  attn::tmem_st_x16(taddr, w);
}

// ----------------------------------------------------- shared utilities --
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Barrier slots (both tile kernels; "res" = the resident pair of tiles,
// "stage" = the streamed pair).
enum : int {
  kBarUnitFull = 0,   // +slot
  kBarUnitEmpty = 2,  // +slot
  kBarResFull = 4,
  kBarResEmpty = 5,
  kBarSFull = 6,      // S (or S^T) product done
  kBarDPFull = 7,     // dP (or dP^T) product done
  kBarSCons = 8,      // dQ kernel: every compute warp has read S
  kBarPFull = 9,      // dK/dV kernel: P written to TMEM
  kBarDSFull = 10,    // dS written to TMEM
  kBarAccFull = 11,   // the unit's accumulators are complete
  kBarAccEmpty = 12,  // the compute warps have read them
  kBarDrain = 13,
  kBarAFull = 14,     // slot s of the (first) streamed ring loaded: kBarAFull + s
  kBarAEmpty = 18,    // and free again: kBarAEmpty + s
  kBarBFull = 22,     // dQ kernel's second ring (V) likewise
  kBarBEmpty = 26,
  kBarQTmemFull = 30, // dQ kernel: the unit's Q and dO are in TMEM
  kBarQTmemEmpty = 31,// dQ kernel: the unit's products no longer read them
  kMaxBars = 32,
};

struct Shared {
  uint64_t bars[kMaxBars];
  uint32_t tmem_base;
  volatile int abort_flag;
  volatile int unit_ring[kUnitSlots];
};

__device__ __forceinline__ uint32_t bar_addr(Shared& ss, int b) { return smem_u32(&ss.bars[b]); }

__device__ __forceinline__ bool wait_bar(Shared& ss, int b, uint32_t parity, const BwdParams& p,
                                         int where) {
  const uint32_t a = bar_addr(ss, b);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (ss.abort_flag) return false;
    if (globaltimer_ns() - t0 > p.timeout_ns) {
      ss.abort_flag = 1;
      atomicOr(p.err, kErrTimeout);
      atomicCAS(p.err + 1, 0, where);
      return false;
    }
  }
}

// The unit published by the producer in ring slot uslot (-1: no more work).
__device__ __forceinline__ bool next_unit(Shared& ss, const BwdParams& p, uint32_t& uslot,
                                          bool whole_warp, int& u) {
  const int slot = uslot % kUnitSlots;
  bool ok = wait_bar(ss, kBarUnitFull + slot, (uslot / kUnitSlots) & 1, p, 130);
  if (whole_warp) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return false;
  u = ss.unit_ring[slot];
  if (whole_warp) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar_addr(ss, kBarUnitEmpty + slot));
  } else {
    mbar_arrive(bar_addr(ss, kBarUnitEmpty + slot));
  }
  ++uslot;
  return true;
}

// Publishes unit u (or -1) to the consumers; false if the kernel is stopping.
__device__ __forceinline__ bool publish_unit(Shared& ss, const BwdParams& p, uint32_t& uslot, int u) {
  const int slot = uslot % kUnitSlots;
  const uint32_t n = uslot / kUnitSlots;
  if (n > 0 && !wait_bar(ss, kBarUnitEmpty + slot, (n - 1) & 1, p, 101)) return false;
  ss.unit_ring[slot] = u;
  mbar_arrive(bar_addr(ss, kBarUnitFull + slot));
  ++uslot;
  return true;
}

// Query tiles [o0, o0 + n) holding a query that sees some key of key tile t
// (nominal keys [128 t, min(128 t + 127, L - 1)]) of a sequence of length L.
__host__ __device__ __forceinline__ void kv_range(int L, int t, int causal, int wl, int wr, int& o0,
                                                  int& n) {
  const int kh = min(t * kTile + kTile - 1, L - 1);
  int lo = causal ? t * kTile : 0;
  if (wr >= 0) lo = max(lo, t * kTile - wr);
  int hi = L - 1;
  if (wl >= 0) hi = min(hi, kh + wl);
  lo = max(lo, 0);
  o0 = lo / kTile;
  n = hi / kTile + 1 - o0;
}

// Key tiles [o0, o0 + n) holding a key some row of query tile t sees.
__host__ __device__ __forceinline__ void q_range(int L, int t, int causal, int wl, int wr, int& o0,
                                                 int& n) {
  const int rh = min(t * kTile + kTile - 1, L - 1);
  const int lo = wl >= 0 ? max(0, t * kTile - wl) : 0;
  int hi = causal ? rh : L - 1;
  if (wr >= 0) hi = min(hi, rh + wr);
  o0 = lo / kTile;
  n = hi / kTile + 1 - o0;
}

// Key j visible to query i (both sequence-relative).
__device__ __forceinline__ bool visible(const BwdParams& p, int i, int j) {
  return (!p.causal || j <= i) && (p.wl < 0 || j >= i - p.wl) && (p.wr < 0 || j <= i + p.wr);
}

// One unit: (sequence b, head h, tile t of 128 rows) and the range of tiles
// of the other operand it visits, [o0, o0 + n); tok0 and L place the
// sequence in the packed tensors, tile0 its first tile in the per-row vectors.
// Longest first: the dK/dV kernel's causal cost T - t grows as t falls, the
// dQ kernel's t + 1 as t rises (dense: closed form; packed: the scheduler
// kernel's sorted lists).
struct Unit {
  int b, h, t, o0, n;
  int tok0, L, tile0;
};

__device__ __forceinline__ int total_tiles(const BwdParams& p) {
  return p.cu_seqlens ? *p.num_tiles : p.B * p.T;
}

__device__ __forceinline__ void place(const BwdParams& p, Unit& un) {
  if (p.cu_seqlens) {
    un.tok0 = p.cu_seqlens[un.b];
    un.L = p.cu_seqlens[un.b + 1] - un.tok0;
    un.tile0 = p.tile_off[un.b];
  } else {
    un.tok0 = un.b * p.N;
    un.L = p.N;
    un.tile0 = un.b * p.T;
  }
}

// Packed batches with p.head_group set: heads in groups of that many, one
// group after the other; within a group the sorted list, then head (the
// streamed tiles of a group stay in L2).  e: the list entry, h: the head.
__device__ __forceinline__ void packed_entry(const BwdParams& p, int u, int& e, int& h) {
  const int E = *p.num_tiles;
  const int G = p.head_group;
  const int full = p.H / G;
  int gi, r, ng;
  if (u < full * G * E) {
    gi = u / (G * E);
    r = u - gi * G * E;
    ng = G;
  } else {
    gi = full;
    r = u - full * G * E;
    ng = p.H - full * G;
  }
  e = r / ng;
  h = gi * G + (r - e * ng);
}

__device__ __forceinline__ Unit kv_unit(const BwdParams& p, int u) {
  Unit un;
  int e = u / p.H;
  un.h = u - e * p.H;
  if (p.cu_seqlens && p.head_group > 0 && p.head_group < p.H) packed_entry(p, u, e, un.h);
  if (p.cu_seqlens) {
    un.b = p.kv_list[2 * e];
    un.t = p.kv_list[2 * e + 1];
  } else if (p.pair_group > 0 && p.pair_group < p.B * p.H) {
    dense_grouped(p, u, un.t, un.b, un.h);
  } else {
    un.t = e / p.B;
    un.b = e - un.t * p.B;
  }
  place(p, un);
  kv_range(un.L, un.t, p.causal, p.wl, p.wr, un.o0, un.n);
  return un;
}

__device__ __forceinline__ Unit q_unit(const BwdParams& p, int u) {
  Unit un;
  int e = u / p.H;
  un.h = u - e * p.H;
  if (p.cu_seqlens && p.head_group > 0 && p.head_group < p.H) packed_entry(p, u, e, un.h);
  if (p.cu_seqlens) {
    un.b = p.q_list[2 * e];
    un.t = p.q_list[2 * e + 1];
  } else if (p.pair_group > 0 && p.pair_group < p.B * p.H) {
    int rank;
    dense_grouped(p, u, rank, un.b, un.h);
    un.t = p.T - 1 - rank;
  } else {
    const int rank = e / p.B;
    un.b = e - rank * p.B;
    un.t = p.T - 1 - rank;
  }
  place(p, un);
  q_range(un.L, un.t, p.causal, p.wl, p.wr, un.o0, un.n);
  return un;
}

// Index of row slot 0 of tile t of the unit's sequence in the per-row vectors.
__device__ __forceinline__ size_t vec_index(const BwdParams& p, const Unit& un, int t) {
  return ((size_t)un.h * total_tiles(p) + un.tile0 + t) * kTile;
}

// ------------------------------------------------------------ prologue --
// D_i = <dO_i, O_i> (fp32 sum of bf16 products) and LSE_i log2(e), written
// for every row slot of every query tile.  A row of D bf16 is read by D/8
// lanes, 16 bytes each; a warp covers kRowsPerLoad rows per load and takes
// kIters such groups, all its loads of O and dO issued before the first is
// used (the kernel moves 2 x 33.5 MB on the long workloads: bandwidth, not
// arithmetic).
template <int D>
struct PrepCfg {
  static constexpr int kLanesPerRow = D / 8;
  static constexpr int kRowsPerLoad = 32 / kLanesPerRow;
  static constexpr int kIters = 2;
  static constexpr int kRowsPerWarp = kRowsPerLoad * kIters;
  static_assert(kTile % kRowsPerWarp == 0, "the rows of a warp lie in one tile");
};

template <int D>
__global__ void __launch_bounds__(256)
bwd_prep_kernel(const __nv_bfloat16* o, const __nv_bfloat16* dout, const float* lse, BwdParams p,
                long long slots) {
  using C = PrepCfg<D>;
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const long long s0 = w * C::kRowsPerWarp;  // first row slot of this warp
  if (s0 >= slots) return;
  const int tiles = total_tiles(p);
  if (tiles <= 0) return;
  const long long gt = s0 / kTile;
  const int g = (int)(gt % tiles);
  const int h = (int)(gt / tiles);
  if (h >= p.H) return;  // (packed: the grid covers an upper bound of the tiles)
  Unit un;
  un.h = h;
  int t;
  if (p.cu_seqlens) {
    un.b = p.tile_list[2 * g];
    t = p.tile_list[2 * g + 1];
  } else {
    un.b = g / p.T;
    t = g - un.b * p.T;
  }
  place(p, un);
  const int chunk = lane % C::kLanesPerRow;  // elements 8 chunk .. 8 chunk + 7 of the row
  int r[C::kIters], row[C::kIters];
  bool valid[C::kIters];
  uint4 xo[C::kIters], xd[C::kIters];
#pragma unroll
  for (int it = 0; it < C::kIters; ++it) {
    r[it] = (int)(s0 % kTile) + it * C::kRowsPerLoad + lane / C::kLanesPerRow;
    row[it] = tile_start(t, un.L) + r[it];
    valid[it] = row[it] >= t * kTile;  // (and row < L: the tile ends at L)
    xo[it] = make_uint4(0u, 0u, 0u, 0u);
    xd[it] = xo[it];
    if (valid[it]) {
      const size_t base = ((size_t)(un.tok0 + row[it]) * p.H + h) * D + 8 * chunk;
      xo[it] = *reinterpret_cast<const uint4*>(o + base);
      xd[it] = *reinterpret_cast<const uint4*>(dout + base);
    }
  }
#pragma unroll
  for (int it = 0; it < C::kIters; ++it) {
    const uint32_t a[4] = {xo[it].x, xo[it].y, xo[it].z, xo[it].w};
    const uint32_t b[4] = {xd[it].x, xd[it].y, xd[it].z, xd[it].w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(a[i] << 16), __uint_as_float(b[i] << 16), acc);
      acc = fmaf(__uint_as_float(a[i] & 0xffff0000u), __uint_as_float(b[i] & 0xffff0000u), acc);
    }
#pragma unroll
    for (int off = C::kLanesPerRow / 2; off > 0; off >>= 1)
      acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (chunk == 0) {
      const size_t idx = vec_index(p, un, t) + r[it];
      float* dd = const_cast<float*>(p.dd);
      float* lse2 = const_cast<float*>(p.lse2);
      dd[idx] = acc;
      size_t li = 0;
      if (valid[it])
        li = p.cu_seqlens ? (size_t)h * p.cu_seqlens[p.B] + un.tok0 + row[it]
                          : ((size_t)un.b * p.H + h) * p.N + row[it];
      lse2[idx] = valid[it] ? lse[li] * 1.4426950408889634f : INFINITY;
    }
  }
}

// Packed batches: validates cu_seqlens, lays out the 128-row tiles of every
// sequence (tile_off, tile_list) and sorts them longest first for each tile
// kernel (a counting sort over the cost in tiles), and zeroes both kernels'
// unit counters.  One CTA.  base: [0] tile count, then tile_off [nseq + 1],
// tile_list, kv_list, q_list (2 ints per entry, max_entries entries each).
__global__ void __launch_bounds__(1024)
bwd_worklist_kernel(const int* cu_seqlens, int nseq, int max_len, int causal, int wl, int wr,
                    int* count, int* tile_off, int* tile_list, int* kv_list, int* q_list, int* err,
                    int max_entries, int* sched_kv, int* sched_q) {
  extern __shared__ int hist[];  // [2][ncost + 1]
  __shared__ int bad, total;
  const int ncost = (max_len + kTile - 1) / kTile;
  int* hkv = hist;
  int* hq = hist + ncost + 1;
  for (int i = threadIdx.x; i <= ncost; i += blockDim.x) hkv[i] = hq[i] = 0;
  if (threadIdx.x == 0) {
    bad = cu_seqlens[0] != 0;
    sched_kv[0] = sched_kv[1] = 0;
    sched_q[0] = sched_q[1] = 0;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    if (L < 0 || L > max_len) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) {
      *count = 0;
      atomicOr(err, kErrSeqlens);
    }
    return;
  }
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int s = 0; s < nseq; ++s) {
      tile_off[s] = acc;
      acc += (cu_seqlens[s + 1] - cu_seqlens[s] + kTile - 1) / kTile;
    }
    tile_off[nseq] = acc;
    total = acc;
  }
  __syncthreads();
  if (total > max_entries) {
    if (threadIdx.x == 0) {
      *count = 0;
      atomicOr(err, kErrWorklist);
    }
    return;
  }
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    const int T = (L + kTile - 1) / kTile;
    for (int t = 0; t < T; ++t) {
      tile_list[2 * (tile_off[s] + t)] = s;
      tile_list[2 * (tile_off[s] + t) + 1] = t;
      int o0, nkv, nq;
      kv_range(L, t, causal, wl, wr, o0, nkv);
      q_range(L, t, causal, wl, wr, o0, nq);
      atomicAdd(&hkv[nkv], 1);
      atomicAdd(&hq[nq], 1);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int okv = 0, oq = 0;
    for (int c = ncost; c >= 0; --c) {
      const int a = hkv[c], b = hq[c];
      hkv[c] = okv;
      hq[c] = oq;
      okv += a;
      oq += b;
    }
  }
  __syncthreads();
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    const int T = (L + kTile - 1) / kTile;
    for (int t = 0; t < T; ++t) {
      int o0, nkv, nq;
      kv_range(L, t, causal, wl, wr, o0, nkv);
      q_range(L, t, causal, wl, wr, o0, nq);
      const int a = atomicAdd(&hkv[nkv], 1);
      const int b = atomicAdd(&hq[nq], 1);
      kv_list[2 * a] = s;
      kv_list[2 * a + 1] = t;
      q_list[2 * b] = s;
      q_list[2 * b + 1] = t;
    }
  }
  if (threadIdx.x == 0) *count = total;
}

// -------------------------------------------------------- dK/dV kernel --
template <int D>
__device__ __forceinline__ void kv_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                            const CUtensorMap* tm_v, const CUtensorMap* tm_do,
                                            const BwdParams& p, Shared& ss, uint8_t* sK,
                                            uint8_t* sV, uint8_t* sStage, int n_units) {
  using C = BwdCfg<D>;
  uint32_t ring = 0, uslot = 0;
  int units_done = 0;
  int u = blockIdx.x;
  for (;;) {
    if (u >= n_units) u = -1;
    if (!publish_unit(ss, p, uslot, u) || u < 0) return;
    const int next_u = (int)gridDim.x + atomicAdd(p.sched, 1);
    const Unit un = kv_unit(p, u);
    if (units_done > 0 && !wait_bar(ss, kBarResEmpty, (units_done - 1) & 1, p, 102)) return;
    mbar_arrive_expect_tx(bar_addr(ss, kBarResFull), 2 * C::kTileBytes);
    const int k0 = un.tok0 + tile_start(un.t, un.L);
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(smem_u32(sK + c * kChunkBytes), tm_k, bar_addr(ss, kBarResFull), c * 64, un.h, k0);
      tma_load_3d(smem_u32(sV + c * kChunkBytes), tm_v, bar_addr(ss, kBarResFull), c * 64, un.h, k0);
    }
    for (int i = un.o0; i < un.o0 + un.n; ++i) {
      const int slot = ring % C::kKvStages;
      const uint32_t n = ring / C::kKvStages;
      if (n > 0 && !wait_bar(ss, kBarAEmpty + slot, (n - 1) & 1, p, 103)) return;
      const uint32_t full = bar_addr(ss, kBarAFull + slot);
      uint8_t* st = sStage + slot * C::kKvStageBytes;
      mbar_arrive_expect_tx(full, C::kKvStageBytes);
      const int q0 = un.tok0 + tile_start(i, un.L);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem_u32(st + c * kChunkBytes), tm_q, full, c * 64, un.h, q0);
        tma_load_3d(smem_u32(st + C::kTileBytes + c * kChunkBytes), tm_do, full, c * 64, un.h, q0);
      }
      const size_t vec = vec_index(p, un, i);
      bulk_load(smem_u32(st + 2 * C::kTileBytes), p.lse2 + vec, 512, full);
      bulk_load(smem_u32(st + 2 * C::kTileBytes + 512), p.dd + vec, 512, full);
      ++ring;
    }
    ++units_done;
    u = next_u;
  }
}

template <int D>
__device__ __forceinline__ void kv_mma(const BwdParams& p, Shared& ss, uint8_t* sK, uint8_t* sV,
                                       uint8_t* sStage, uint32_t tmem) {
  using C = BwdCfg<D>;
  constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + 128;
  const uint32_t k_smem = smem_u32(sK), v_smem = smem_u32(sV);
  auto q_smem = [&](uint32_t pos) { return smem_u32(sStage + (pos % C::kKvStages) * C::kKvStageBytes); };
  auto do_smem = [&](uint32_t pos) { return q_smem(pos) + C::kTileBytes; };
  auto stage_full = [&](uint32_t pos) {
    return wait_bar(ss, kBarAFull + pos % C::kKvStages, (pos / C::kKvStages) & 1, p, 110);
  };
  uint32_t ring = 0, uslot = 0, pcount = 0, dscount = 0;
  int units_done = 0;
  for (;;) {
    int u;
    if (!next_unit(ss, p, uslot, false, u) || u < 0) return;
    const Unit un = kv_unit(p, u);
    if (!wait_bar(ss, kBarResFull, units_done & 1, p, 111)) return;
    if (!stage_full(ring)) return;
    tc_fence_after();
    mma_rows_rows<D>(tmem + kColS, k_smem, q_smem(ring));     // S^T = K Q^T
    mma_commit(bar_addr(ss, kBarSFull));
    mma_rows_rows<D>(tmem + kColDP, v_smem, do_smem(ring));   // dP^T = V dO^T
    mma_commit(bar_addr(ss, kBarDPFull));
    for (int i = 0; i < un.n; ++i) {
      const uint32_t pos = ring + i;
      const bool more = i + 1 < un.n;
      if (!wait_bar(ss, kBarPFull, pcount++ & 1, p, 112)) return;
      if (i == 0 && units_done > 0 && !wait_bar(ss, kBarAccEmpty, (units_done - 1) & 1, p, 113))
        return;
      tc_fence_after();
      mma_tmem_rows<D>(tmem + kColDV, tmem + kColS, do_smem(pos), i > 0);   // dV += P^T dO
      if (more) {
        if (!stage_full(pos + 1)) return;
        tc_fence_after();
        mma_rows_rows<D>(tmem + kColS, k_smem, q_smem(pos + 1));
        mma_commit(bar_addr(ss, kBarSFull));
      }
      if (!wait_bar(ss, kBarDSFull, dscount++ & 1, p, 114)) return;
      tc_fence_after();
      mma_tmem_rows<D>(tmem + kColDK, tmem + kColDP, q_smem(pos), i > 0);   // dK += dS^T Q
      mma_commit(bar_addr(ss, kBarAEmpty + pos % C::kKvStages));           // stage free
      if (more) {
        mma_rows_rows<D>(tmem + kColDP, v_smem, do_smem(pos + 1));
        mma_commit(bar_addr(ss, kBarDPFull));
      }
    }
    ring += un.n;
    mma_commit(bar_addr(ss, kBarAccFull));
    mma_commit(bar_addr(ss, kBarResEmpty));
    ++units_done;
  }
}

template <int D>
__device__ __forceinline__ void kv_compute(const BwdParams& p, Shared& ss, uint8_t* sStage,
                                           uint32_t tmem) {
  using C = BwdCfg<D>;
  constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + 128;
  constexpr int kAccCols = D / 4;  // accumulator columns stored by one warp
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quadrant = warp % 4, cg = warp / 4;
  const int kr = quadrant * 32 + lane;  // key row of the tile = TMEM lane
  const uint32_t lane_addr = tmem + ((uint32_t)(quadrant * 32) << 16);
  const float c2 = p.scale_log2;
  uint32_t ring = 0, uslot = 0, scount = 0;
  int units_done = 0;
  for (;;) {
    int u = -1;
    if (!next_unit(ss, p, uslot, true, u) || u < 0) return;
    const Unit un = kv_unit(p, u);
    const int ks = tile_start(un.t, un.L);
    const int key = ks + kr;
    for (int i = 0; i < un.n; ++i) {
      const uint32_t pos = ring + i;
      const float* sl = reinterpret_cast<const float*>(sStage + (pos % C::kKvStages) * C::kKvStageBytes +
                                                       2 * C::kTileBytes);
      const int q0 = tile_start(un.o0 + i, un.L) + 32 * cg;  // query of this warp's column 0
      // the stage's LSE and D vectors are read below: wait for its copies too
      if (!__all_sync(0xffffffffu, wait_bar(ss, kBarAFull + pos % C::kKvStages,
                                            (pos / C::kKvStages) & 1, p, 123)))
        return;
      if (!__all_sync(0xffffffffu, wait_bar(ss, kBarSFull, scount & 1, p, 120))) return;
      tc_fence_after();
      uint32_t r[32];
      attn::tmem_ld_x32(lane_addr + kColS + 32 * cg, r);
      attn::tmem_ld_wait_x32(r);
      // P^T = 2^(c s - LSE log2 e); 0 where the query does not see the key
      // (causal, sliding window); decided per tile pair, applied per element
      const int qs = tile_start(un.o0 + i, un.L);
      const bool diag = (p.causal && ks + kTile - 1 > qs) ||
                        (p.wl >= 0 && ks < qs + kTile - 1 - p.wl) ||
                        (p.wr >= 0 && ks + kTile - 1 > qs + p.wr);
      float pf[32];
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(sl + 32 * cg + c);
        pf[c + 0] = ex2_approx(fmaf(__uint_as_float(r[c + 0]), c2, -l4.x));
        pf[c + 1] = ex2_approx(fmaf(__uint_as_float(r[c + 1]), c2, -l4.y));
        pf[c + 2] = ex2_approx(fmaf(__uint_as_float(r[c + 2]), c2, -l4.z));
        pf[c + 3] = ex2_approx(fmaf(__uint_as_float(r[c + 3]), c2, -l4.w));
      }
      if (diag) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (!visible(p, q0 + c, key)) pf[c] = 0.f;
      }
      uint32_t w[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) w[c] = pack_bf16x2(pf[2 * c], pf[2 * c + 1]);
      attn::tmem_st_x16(lane_addr + kColS + 32 * cg, w);
      attn::tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(ss, kBarPFull));
      // dS^T = P^T (dP^T - D)
      if (!__all_sync(0xffffffffu, wait_bar(ss, kBarDPFull, scount & 1, p, 121))) return;
      ++scount;
      tc_fence_after();
      attn::tmem_ld_x32(lane_addr + kColDP + 32 * cg, r);
      attn::tmem_ld_wait_x32(r);
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 d4 = *reinterpret_cast<const float4*>(sl + kTile + 32 * cg + c);
        pf[c + 0] *= __uint_as_float(r[c + 0]) - d4.x;
        pf[c + 1] *= __uint_as_float(r[c + 1]) - d4.y;
        pf[c + 2] *= __uint_as_float(r[c + 2]) - d4.z;
        pf[c + 3] *= __uint_as_float(r[c + 3]) - d4.w;
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) w[c] = pack_bf16x2(pf[2 * c], pf[2 * c + 1]);
      attn::tmem_st_x16(lane_addr + kColDP + 32 * cg, w);
      attn::tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(ss, kBarDSFull));
    }
    ring += un.n;
    // epilogue: dV and scale * dK of this warp's rows and columns -> bf16
    if (!__all_sync(0xffffffffu, wait_bar(ss, kBarAccFull, units_done & 1, p, 122))) return;
    tc_fence_after();
    const bool store = key >= un.t * kTile;  // (key < N: the tile ends at N)
    const size_t row_off = ((size_t)(store ? un.tok0 + key : 0) * p.H + un.h) * D + cg * kAccCols;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t col = (which == 0 ? kColDV : kColDK) + cg * kAccCols;
      const float mul = which == 0 ? 1.0f : p.scale;
      __nv_bfloat16* dst = (which == 0 ? p.dv : p.dk) + row_off;
      uint32_t a[kAccCols];
      if constexpr (kAccCols == 32) {
        attn::tmem_ld_x32(lane_addr + col, a);
        attn::tmem_ld_wait_x32(a);
      } else {
        attn::tmem_ld_x16(lane_addr + col, a);
        attn::tmem_ld_wait_x16(a);
      }
      if (store) {
#pragma unroll
        for (int c = 0; c < kAccCols; c += 8) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(a[c + 0]) * mul, __uint_as_float(a[c + 1]) * mul);
          v.y = pack_bf16x2(__uint_as_float(a[c + 2]) * mul, __uint_as_float(a[c + 3]) * mul);
          v.z = pack_bf16x2(__uint_as_float(a[c + 4]) * mul, __uint_as_float(a[c + 5]) * mul);
          v.w = pack_bf16x2(__uint_as_float(a[c + 6]) * mul, __uint_as_float(a[c + 7]) * mul);
          *reinterpret_cast<uint4*>(dst + c) = v;
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(ss, kBarAccEmpty));
    ++units_done;
  }
}

// ----------------------------------------------------------- dQ kernel --
template <int D>
__device__ __forceinline__ void q_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                           const CUtensorMap* tm_v, const CUtensorMap* tm_do,
                                           const BwdParams& p, Shared& ss, uint8_t* sQ,
                                           uint8_t* sDO, uint8_t* sA, uint8_t* sB, int n_units) {
  using C = BwdCfg<D>;
  uint32_t ringA = 0, ringB = 0, uslot = 0;
  int units_done = 0;
  int u = blockIdx.x;
  for (;;) {
    if (u >= n_units) u = -1;
    if (!publish_unit(ss, p, uslot, u) || u < 0) return;
    const int next_u = (int)gridDim.x + atomicAdd(p.sched, 1);
    const Unit un = q_unit(p, u);
    if (units_done > 0 && !wait_bar(ss, kBarResEmpty, (units_done - 1) & 1, p, 104)) return;
    mbar_arrive_expect_tx(bar_addr(ss, kBarResFull), 2 * C::kTileBytes);
    const int q0 = un.tok0 + tile_start(un.t, un.L);
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(smem_u32(sQ + c * kChunkBytes), tm_q, bar_addr(ss, kBarResFull), c * 64, un.h, q0);
      tma_load_3d(smem_u32(sDO + c * kChunkBytes), tm_do, bar_addr(ss, kBarResFull), c * 64, un.h, q0);
    }
    for (int j = un.o0; j < un.o0 + un.n; ++j) {
      const int k0 = un.tok0 + tile_start(j, un.L);
      {  // K (ring A)
        const int slot = ringA % C::kQASlots;
        const uint32_t n = ringA / C::kQASlots;
        if (n > 0 && !wait_bar(ss, kBarAEmpty + slot, (n - 1) & 1, p, 105)) return;
        const uint32_t full = bar_addr(ss, kBarAFull + slot);
        uint8_t* st = sA + slot * C::kTileBytes;
        mbar_arrive_expect_tx(full, C::kTileBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem_u32(st + c * kChunkBytes), tm_k, full, c * 64, un.h, k0);
        ++ringA;
      }
      {  // V (ring B)
        const int slot = ringB % C::kQBSlots;
        const uint32_t n = ringB / C::kQBSlots;
        if (n > 0 && !wait_bar(ss, kBarBEmpty + slot, (n - 1) & 1, p, 107)) return;
        const uint32_t full = bar_addr(ss, kBarBFull + slot);
        uint8_t* st = sB + slot * C::kTileBytes;
        mbar_arrive_expect_tx(full, C::kTileBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem_u32(st + c * kChunkBytes), tm_v, full, c * 64, un.h, k0);
        ++ringB;
      }
    }
    ++units_done;
    u = next_u;
  }
}

template <int D>
__device__ __forceinline__ void q_mma(const BwdParams& p, Shared& ss, uint8_t* sA, uint8_t* sB,
                                      uint32_t tmem) {
  using C = BwdCfg<D>;
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColQ = 256 + D, kColDO = 256 + D + D / 2;
  auto k_smem = [&](uint32_t pos) { return smem_u32(sA + (pos % C::kQASlots) * C::kTileBytes); };
  auto v_smem = [&](uint32_t pos) { return smem_u32(sB + (pos % C::kQBSlots) * C::kTileBytes); };
  auto a_full = [&](uint32_t pos) {
    return wait_bar(ss, kBarAFull + pos % C::kQASlots, (pos / C::kQASlots) & 1, p, 140);
  };
  auto b_full = [&](uint32_t pos) {
    return wait_bar(ss, kBarBFull + pos % C::kQBSlots, (pos / C::kQBSlots) & 1, p, 145);
  };
  // dP of tile j (V's slot is free once it is done)
  auto issue_dp = [&](uint32_t pos) {
    if (!b_full(pos)) return false;
    tc_fence_after();
    mma_cols_rows<D>(tmem + kColDP, tmem + kColDO, v_smem(pos));   // dP = dO V^T
    mma_commit(bar_addr(ss, kBarDPFull));
    mma_commit(bar_addr(ss, kBarBEmpty + pos % C::kQBSlots));
    return true;
  };
  auto issue_s = [&](uint32_t pos) {
    if (!a_full(pos)) return false;
    tc_fence_after();
    mma_cols_rows<D>(tmem + kColS, tmem + kColQ, k_smem(pos));     // S = Q K^T
    mma_commit(bar_addr(ss, kBarSFull));
    return true;
  };
  uint32_t ring = 0, uslot = 0, scons = 0, dscount = 0;
  int units_done = 0;
  for (;;) {
    int u;
    if (!next_unit(ss, p, uslot, false, u) || u < 0) return;
    const Unit un = q_unit(p, u);
    // Q and dO of the unit, copied into TMEM by the compute warps
    if (!wait_bar(ss, kBarQTmemFull, units_done & 1, p, 141)) return;
    // Product order per tile j: dQ(j), dP(j+1), then S(j+2) (S(j+1) was
    // issued one tile earlier), so the compute warps find S and dP of the next
    // tile ready and the K slot of tile j+2 has had a whole tile to arrive.
    // S is overwritten only after every compute warp has read it (SCons).
    if (!issue_s(ring) || !issue_dp(ring)) return;
    if (!wait_bar(ss, kBarSCons, scons++ & 1, p, 142)) return;
    if (un.n > 1 && !issue_s(ring + 1)) return;
    for (int j = 0; j < un.n; ++j) {
      const uint32_t pos = ring + j;
      if (!wait_bar(ss, kBarDSFull, dscount++ & 1, p, 143)) return;
      if (j == 0 && units_done > 0 && !wait_bar(ss, kBarAccEmpty, (units_done - 1) & 1, p, 144))
        return;
      tc_fence_after();
      mma_tmem_rows<D>(tmem + kColDQ, tmem + kColDP, k_smem(pos), j > 0);   // dQ += dS K
      mma_commit(bar_addr(ss, kBarAEmpty + pos % C::kQASlots));               // K slot free
      if (j + 1 < un.n) {
        if (!issue_dp(pos + 1)) return;
        if (!wait_bar(ss, kBarSCons, scons++ & 1, p, 146)) return;
        if (j + 2 < un.n && !issue_s(pos + 2)) return;
      }
    }
    ring += un.n;
    mma_commit(bar_addr(ss, kBarAccFull));
    mma_commit(bar_addr(ss, kBarQTmemEmpty));
    ++units_done;
  }
}

template <int D>
__device__ __forceinline__ void q_compute(const BwdParams& p, Shared& ss, const uint8_t* sQ,
                                          const uint8_t* sDO, uint32_t tmem) {
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColQ = 256 + D, kColDO = 256 + D + D / 2;
  constexpr int kAccCols = D / 4;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quadrant = warp % 4, cg = warp / 4;
  const int qr = quadrant * 32 + lane;  // query row of the tile = TMEM lane
  const uint32_t lane_addr = tmem + ((uint32_t)(quadrant * 32) << 16);
  const float c2 = p.scale_log2;
  uint32_t uslot = 0, scount = 0;
  int units_done = 0;
  for (;;) {
    int u = -1;
    if (!next_unit(ss, p, uslot, true, u) || u < 0) return;
    const Unit un = q_unit(p, u);
    const int row = tile_start(un.t, un.L) + qr;
    const size_t vec = vec_index(p, un, un.t) + qr;
    const float neg_lse2 = -p.lse2[vec];
    const float d_row = p.dd[vec];
    // Q and dO from the producer's tiles into TMEM (once the previous unit's
    // products are done with it); the tiles are then free for the next unit
    if (!__all_sync(0xffffffffu, wait_bar(ss, kBarResFull, units_done & 1, p, 153))) return;
    if (units_done > 0 &&
        !__all_sync(0xffffffffu, wait_bar(ss, kBarQTmemEmpty, (units_done - 1) & 1, p, 154)))
      return;
    tc_fence_after();
    if (cg < D / 32) {
      tile_row_to_tmem<D>(sQ, lane_addr + kColQ + 16 * cg, qr, cg);
      tile_row_to_tmem<D>(sDO, lane_addr + kColDO + 16 * cg, qr, cg);
    }
    attn::tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(bar_addr(ss, kBarResEmpty));
      mbar_arrive(bar_addr(ss, kBarQTmemFull));
    }
    for (int j = 0; j < un.n; ++j) {
      const int jt = un.o0 + j;
      const int k0 = tile_start(jt, un.L) + 32 * cg;  // key of this warp's column 0
      if (!__all_sync(0xffffffffu, wait_bar(ss, kBarSFull, scount & 1, p, 150))) return;
      tc_fence_after();
      uint32_t s[32];
      attn::tmem_ld_x32(lane_addr + kColS + 32 * cg, s);
      attn::tmem_ld_wait_x32(s);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(ss, kBarSCons));
      float pf[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) pf[c] = ex2_approx(fmaf(__uint_as_float(s[c]), c2, neg_lse2));
      // keys of the previous tile (pulled-back tail) or before the sequence,
      // and keys after the query when causal, contribute nothing
      const int klo = jt * kTile;
      const bool edge = k0 < klo || (p.causal && k0 + 31 > row) ||
                        (p.wl >= 0 && k0 < row - p.wl) || (p.wr >= 0 && k0 + 31 > row + p.wr);
      if (__any_sync(0xffffffffu, edge)) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (k0 + c < klo || !visible(p, row, k0 + c)) pf[c] = 0.f;
      }
      if (!__all_sync(0xffffffffu, wait_bar(ss, kBarDPFull, scount & 1, p, 151))) return;
      ++scount;
      tc_fence_after();
      attn::tmem_ld_x32(lane_addr + kColDP + 32 * cg, s);
      attn::tmem_ld_wait_x32(s);
      uint32_t w[16];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        w[c] = pack_bf16x2(pf[2 * c] * (__uint_as_float(s[2 * c]) - d_row),
                           pf[2 * c + 1] * (__uint_as_float(s[2 * c + 1]) - d_row));
      attn::tmem_st_x16(lane_addr + kColDP + 32 * cg, w);
      attn::tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(ss, kBarDSFull));
    }
    // epilogue: scale * dQ of this warp's columns -> bf16
    if (!__all_sync(0xffffffffu, wait_bar(ss, kBarAccFull, units_done & 1, p, 152))) return;
    tc_fence_after();
    const bool store = row >= un.t * kTile;
    uint32_t a[kAccCols];
    if constexpr (kAccCols == 32) {
      attn::tmem_ld_x32(lane_addr + kColDQ + cg * kAccCols, a);
      attn::tmem_ld_wait_x32(a);
    } else {
      attn::tmem_ld_x16(lane_addr + kColDQ + cg * kAccCols, a);
      attn::tmem_ld_wait_x16(a);
    }
    if (store) {
      __nv_bfloat16* dst = p.dq + ((size_t)(un.tok0 + row) * p.H + un.h) * D + cg * kAccCols;
#pragma unroll
      for (int c = 0; c < kAccCols; c += 8) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(a[c + 0]) * p.scale, __uint_as_float(a[c + 1]) * p.scale);
        v.y = pack_bf16x2(__uint_as_float(a[c + 2]) * p.scale, __uint_as_float(a[c + 3]) * p.scale);
        v.z = pack_bf16x2(__uint_as_float(a[c + 4]) * p.scale, __uint_as_float(a[c + 5]) * p.scale);
        v.w = pack_bf16x2(__uint_as_float(a[c + 6]) * p.scale, __uint_as_float(a[c + 7]) * p.scale);
        *reinterpret_cast<uint4*>(dst + c) = v;
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(ss, kBarAccEmpty));
    ++units_done;
  }
}

// ------------------------------------------------------------- kernels --
// kKv: the dK/dV kernel (else the dQ kernel).  Tensor maps over [tokens, H, D]
// bf16 with a 128-row x 64-element box, 128-byte swizzle.
template <int D, bool kKv>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tile_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared ss;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sRes0 = smem;                     // K (dK/dV kernel) or Q (dQ kernel)
  uint8_t* sRes1 = smem + C::kTileBytes;     // V or dO
  uint8_t* sA = smem + 2 * C::kTileBytes;    // the stage ring (dK/dV) or ring A, then B (dQ)
  uint8_t* sB = sA + C::kQASlots * C::kTileBytes;
  // The dQ kernel reads nothing the dK/dV kernel writes (only the inputs and
  // the prologue's vectors, complete before the dK/dV kernel starts), so it is
  // launched as the dK/dV kernel's dependent and may take the SMs that kernel
  // leaves while its last units run.
  if (kKv && threadIdx.x == 0) attn::grid_dep_launch();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_units = total_tiles(p) * p.H;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(bar_addr(ss, kBarUnitFull + i), 1);
      mbar_init(bar_addr(ss, kBarUnitEmpty + i), 1 + kComputeWarps);
    }
    mbar_init(bar_addr(ss, kBarResFull), 1);
    // (dK/dV kernel: released by the MMA thread; dQ kernel: by the compute
    // warps once they have copied Q and dO into TMEM)
    mbar_init(bar_addr(ss, kBarResEmpty), kKv ? 1 : kComputeWarps);
    mbar_init(bar_addr(ss, kBarQTmemFull), kComputeWarps);
    mbar_init(bar_addr(ss, kBarQTmemEmpty), 1);
    mbar_init(bar_addr(ss, kBarSFull), 1);
    mbar_init(bar_addr(ss, kBarDPFull), 1);
    mbar_init(bar_addr(ss, kBarSCons), kComputeWarps);
    mbar_init(bar_addr(ss, kBarPFull), kComputeWarps);
    mbar_init(bar_addr(ss, kBarDSFull), kComputeWarps);
    mbar_init(bar_addr(ss, kBarAccFull), 1);
    mbar_init(bar_addr(ss, kBarAccEmpty), kComputeWarps);
    mbar_init(bar_addr(ss, kBarDrain), 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar_addr(ss, kBarAFull + s), 1);
      mbar_init(bar_addr(ss, kBarAEmpty + s), 1);
      mbar_init(bar_addr(ss, kBarBFull + s), 1);
      mbar_init(bar_addr(ss, kBarBEmpty + s), 1);
    }
    ss.abort_flag = 0;
    attn::fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == kMmaWarp) {
    attn::tmem_alloc(smem_u32(&ss.tmem_base), C::kTmemCols);
    attn::tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ss.tmem_base;

  if (warp >= kComputeWarps) {
    setmaxnreg_dec<kControlRegs>();
    if (warp == kProducerWarp) {
      if (lane == 0) {
        if (kKv)
          kv_producer<D>(&tm_q, &tm_k, &tm_v, &tm_do, p, ss, sRes0, sRes1, sA, n_units);
        else
          q_producer<D>(&tm_q, &tm_k, &tm_v, &tm_do, p, ss, sRes0, sRes1, sA, sB, n_units);
      }
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        if (kKv)
          kv_mma<D>(p, ss, sRes0, sRes1, sA, tmem);
        else
          q_mma<D>(p, ss, sA, sB, tmem);
        // every MMA issued by this thread has finished before TMEM is freed
        mma_commit(bar_addr(ss, kBarDrain));
        mbar_wait(bar_addr(ss, kBarDrain), 0, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    setmaxnreg_inc<kComputeRegs>();
    if (kKv)
      kv_compute<D>(p, ss, sA, tmem);
    else
      q_compute<D>(p, ss, sRes0, sRes1, tmem);
    __syncwarp();
  }

  if (ss.abort_flag) {
    // copies issued before the abort may still be landing: give them 1 ms
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    attn::tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
      __threadfence();
    }
  }
  // the dQ kernel ends only after the dK/dV kernel: the call completes with
  // both, for whatever the stream runs next
  if (!kKv) attn::grid_dep_wait();
}

}  // namespace bwd
