// Fused exact softmax-attention forward for sm_103a (GB300).
//
// O = softmax(scale * Q K^T) V and LSE = log(sum exp(scale * Q K^T)) per row,
// computed tile by tile with a running row max m and running row sum l, so the
// N x N score (S) and probability (P) matrices never reach HBM.
//   - tiling + online softmax + one fused kernel: "flash-attention-evolution"
//     (letsgetai), FlashAttention section "核心机制" (items 1-2 and the
//     two-segment merge equations); "FlashAttention" (compassingai), section 3;
//   - query-tile-outer / KV-tile-inner loop, query tiles spread over CTAs:
//     "FlashAttention 1-4 演进速查" (argus-lessons), FlashAttention-2 items;
//   - producer warp + MMA warp + softmax warps (warp specialisation) and the
//     softmax of one tile overlapping the MMAs of another (ping-pong), with
//     registers moved between warp roles (setmaxnreg): same page,
//     FlashAttention-3 items;
//   - accumulators in tensor memory (TMEM), asynchronous MMA pipeline,
//     conditional rescaling of O, longest-processing-time-first scheduling:
//     same page, FlashAttention-4 items.
//
// Scheduling: a persistent CTA takes units in longest-first order: its first
// unit is blockIdx.x, every further one comes from an atomic counter (the
// producer pops it and publishes it to the MMA and softmax warps through a
// two-slot ring in shared memory), so CTAs that drew short units take more.
//
// CTA layout (640 threads = 5 warpgroups, one CTA per SM, persistent):
//   warps 0-7   softmax group 0 (query tile 0 of the unit), warps 8-15 group 1:
//               warp w reads TMEM lanes 32*(w%4).. (its 32 rows) and handles
//               key columns [64*h, 64*h+64) with h = (w%8)/4, so two warps
//               share each row; they combine row maxima and sums through
//               shared memory under a named barrier
//   warp  16    TMA producer (lane 0): Q tiles, then K_j, V_j into a ring
//   warp  17    MMA issuer (lane 0) and TMEM owner
//   warps 18-19 idle
// Registers are moved from the control warpgroup to the softmax warpgroups
// with setmaxnreg (launch: 640 x 96; after: 512 x 104 + 128 x 64).
// A work unit is (sequence, head, 256 query rows) = two 128-row query tiles.
// Per KV tile j the tensor core runs, in order,
//   O0 += P0 V_{j-1};  S0 = Q0 K_j^T;  O1 += P1 V_{j-1};  S1 = Q1 K_j^T
// so softmax group 0 works on S0 while the tensor core runs group 1's MMAs
// and the other way round.  P_g is written back into the TMEM columns of S_g
// (bf16 pairs) and read from there as the A operand of the PV product.
//
// TMEM (512 columns x 128 lanes x 32 bit): S0 [0,128), S1 [128,256),
// O0 [256, 256+D), O1 [256+D, 256+2D).
//
// Every wait is bounded; on a timeout the kernel records an error word, stops
// issuing work, lets copies in flight land, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "sm100_ptx.cuh"

namespace attn {

constexpr int kBM = 128;               // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;               // keys per KV tile
constexpr int kQTiles = 2;             // query tiles per work unit
constexpr int kUnitRows = kBM * kQTiles;
constexpr int kGroupWarps = 8;           // softmax warps per query tile
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr int kSoftmaxWarps = kQTiles * kGroupWarps;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr int kThreads = 32 * (kSoftmaxWarps + 4);
constexpr int kLaunchRegs = 96;          // 65536 / 640, rounded down to 8
constexpr int kSoftmaxRegs = 104;
constexpr int kControlRegs = 64;
static_assert(kThreads == 640, "five warpgroups");
static_assert(kSoftmaxWarps * 32 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allotment");
constexpr int kHalfCols = kBN / 2;       // key columns per softmax thread
constexpr int kChunkBytes = kBM * 128; // 128 rows x 64 bf16 (one 128-byte swizzle span)
// Rescale O only if the row max grew by more than 2^16: a stale-max probability
// stays below 2^16, far inside the bf16 (P) and fp32 (O, l) exponent range.
constexpr float kRescaleLog2 = 16.0f;

// Device error word bits.
constexpr int kErrTimeout = 1;
constexpr int kErrSeqlens = 2;
constexpr int kErrWorklist = 4;

struct FwdParams {
  __nv_bfloat16* o;        // [tokens, H, D]
  float* lse;              // dense [B, H, N]; varlen [H, tokens]
  const int* cu_seqlens;   // null: dense batch of B sequences of length N
  const int* work;         // varlen: LPT-ordered (seq, q-block) pairs
  const int* num_entries;  // varlen: number of pairs in `work`
  int* err;                // err[0]: error bits; err[1]: where a wait gave up
  int* sched;              // [0] next-unit counter, [1] finished CTAs; zero at launch,
                           // reset to zero by the last CTA to finish
  int B, H, N;
  int causal;
  int wl, wr;              // sliding window: keys i - wl <= j <= i + wr (-1: unbounded)
  // split-KV mode (dense only): queries [B, Nq = N, H, D], keys [B, Nk, H, D];
  // query row r sits at key position q_off + r (q_off = Nk - Nq when causal);
  // the visible KV tiles of a q-block are cut into num_splits ranges whose
  // partial results (O / l in fp32, LSE) go to o_part / lse_part.
  int Nk, q_off, num_splits;
  float* o_part;           // [num_splits][B * Nq][H][D]
  float* lse_part;         // [num_splits][B][H][Nq]
  float scale;             // softmax scale on the logits
  float scale_log2;        // scale * log2(e)
  unsigned long long timeout_ns;
  int fault_inject;        // 1: CTA 0 never issues its first K copy (test hook)
  int pair_group;          // not split: dense, (batch, head) pairs per group of the
                           // unit order; packed, heads per group (0: one group)
};

template <int D>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;   // one 128 x D bf16 tile
  static constexpr int kStages = D == 128 ? 4 : 8;           // K/V ring slots
  static constexpr int kSmemQ = kQTiles * kTileBytes;
  static constexpr int kSmemRing = kStages * kTileBytes;
  static constexpr int kSmemBytes = kSmemQ + kSmemRing + 1024;  // + alignment slack
  // TMEM column of S_g (P_g aliases its first 64 columns) and of O_g
  __host__ __device__ static constexpr uint32_t col_s(int g) { return (uint32_t)g * 128u; }
  __host__ __device__ static constexpr uint32_t col_o(int g) { return 256u + (uint32_t)g * D; }
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescS = make_idesc_bf16(kBM, kBN, false);
  static constexpr uint32_t kIdescPV = make_idesc_bf16(kBM, D, true);
};

// Barrier slots in shared memory.
enum : int {
  kBarQFull = 0,
  kBarQEmpty = 1,
  kBarSFull = 2,   // +g
  kBarPFull = 4,   // +g
  kBarOFull = 6,   // +g
  kBarDrain = 8,
  kBarUnitFull = 9,    // +slot
  kBarUnitEmpty = 11,  // +slot
  kBarKV = 13,     // kv_full[s] = kBarKV + s, kv_empty[s] = kBarKV + kStages + s
  kBarQFull1 = 29,   // second Q buffer (kernels that double-buffer Q by unit)
  kBarQEmpty1 = 30,
  kBarSFree = 31,    // +g: the softmax of group g has read S_g (kernels with P apart from S)
  kBarPFree = 33,    // +g: the P V product of group g finished (same kernels)
  kBarDrain1 = 35,   // a second MMA-issuing thread's products all finished
};
constexpr int kMaxBars = kBarDrain1 + 1;
static_assert(kBarKV + 2 * 8 <= kBarQFull1, "K/V ring barriers");
// Barriers of Q buffer b.
__device__ __forceinline__ int bar_qfull(int b) { return b == 0 ? kBarQFull : kBarQFull1; }
__device__ __forceinline__ int bar_qempty(int b) { return b == 0 ? kBarQEmpty : kBarQEmpty1; }
constexpr int kUnitSlots = 2;            // unit indices published by the producer
constexpr int kUnitConsumers = 1 + kSoftmaxWarps;  // the MMA thread and every softmax warp

// Kernel modes (separate instantiations): plain attention, sliding window,
// split-KV with separate query and key lengths.
enum : int { kModePlain = 0, kModeWindow = 1, kModeSplit = 2, kModeSplitPair = 3 };
// Split-KV modes.  kModeSplitPair serves query blocks with at most 128 rows
// (one real query tile): its two softmax groups take the same query tile and
// two different KV ranges, 2 s and 2 s + 1, of an even number of ranges.
__host__ __device__ constexpr bool is_split_mode(int m) { return m == kModeSplit || m == kModeSplitPair; }

// One work unit: rows [256 qb, 256 qb + 256) of head h of one sequence
// (split-KV: and one range of its KV tiles).
struct Unit {
  int seq, h, qb;
  int tok0;   // first query token of the sequence in the packed tensors
  int L;      // query length of the sequence
  int k_tok0; // first key token (split-KV; else tok0)
  int Lk;     // key length (split-KV; else L)
  int kv0;    // first KV tile visited
  int nkv;    // KV tiles visited
  int split;  // KV range index (split-KV; else 0); kModeSplitPair: the pair of ranges
  int kv0b, nkvb;  // kModeSplitPair: the second group's KV tiles (else 0, 0)
};

// KV tiles [kv0, kv0 + nkv) that hold a key visible to some row of q-block qb
// (rows [256 qb, 256 qb + 256) of a sequence of length L): every key, or keys
// up to the row when causal, narrowed by the sliding window.  Tiles outside
// are skipped; the cost of the unit is nkv.
__host__ __device__ __forceinline__ void unit_kv_range(int L, int qb, int causal, int wl, int wr,
                                                       int& kv0, int& nkv) {
  const int r_lo = qb * kUnitRows;
  const int r_hi = min(qb * kUnitRows + kUnitRows, L) - 1;
  int k_lo = 0, k_hi = causal ? r_hi : L - 1;
  if (wl >= 0) k_lo = max(0, r_lo - wl);
  if (wr >= 0) k_hi = min(k_hi, r_hi + wr);
  kv0 = k_lo / kBN;
  nkv = k_hi / kBN + 1 - kv0;
}

template <int kMode>
__device__ __forceinline__ int num_units(const FwdParams& p) {
  if (!is_split_mode(kMode) && p.cu_seqlens) return *p.num_entries * p.H;
  const int nqb = (p.N + kUnitRows - 1) / kUnitRows;
  const int ranges = kMode == kModeSplitPair ? p.num_splits / 2 : (p.num_splits > 1 ? p.num_splits : 1);
  return p.B * p.H * nqb * ranges;
}

// Unit u of the longest-first order.  Dense: the (batch, head) pairs in
// groups of p.pair_group, one group after the other; within a group
// q-blocks in decreasing cost (causal cost grows with the q-block index),
// then batch, then head.  A group's keys and values fit in a part of L2, so
// the units running at one time re-read them from L2 rather than HBM.  Varlen:
// the scheduler kernel's sorted (seq, q-block) list, then head.  Split-KV:
// q-blocks in decreasing cost, then KV range, then batch, then head.
template <int kMode>
__device__ __forceinline__ Unit decode_unit(const FwdParams& p, int u) {
  Unit un;
  const int e = u / p.H;
  un.h = u - e * p.H;
  un.split = 0;
  un.kv0b = 0;
  un.nkvb = 0;
  if (!is_split_mode(kMode) && p.cu_seqlens) {
    if (p.pair_group > 0 && p.pair_group < p.H) {
      // heads in groups of p.pair_group, one group after the other; within
      // a group the sorted list, then head
      const int E = *p.num_entries;
      const int G = p.pair_group;
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
      const int ee = r / ng;
      un.h = gi * G + (r - ee * ng);
      un.seq = p.work[2 * ee];
      un.qb = p.work[2 * ee + 1];
    } else {
      un.seq = p.work[2 * e];
      un.qb = p.work[2 * e + 1];
    }
    un.tok0 = p.cu_seqlens[un.seq];
    un.L = p.cu_seqlens[un.seq + 1] - un.tok0;
  } else {
    const int nqb = (p.N + kUnitRows - 1) / kUnitRows;
    int rank;
    if (is_split_mode(kMode)) {
      const int ranges = kMode == kModeSplitPair ? p.num_splits / 2 : p.num_splits;
      rank = e / (p.B * ranges);
      const int rem = e - rank * p.B * ranges;
      un.split = rem / p.B;
      un.seq = rem - un.split * p.B;
    } else {
      const int P = p.B * p.H;
      const int G = (p.pair_group > 0 && p.pair_group < P) ? p.pair_group : P;
      const int full = P / G;
      int gi, r, npg;
      if (u < full * G * nqb) {
        gi = u / (G * nqb);
        r = u - gi * G * nqb;
        npg = G;
      } else {
        gi = full;
        r = u - full * G * nqb;
        npg = P - full * G;
      }
      rank = r / npg;
      const int pair = gi * G + (r - rank * npg);
      un.seq = pair / p.H;
      un.h = pair - un.seq * p.H;
    }
    un.qb = nqb - 1 - rank;
    un.tok0 = un.seq * p.N;
    un.L = p.N;
  }
  if (is_split_mode(kMode)) {
    // visible KV tiles of the q-block, cut into num_splits near-equal ranges
    un.k_tok0 = un.seq * p.Nk;
    un.Lk = p.Nk;
    const int r_hi = min(un.qb * kUnitRows + kUnitRows, un.L) - 1;
    const int k_hi = p.causal ? min(p.Nk - 1, p.q_off + r_hi) : p.Nk - 1;
    const int n = k_hi / kBN + 1;
    const int s0 = kMode == kModeSplitPair ? 2 * un.split : un.split;
    un.kv0 = (int)((long long)n * s0 / p.num_splits);
    un.nkv = (int)((long long)n * (s0 + 1) / p.num_splits) - un.kv0;
    if (kMode == kModeSplitPair) {
      un.kv0b = (int)((long long)n * (s0 + 1) / p.num_splits);
      un.nkvb = (int)((long long)n * (s0 + 2) / p.num_splits) - un.kv0b;
    }
  } else {
    un.k_tok0 = un.tok0;
    un.Lk = un.L;
    unit_kv_range(un.L, un.qb, p.causal, p.wl, p.wr, un.kv0, un.nkv);
  }
  return un;
}

// First row (sequence-relative) actually loaded for query tile g: the nominal
// start, pulled back so the 128-row tile ends at the sequence end at the
// latest.  Rows before the nominal start are recomputed but never stored.
__device__ __forceinline__ int q_tile_start(const Unit& un, int g) {
  return min(un.qb * kUnitRows + g * kBM, un.L - kBM);
}
// First key actually loaded for KV tile j (same pull-back at the sequence end;
// keys before 128*j were already visited and are masked out).
__device__ __forceinline__ int kv_tile_start(const Unit& un, int j) {
  return min(j * kBN, un.Lk - kBN);
}

// KV tiles the lower query tile (group 0) of a unit visits: the unit's nkv,
// except that under a causal mask (or a right window) the unit's last tile is
// skipped when none of its keys not visited before is visible to any row of
// the lower tile (its first new key lies past the tile's last row): its S
// product, softmax and P V product would all be of masked keys.  The upper
// tile (group 1) visits every tile of the unit.
template <int kMode>
__device__ __forceinline__ int lower_tiles(const FwdParams& p, const Unit& un) {
  if (is_split_mode(kMode) || un.nkv < 2) return un.nkv;
  const int last_row = q_tile_start(un, 0) + kBM - 1;
  int k_hi = p.causal ? last_row : un.L - 1;
  if (kMode == kModeWindow && p.wr >= 0) k_hi = min(k_hi, last_row + p.wr);
  return k_hi < (un.kv0 + un.nkv - 1) * kBN ? un.nkv - 1 : un.nkv;
}

struct SharedState {
  uint64_t bars[kMaxBars];
  uint32_t tmem_base;
  volatile int abort_flag;
  volatile int unit_ring[kUnitSlots];
  Unit unit_dec[kUnitSlots];   // the published units, decoded by the producer
};

// Row maxima and sums exchanged by the two softmax warps that share rows.
struct RowExchange {
  float row_max[2][kQTiles][2][kBM];   // [tile parity][group][column half][row]
  float row_sum[kQTiles][2][2][kBM];   // [group][column half][l, l_fix][row]
};

// Bounded wait on an mbarrier phase; gives up on timeout or when another warp
// has aborted.  `where` identifies the wait in the error record.
__device__ __forceinline__ bool wait_bar(SharedState& ss, int bar, uint32_t parity,
                                         const FwdParams& p, int where) {
  const uint32_t a = smem_u32(&ss.bars[bar]);
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

__device__ __forceinline__ uint32_t bar_addr(SharedState& ss, int bar) {
  return smem_u32(&ss.bars[bar]);
}

// ------------------------------------------------------------ producer --
// kStages: slots of the K/V ring (the kernel's shared-memory layout decides);
// kQBufs: Q buffers, 1 or 2 (with 2 the Q tiles of unit n go to buffer n % 2,
// so they load while unit n - 1 still runs).
template <int D, int kMode, int kStages = FwdCfg<D>::kStages, int kQBufs = 1>
__device__ __forceinline__ void producer_loop(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                              const CUtensorMap* tm_v, const FwdParams& p,
                                              SharedState& ss, uint8_t* sQ, uint8_t* sRing,
                                              int n_units) {
  using C = FwdCfg<D>;
  uint32_t ring = 0;
  int units_done = 0;
  bool injected = false;
  uint32_t uslot = 0;
  int u = blockIdx.x;  // first unit static, then longest-first order by atomic pop
  for (;;) {
    if (u >= n_units) u = -1;
    // the unit is decoded once, here, and published with its index (the
    // producer runs ahead of its consumers, so the divisions are off their path)
    Unit un{};
    if (u >= 0) un = decode_unit<kMode>(p, u);
    {
      const int slot = uslot % kUnitSlots;
      const uint32_t n = uslot / kUnitSlots;
      if (n > 0 && !wait_bar(ss, kBarUnitEmpty + slot, (n - 1) & 1, p, 3)) return;
      ss.unit_dec[slot] = un;
      ss.unit_ring[slot] = u;
      mbar_arrive(bar_addr(ss, kBarUnitFull + slot));
      ++uslot;
    }
    if (u < 0) return;
    // next unit index, fetched while this unit's copies are issued
    const int next_u = (int)gridDim.x + atomicAdd(p.sched, 1);
    if (is_split_mode(kMode) && un.nkv <= 0 && un.nkvb <= 0) {  // empty KV ranges: nothing to copy
      u = next_u;
      continue;
    }
    {
      const int qb = units_done % kQBufs;
      const int qn = units_done / kQBufs;
      if (qn > 0 && !wait_bar(ss, bar_qempty(qb), (qn - 1) & 1, p, 1)) return;
      const uint32_t qfull = bar_addr(ss, bar_qfull(qb));
      uint8_t* sQb = sQ + qb * C::kSmemQ;
      mbar_arrive_expect_tx(qfull, kQTiles * C::kTileBytes);
      for (int g = 0; g < kQTiles; ++g) {
        // (paired ranges: both groups hold the unit's one query tile)
        const int r0 = un.tok0 + q_tile_start(un, kMode == kModeSplitPair ? 0 : g);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem_u32(sQb + g * C::kTileBytes + c * kChunkBytes), tm_q, qfull, c * 64,
                      un.h, r0);
      }
    }
    if constexpr (kMode == kModeSplitPair) {
      // the MMA thread's order: K_0(0), K_1(0), then per step j: V_0(j-1),
      // K_0(j), V_1(j-1), K_1(j), each while the group's range lasts
      const int nk[2] = {un.nkv, un.nkvb}, k0s[2] = {un.kv0, un.kv0b};
      auto push = [&](int kind, int g, int j) -> bool {
        const int slot = ring % kStages;
        const uint32_t n = ring / kStages;
        if (n > 0 && !wait_bar(ss, kBarKV + kStages + slot, (n - 1) & 1, p, 4)) return false;
        const uint32_t full = bar_addr(ss, kBarKV + slot);
        mbar_arrive_expect_tx(full, C::kTileBytes);
        const int k0 = un.k_tok0 + kv_tile_start(un, k0s[g] + j);
        const CUtensorMap* tm = kind == 0 ? tm_k : tm_v;
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem_u32(sRing + slot * C::kTileBytes + c * kChunkBytes), tm, full, c * 64,
                      un.h, k0);
        ++ring;
        return true;
      };
      for (int g = 0; g < kQTiles; ++g)
        if (nk[g] > 0 && !push(0, g, 0)) return;
      const int steps = max(nk[0], nk[1]);
      for (int j = 1; j <= steps; ++j)
        for (int g = 0; g < kQTiles; ++g) {
          if (j - 1 < nk[g] && !push(1, g, j - 1)) return;
          if (j < nk[g] && !push(0, g, j)) return;
        }
    } else {
      for (int j = 0; j < un.nkv; ++j) {
        const int k0 = un.k_tok0 + kv_tile_start(un, un.kv0 + j);
        for (int kind = 0; kind < 2; ++kind) {
          const int slot = ring % kStages;
          const uint32_t n = ring / kStages;
          if (n > 0 && !wait_bar(ss, kBarKV + kStages + slot, (n - 1) & 1, p, 2)) return;
          const uint32_t full = bar_addr(ss, kBarKV + slot);
          mbar_arrive_expect_tx(full, C::kTileBytes);
          if (p.fault_inject == 1 && blockIdx.x == 0 && !injected && kind == 0) {
            injected = true;  // test hook: the bytes this barrier waits for never come
          } else {
            const CUtensorMap* tm = kind == 0 ? tm_k : tm_v;
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(smem_u32(sRing + slot * C::kTileBytes + c * kChunkBytes), tm, full,
                          c * 64, un.h, k0);
          }
          ++ring;
        }
      }
    }
    ++units_done;
    u = next_u;
  }
}

// Unit index published by the producer for the consumer's next unit
// (-1: no more work), and with `un` the unit decoded.  `whole_warp`: the
// arrive on the slot's empty barrier comes from lane 0 of a warp after every
// lane has read it.
__device__ __forceinline__ bool next_unit(SharedState& ss, const FwdParams& p, uint32_t& uslot,
                                          bool whole_warp, int& u, Unit* un = nullptr) {
  const int slot = uslot % kUnitSlots;
  bool ok = wait_bar(ss, kBarUnitFull + slot, (uslot / kUnitSlots) & 1, p, 30);
  if (whole_warp) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return false;
  u = ss.unit_ring[slot];
  if (un) *un = ss.unit_dec[slot];
  if (whole_warp) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar_addr(ss, kBarUnitEmpty + slot));
  } else {
    mbar_arrive(bar_addr(ss, kBarUnitEmpty + slot));
  }
  ++uslot;
  return true;
}

// ----------------------------------------------------------------- MMA --
// S = Q K^T over D/16 MMAs of K-depth 16.  Both operands K-major, 128-byte
// swizzle: 64-element chunks of 128 rows each (16 KB apart), 8-row groups
// 1024 bytes apart; a 16-element step inside a chunk advances the start
// address by 32 bytes.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  using C = FwdCfg<D>;
  const uint64_t a0 = make_sdesc(q_smem, 16, 1024, kSwizzle128B);
  const uint64_t b0 = make_sdesc(k_smem, 16, 1024, kSwizzle128B);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (uint64_t)(((kk / 4) * kChunkBytes + (kk % 4) * 32) >> 4);
    mma_ss(d_tmem, a0 + off, b0 + off, C::kIdescS, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V over 128/16 MMAs.  P: bf16 pairs in TMEM (8 columns per 16
// keys).  V: MN-major (d contiguous), 128-byte swizzle: 64-element d chunks
// 16 KB apart (leading offset), 8-key groups 1024 bytes apart (stride
// offset); 16 keys advance the start address by 2048 bytes.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate) {
  using C = FwdCfg<D>;
  const uint64_t b0 = make_sdesc(v_smem, kChunkBytes, 1024, kSwizzle128B);
  const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk)
    mma_ts(d_tmem, p_tmem + kk * 8, b0 + (uint64_t)((kk * 2048) >> 4), C::kIdescPV,
           kk > 0 ? 1u : acc0);
}

// One unit of paired split-KV ranges: group g multiplies the unit's query
// tile with the KV tiles of its own range (group 0: kv0 .., group 1: kv0b ..),
// in the producer's order.  False when a wait gave up.
template <int D>
__device__ __forceinline__ bool mma_unit_pair(const FwdParams& p, SharedState& ss,
                                              const uint32_t (&q_smem)[2], uint8_t* sRing,
                                              uint32_t tmem, const Unit& un, int units_done,
                                              uint32_t& ring, uint32_t (&pcount)[2]) {
  using C = FwdCfg<D>;
  auto slot_smem = [&](uint32_t pos) { return smem_u32(sRing + (pos % C::kStages) * C::kTileBytes); };
  auto wait_full = [&](uint32_t pos) {
    return wait_bar(ss, kBarKV + pos % C::kStages, (pos / C::kStages) & 1, p, 15);
  };
  auto release = [&](uint32_t pos) { mma_commit(bar_addr(ss, kBarKV + C::kStages + pos % C::kStages)); };
  const int nk[2] = {un.nkv, un.nkvb};
  int s_left = nk[0] + nk[1];  // S products still to issue (Q is free after the last)
  if (!wait_bar(ss, kBarQFull, units_done & 1, p, 16)) return false;
  tc_fence_after();
  for (int g = 0; g < kQTiles; ++g) {
    if (nk[g] <= 0) continue;
    const uint32_t pos = ring++;
    if (!wait_full(pos)) return false;
    tc_fence_after();
    issue_qk<D>(tmem + C::col_s(g), q_smem[g], slot_smem(pos));
    mma_commit(bar_addr(ss, kBarSFull + g));
    release(pos);
    if (--s_left == 0) mma_commit(bar_addr(ss, kBarQEmpty));
  }
  const int steps = max(nk[0], nk[1]);
  for (int j = 1; j <= steps; ++j) {
    for (int g = 0; g < kQTiles; ++g) {
      if (j - 1 >= nk[g]) continue;
      const uint32_t posV = ring++;
      if (!wait_full(posV)) return false;
      // P_g of tile j-1 is in TMEM (and O_g rescaled if needed)
      if (!wait_bar(ss, kBarPFull + g, pcount[g] & 1, p, 17 + g)) return false;
      ++pcount[g];
      tc_fence_after();
      issue_pv<D>(tmem + C::col_o(g), tmem + C::col_s(g), slot_smem(posV), j > 1);
      release(posV);
      if (j < nk[g]) {
        const uint32_t posK = ring++;
        if (!wait_full(posK)) return false;
        tc_fence_after();
        issue_qk<D>(tmem + C::col_s(g), q_smem[g], slot_smem(posK));
        mma_commit(bar_addr(ss, kBarSFull + g));
        release(posK);
        if (--s_left == 0) mma_commit(bar_addr(ss, kBarQEmpty));
      } else {
        mma_commit(bar_addr(ss, kBarOFull + g));
      }
    }
  }
  return true;
}

// kQBufs: as for producer_loop.
template <int D, int kMode, int kQBufs = 1>
__device__ __forceinline__ void mma_loop(const FwdParams& p, SharedState& ss, uint8_t* sQ,
                                         uint8_t* sRing, uint32_t tmem, int n_units) {
  using C = FwdCfg<D>;
  uint32_t ring = 0;
  uint32_t pcount[2] = {0, 0};
  int units_done = 0;
  auto slot_smem = [&](uint32_t pos) { return smem_u32(sRing + (pos % C::kStages) * C::kTileBytes); };
  auto wait_full = [&](uint32_t pos) {
    return wait_bar(ss, kBarKV + pos % C::kStages, (pos / C::kStages) & 1, p, 10);
  };
  auto release = [&](uint32_t pos) { mma_commit(bar_addr(ss, kBarKV + C::kStages + pos % C::kStages)); };

  uint32_t uslot = 0;
  for (;;) {
    int u;
    if (!next_unit(ss, p, uslot, false, u) || u < 0) return;
    const Unit un = decode_unit<kMode>(p, u);
    // an empty KV range (split-KV with more ranges than tiles) has no copy,
    // no MMA and no barrier traffic: the softmax warps write its empty result
    if (kMode == kModeSplit && un.nkv <= 0) continue;
    if (kMode == kModeSplitPair) {
      if (un.nkv <= 0 && un.nkvb <= 0) continue;
      const uint32_t q_smem[2] = {smem_u32(sQ), smem_u32(sQ + C::kTileBytes)};
      if (!mma_unit_pair<D>(p, ss, q_smem, sRing, tmem, un, units_done, ring, pcount)) return;
      ++units_done;
      continue;
    }
    const int qb = units_done % kQBufs;
    const uint32_t q_smem[2] = {smem_u32(sQ + qb * C::kSmemQ),
                                smem_u32(sQ + qb * C::kSmemQ + C::kTileBytes)};
    if (!wait_bar(ss, bar_qfull(qb), (units_done / kQBufs) & 1, p, 11)) return;
    tc_fence_after();
    // group 0 may skip the unit's last tile (lower_tiles); group 1 visits all
    const int n0 = lower_tiles<kMode>(p, un);
    uint32_t posK = ring, posV = ring + 1;
    ring += 2;
    if (!wait_full(posK)) return;
    tc_fence_after();
    for (int g = 0; g < kQTiles; ++g) {
      issue_qk<D>(tmem + C::col_s(g), q_smem[g], slot_smem(posK));
      mma_commit(bar_addr(ss, kBarSFull + g));
    }
    release(posK);
    // Q is free for a later unit's copy once the unit's last S product is done
    if (un.nkv == 1) mma_commit(bar_addr(ss, bar_qempty(qb)));
    for (int j = 1; j <= un.nkv; ++j) {
      const bool more = j < un.nkv;
      uint32_t nextK = 0, nextV = 0;
      if (more) {
        nextK = ring;
        nextV = ring + 1;
        ring += 2;
      }
      if (!wait_full(posV)) return;
      // the next K tile before the first P: no wait between a group's P V
      // product and its next S product
      if (more && !wait_full(nextK)) return;
#pragma unroll
      for (int g = 0; g < kQTiles; ++g) {
        const int ng = g == 0 ? n0 : un.nkv;
        if (j <= ng) {
          // P_g of tile j-1 is in TMEM (and O_g rescaled if needed)
          if (!wait_bar(ss, kBarPFull + g, pcount[g] & 1, p, 12 + g)) return;
          ++pcount[g];
          tc_fence_after();
          issue_pv<D>(tmem + C::col_o(g), tmem + C::col_s(g), slot_smem(posV), j > 1);
        }
        if (g == kQTiles - 1) release(posV);
        if (more && j < ng) {
          issue_qk<D>(tmem + C::col_s(g), q_smem[g], slot_smem(nextK));
          mma_commit(bar_addr(ss, kBarSFull + g));
        } else if (j == ng) {
          mma_commit(bar_addr(ss, kBarOFull + g));
        }
      }
      if (more) {
        release(nextK);
        if (j == un.nkv - 1) mma_commit(bar_addr(ss, bar_qempty(qb)));
        posV = nextV;
      }
    }
    ++units_done;
  }
}

// ------------------------------------------------------------- softmax --
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// x rounded to the nearest bf16 (ties to even), as fp32.
__device__ __forceinline__ float bf16_round_f32(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (d0, d1) = (a0, a1) * b + c, one packed fp32x2 instruction.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n .reg .b64 x, y, z, r;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %4};\n"
      " mov.b64 z, {%5, %5};\n fma.rn.f32x2 r, x, y, z;\n mov.b64 {%0, %1}, r;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// (a0, a1) += (b0, b1), one packed fp32x2 instruction.
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{\n .reg .b64 x, y, r;\n mov.b64 x, {%0, %1};\n mov.b64 y, {%2, %3};\n"
      " add.rn.f32x2 r, x, y;\n mov.b64 {%0, %1}, r;\n}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// Barriers of the two warps that share a 32-row quadrant of a group: a named
// hardware barrier of 64 threads.  Both warps pass the same sequence of these
// barriers, also after a wait has given up: a warp whose wait failed goes on
// through the rest of its unit with the values it has (they are not a
// result; the kernel is stopping).  After every unit hand-off the pair passes
// one checking barrier, which leaves both warps with the OR of their failure
// flags; then both leave together if either failed, so neither is ever left
// waiting for a partner that has gone.
__device__ __forceinline__ void pair_sync(int g, int quadrant) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + g * 4 + quadrant) : "memory");
}

__device__ __forceinline__ bool pair_sync_check(int g, int quadrant, bool fail) {
  uint32_t any;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, %2, 64, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(any)
      : "r"(fail ? 1u : 0u), "r"(1 + g * 4 + quadrant)
      : "memory");
  return any != 0;
}

template <int D, int kMode>
__device__ __forceinline__ void softmax_loop(const FwdParams& p, SharedState& ss, RowExchange& xs,
                                             uint32_t tmem, int g, int n_units) {
  using C = FwdCfg<D>;
  constexpr int kOCols = D / 2;             // O columns rescaled / stored by this thread
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int quadrant = warp % 4;
  const int half = (warp % kGroupWarps) / 4;   // which 64 key columns
  const int trow = quadrant * 32 + lane;       // row within the tile = TMEM lane
  const uint32_t lane_addr = tmem + ((uint32_t)(quadrant * 32) << 16);
  const uint32_t colS = C::col_s(g) + half * kHalfCols;     // this thread's S columns
  const uint32_t colP = C::col_s(g) + half * (kHalfCols / 2);  // its packed P columns
  const uint32_t colO = C::col_o(g) + half * kOCols;
  const float c2 = p.scale_log2;
  uint32_t scount = 0;
  int units_done = 0;  // units with an O result (every unit but empty split-KV ranges)
  int tokens_total = 0;
  if (p.cu_seqlens) tokens_total = p.cu_seqlens[p.B];

  uint32_t uslot = 0;
  // A wait of this warp gave up: the pair leaves at the next checking barrier.
  // The next unit's index is taken in the epilogue of the current one, before
  // the checking barrier that ends it.
  int u = -1;
  bool fail = !next_unit(ss, p, uslot, true, u);
  if (pair_sync_check(g, quadrant, fail)) return;
  for (;;) {
    if (u < 0) return;
    Unit un = decode_unit<kMode>(p, u);
    // paired split-KV ranges: this group's range, its index, the one query tile
    const int tg = kMode == kModeSplitPair ? 0 : g;
    const int split_idx = kMode == kModeSplitPair ? 2 * un.split + g : un.split;
    if (kMode == kModeSplitPair && g == 1) {
      un.kv0 = un.kv0b;
      un.nkv = un.nkvb;
    }
    constexpr bool kWindow = kMode == kModeWindow;
    const int Lk = is_split_mode(kMode) ? un.Lk : un.L;
    const int q_off = is_split_mode(kMode) ? p.q_off : 0;  // key position of query row 0
    const int a0 = q_tile_start(un, tg);
    const int row = a0 + trow;                       // sequence-relative row of this thread
    const int nominal0 = un.qb * kUnitRows + tg * kBM;
    const int n_tiles = g == 0 ? lower_tiles<kMode>(p, un) : un.nkv;
    float m_used = -INFINITY;
    float l = 0.f;     // sum of the fp32 probabilities (this half): the LSE
    float l_fix = 0.f; // rounding change of each tile's largest probability (this half)
    for (int j = 0; j < n_tiles; ++j) {
      fail |= !__all_sync(0xffffffffu, wait_bar(ss, kBarSFull + g, scount & 1, p, 20 + g));
      ++scount;
      tc_fence_after();
      // (after a failed wait the loads read stale columns; the unit goes on
      // with them, its results are dropped and the warp leaves after it)
      float s[kHalfCols];
      {
        uint32_t r0[32], r1[32];
        tmem_ld_x32(lane_addr + colS, r0);
        tmem_ld_x32(lane_addr + colS + 32, r1);
        tmem_ld_wait_x32(r0);
        tmem_ld_wait_x32(r1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(r0[i]);
          s[32 + i] = __uint_as_float(r1[i]);
        }
      }
      // Mask: keys already visited by the previous tile (pulled-back last
      // tile), keys after this row when causal, keys outside the sliding
      // window.  The pull-back keeps every loaded key inside the sequence.
      // Decided per group, applied per row; column c of this thread is key
      // column half*64 + c.
      const int jt = un.kv0 + j;  // tile index within the sequence
      const int b0 = kv_tile_start(un, jt);
      // keys every row of the group may see: [max_klo, min_khi]
      const int max_klo = (kWindow && p.wl >= 0) ? max(0, a0 + kBM - 1 - p.wl) : 0;
      int min_khi = p.causal ? q_off + a0 : Lk - 1;
      if (kWindow && p.wr >= 0) min_khi = min(min_khi, a0 + p.wr);
      const bool need_mask = jt * kBN > b0 || b0 < max_klo || b0 + kBN - 1 > min_khi;
      if (need_mask) {
        // this row's keys [klo, khi]; keys below jt*128 were visited by the
        // previous tile (pulled-back last tile)
        int klo = (kWindow && p.wl >= 0) ? max(0, row - p.wl) : 0;
        int khi = p.causal ? q_off + row : Lk - 1;
        if (kWindow && p.wr >= 0) khi = min(khi, row + p.wr);
        klo = max(klo, jt * kBN);
        const int lo = klo - b0 - half * kHalfCols;
        const int hi = min(khi - b0, kBN - 1) - half * kHalfCols;
        // The visible columns [lo, hi] of a row are one range: each 32-column
        // chunk is masked from a bit mask of its visible columns.
#pragma unroll
        for (int k = 0; k < kHalfCols / 32; ++k) {
          const int lo_k = lo - 32 * k, hi_k = hi - 32 * k;
          const bool none = hi_k < 0 || lo_k > 31 || hi_k < lo_k;
          const uint32_t vis =
              none ? 0u : (0xffffffffu >> (31 - min(hi_k, 31))) & (0xffffffffu << max(lo_k, 0));
#pragma unroll
          for (int i = 0; i < 32; ++i) s[32 * k + i] = (vis >> i) & 1u ? s[32 * k + i] : -INFINITY;
        }
      }
      // row max: partial over this half (four 3-input max chains), then the
      // partner's half through shared memory
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
      float mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int c = 8; c < kHalfCols; c += 8) {
        mx0 = max3(mx0, s[c], s[c + 1]);
        mx1 = max3(mx1, s[c + 2], s[c + 3]);
        mx2 = max3(mx2, s[c + 4], s[c + 5]);
        mx3 = max3(mx3, s[c + 6], s[c + 7]);
      }
      const float mine = fmaxf(max3(mx0, mx1, mx2), mx3);
      xs.row_max[j & 1][g][half][trow] = mine;
      // (also orders both halves' S loads before any P store)
      pair_sync(g, quadrant);
      const float mx = fmaxf(mine, xs.row_max[j & 1][g][half ^ 1][trow]);
      const float m_new = fmaxf(m_used, mx);
      // O correction decision: only when the row max grew by more than 2^16
      // (warp-uniform; the partner warp holds the same rows and decides alike)
      // (a row whose keys so far were all hidden has O = 0 and l = 0: its
      // first visible key sets the reference without a rescale)
      float alpha = 1.0f;
      bool resc = false;
      if (m_used == -INFINITY) {
        m_used = m_new;
      } else if ((m_new - m_used) * c2 > kRescaleLog2) {
        resc = true;
        alpha = ex2_approx((m_used - m_new) * c2);
        m_used = m_new;
      }
      const bool rescale_warp = __any_sync(0xffffffffu, resc);
      const float neg = m_used == -INFINITY ? 0.f : -m_used * c2;
      // O is divided by l plus the bf16 rounding change of the largest
      // probability of every 64-key half tile: when one key dominates a row,
      // its rounding then cancels between O and the divisor (the other terms'
      // rounding errors are small and of both signs).  Same arithmetic as the
      // loop below, so this p_max is bit-identical to the one written to P.
      const float p_max = ex2_approx(fmaf(mine, c2, neg));
      const float fix = bf16_round_f32(p_max) - p_max;
      // p = 2^(c2 * s - c2 * m): packed fp32x2 FMA, MUFU ex2, packed sums
      float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
      uint32_t pw[32];
#pragma unroll
      for (int c = 0; c < kHalfCols; c += 4) {
        float x0, x1, x2, x3;
        fma2(x0, x1, s[c], s[c + 1], c2, neg);
        fma2(x2, x3, s[c + 2], s[c + 3], c2, neg);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
        add2(sa0, sa1, p0, p1);
        add2(sb0, sb1, p2, p3);
        pw[c / 2] = pack_bf16x2(p0, p1);
        pw[c / 2 + 1] = pack_bf16x2(p2, p3);
      }
      l = l * alpha + ((sa0 + sa1) + (sb0 + sb1));
      l_fix = l_fix * alpha + fix;
      // O *= alpha before this tile's PV product (after the exps, when the
      // scores no longer occupy registers)
      if (rescale_warp) {
#pragma unroll
        for (int cc = 0; cc < kOCols; cc += 32) {
          uint32_t r[32];
          tmem_ld_x32(lane_addr + colO + cc, r);
          tmem_ld_wait_x32(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st_x32(lane_addr + colO + cc, r);
        }
      }
      tmem_st_x32(lane_addr + colP, pw);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_addr(ss, kBarPFull + g));
    }
    // Epilogue: the two halves' sums are combined; O / l_r -> bf16 (each
    // thread its D/2 columns), LSE = scale * m + ln(l).  Rows before the
    // nominal tile start (recomputed) and rows past the sequence are skipped.
    xs.row_sum[g][half][0][trow] = l;
    xs.row_sum[g][half][1][trow] = l_fix;
    pair_sync(g, quadrant);
    l += xs.row_sum[g][half ^ 1][0][trow];
    const float l_r = l + l_fix + xs.row_sum[g][half ^ 1][1][trow];
    u = -1;
    if (!fail) fail = !next_unit(ss, p, uslot, true, u);
    // (also: both halves have read row_sum before the next unit writes it)
    if (pair_sync_check(g, quadrant, fail)) return;
    // (an empty KV range of split-KV has no MMA work and no O-done signal;
    // after a failed wait the kernel is stopping and what is stored below is
    // not a result)
    const bool has_o = !is_split_mode(kMode) || un.nkv > 0;
    if (has_o) {
      fail |= !__all_sync(0xffffffffu, wait_bar(ss, kBarOFull + g, units_done & 1, p, 22 + g));
      tc_fence_after();
    }
    const bool store = row >= nominal0 && row < un.L && row >= 0;
    if (is_split_mode(kMode)) {
      // partial result of this KV range: O / l_r (fp32) and its LSE; the
      // combine kernel merges the ranges
      const float inv = l_r > 0.f ? 1.0f / l_r : 0.f;
      float* prow = p.o_part + (((size_t)split_idx * p.B * p.N + (store ? un.tok0 + row : 0)) * p.H + un.h) * D +
                    half * kOCols;
#pragma unroll
      for (int cc = 0; cc < kOCols; cc += 32) {
        uint32_t r[32];
        if (has_o) {
          tmem_ld_x32(lane_addr + colO + cc, r);
          tmem_ld_wait_x32(r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (store) {
          float4* dst = reinterpret_cast<float4*>(prow + cc);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                 __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
        }
      }
      if (store && half == 0)
        p.lse_part[(((size_t)split_idx * p.B + un.seq) * p.H + un.h) * p.N + row] =
            l > 0.f ? m_used * p.scale + __log2f(l) * 0.69314718055994531f : -INFINITY;
      tc_fence_before();
      if (has_o) ++units_done;
      continue;
    }
    // O's divisor carries the rounding of each tile's dominant probability;
    // the LSE uses the fp32 sum.
    const float inv_l = l_r > 0.f ? 1.0f / l_r : 0.f;
    __nv_bfloat16* orow =
        p.o + ((size_t)(store ? un.tok0 + row : 0) * p.H + un.h) * D + half * kOCols;
#pragma unroll
    for (int cc = 0; cc < kOCols; cc += 32) {
      uint32_t r[32];
      tmem_ld_x32(lane_addr + colO + cc, r);
      tmem_ld_wait_x32(r);
      if (store) {
        uint4* dst = reinterpret_cast<uint4*>(orow + cc);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l);
          dst[i] = w;
        }
      }
    }
    if (store && half == 0) {
      const float lse = l > 0.f ? m_used * p.scale + __log2f(l) * 0.69314718055994531f : -INFINITY;
      size_t idx;
      if (p.cu_seqlens)
        idx = (size_t)un.h * tokens_total + un.tok0 + row;
      else
        idx = ((size_t)un.seq * p.H + un.h) * p.N + row;
      p.lse[idx] = lse;
    }
    tc_fence_before();
    ++units_done;
  }
}

// -------------------------------------------------------------- kernel --
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// kMode: kModeWindow applies the sliding-window bounds p.wl / p.wr;
// kModeSplit runs split-KV units and writes partial results.  Separate
// instantiations, so plain attention carries none of that arithmetic.
template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ SharedState ss;
  __shared__ RowExchange xs;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::kSmemQ;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(bar_addr(ss, kBarQFull), 1);
    mbar_init(bar_addr(ss, kBarQEmpty), 1);
    for (int g = 0; g < kQTiles; ++g) {
      mbar_init(bar_addr(ss, kBarSFull + g), 1);
      mbar_init(bar_addr(ss, kBarPFull + g), kGroupThreads);
      mbar_init(bar_addr(ss, kBarOFull + g), 1);
    }
    mbar_init(bar_addr(ss, kBarDrain), 1);
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(bar_addr(ss, kBarUnitFull + i), 1);
      mbar_init(bar_addr(ss, kBarUnitEmpty + i), kUnitConsumers);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_addr(ss, kBarKV + s), 1);
      mbar_init(bar_addr(ss, kBarKV + C::kStages + s), 1);
    }
    ss.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&ss.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ss.tmem_base;
  const int n_units = num_units<kMode>(p);

  if (warp >= kSoftmaxWarps) {
    setmaxnreg_dec<kControlRegs>();
    if (warp == kProducerWarp) {
      if (lane == 0) producer_loop<D, kMode>(&tm_q, &tm_k, &tm_v, p, ss, sQ, sRing, n_units);
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        mma_loop<D, kMode>(p, ss, sQ, sRing, tmem, n_units);
        // every MMA issued by this thread has finished before TMEM is freed
        mma_commit(bar_addr(ss, kBarDrain));
        mbar_wait(bar_addr(ss, kBarDrain), 0, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    setmaxnreg_inc<kSoftmaxRegs>();
    softmax_loop<D, kMode>(p, ss, xs, tmem, warp / kGroupWarps, n_units);
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
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0) {
    // every CTA has taken its last unit once all have arrived here: the last
    // one leaves the counters at zero for the next launch on this workspace
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
      __threadfence();
    }
  }
}

// ----------------------------------------------------------- scheduler --
// Builds the longest-first list of (sequence, q-block) pairs of a packed
// variable-length batch, validates cu_seqlens and zeroes the unit counters of
// the attention kernel that follows.  One CTA.  Cost of a pair =
// KV tiles it visits; a counting sort over cost in descending order.
constexpr int kMaxCostBuckets = 8192;

__global__ void __launch_bounds__(1024)
build_worklist_kernel(const int* cu_seqlens, int nseq, int max_len, int causal, int wl, int wr,
                      int* work, int* num_entries, int* err, int max_entries, int* sched) {
  extern __shared__ int hist[];  // [ncost + 1]
  __shared__ int bad;
  __shared__ int total;
  const int ncost = min((max_len + kBN - 1) / kBN, kMaxCostBuckets - 1);
  for (int i = threadIdx.x; i <= ncost; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) {
    bad = cu_seqlens[0] != 0;
    total = 0;
    sched[0] = 0;
    sched[1] = 0;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    if (L < 0 || L > max_len) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) {
      *num_entries = 0;
      atomicOr(err, kErrSeqlens);
    }
    return;
  }
  auto cost_of = [&](int L, int qb) {
    int kv0, nkv;
    unit_kv_range(L, qb, causal, wl, wr, kv0, nkv);
    return min(nkv, ncost);
  };
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    const int nqb = (L + kUnitRows - 1) / kUnitRows;
    for (int qb = 0; qb < nqb; ++qb) atomicAdd(&hist[cost_of(L, qb)], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0;
    for (int c = ncost; c >= 0; --c) {
      const int t = hist[c];
      hist[c] = off;
      off += t;
    }
    total = off;
  }
  __syncthreads();
  if (total > max_entries) {
    if (threadIdx.x == 0) {
      *num_entries = 0;
      atomicOr(err, kErrWorklist);
    }
    return;
  }
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    const int nqb = (L + kUnitRows - 1) / kUnitRows;
    for (int qb = 0; qb < nqb; ++qb) {
      const int pos = atomicAdd(&hist[cost_of(L, qb)], 1);
      work[2 * pos] = s;
      work[2 * pos + 1] = qb;
    }
  }
  if (threadIdx.x == 0) *num_entries = total;
}

// ------------------------------------------------------------- combine --
// Merges the split-KV partial results of every query row with the pages'
// two-segment merge identity applied across the KV ranges
// ("flash-attention-evolution" (letsgetai), FlashAttention "核心机制"): with
// LSE_s = m_s + ln l_s and O_s = f_s / l_s of range s,
//   m = max_s LSE_s,  w_s = e^{LSE_s - m},  LSE = m + ln sum_s w_s,
//   O = sum_s w_s O_s / sum_s w_s.
// One warp per (token, head) row; lane c holds columns c, c+32, ...
// valid: null, or a flag that is 0 when the inputs were rejected on the
// device (nothing is written then).
template <int D>
__global__ void __launch_bounds__(256)
attn_combine_kernel(const float* o_part, const float* lse_part, __nv_bfloat16* o, float* lse,
                    int B, int H, int Nq, int S, const int* valid = nullptr) {
  constexpr int kPer = D / 32;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const long long rows = (long long)B * Nq * H;
  if (warp >= rows || (valid && *valid == 0)) return;
  const long long tok = warp / H;
  const int h = (int)(warp - tok * H);
  const int b = (int)(tok / Nq);
  const int r = (int)(tok - (long long)b * Nq);
  float m = -INFINITY;
  for (int s = 0; s < S; ++s) m = fmaxf(m, lse_part[(((size_t)s * B + b) * H + h) * Nq + r]);
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float ls = lse_part[(((size_t)s * B + b) * H + h) * Nq + r];
      const float w = ls == -INFINITY ? 0.f : __expf(ls - m);
      wsum += w;
      const float* src = o_part + (((size_t)s * B * Nq + tok) * H + h) * D;
#pragma unroll
      for (int i = 0; i < kPer; ++i) acc[i] = fmaf(w, src[lane + 32 * i], acc[i]);
    }
  }
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  __nv_bfloat16* dst = o + (tok * H + h) * D;
#pragma unroll
  for (int i = 0; i < kPer; ++i) dst[lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
  if (lane == 0) lse[((size_t)b * H + h) * Nq + r] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
}

}  // namespace attn
