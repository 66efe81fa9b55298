// Fused exact softmax-attention forward on a pair of SMs (sm_103a), d = 128,
// plain masks (causal or none), dense or packed batches.
//
// The same computation as attn_fwd_kernel (tiles of Q, K, V; running row max
// m and row sum l; S and P never reach HBM; O and the row LSE out), with the
// devices the pages name for Blackwell: accumulators in TMEM, the 2-CTA MMA,
// a fully asynchronous MMA pipeline and conditional rescaling of O
// ("FlashAttention 1-4 演进速查" (argus-lessons), FlashAttention-4 items).
//
// A cluster of two CTAs (ranks 0 and 1, on two SMs) takes a work unit
// (sequence, head, 256 query rows); CTA r holds query tile r (128 rows).  The
// even CTA issues every product as tcgen05.mma.cta_group::2 of M = 256 rows:
//   S = Q K_j^T   A = Q from each CTA's shared memory (its 128 rows), B = K_j
//                 split by keys (CTA r holds keys 64 r .. 64 r + 63 of the tile);
//   O += P_j V_j  A = P_j from each CTA's TMEM, B = V_j split by columns (CTA
//                 r holds d columns 64 r .. 64 r + 63 of all 128 keys).
//
// Two softmax groups take the KV tiles of the stream in turn (tile i: group
// i % 2), each with its own S buffer and its own P area in TMEM, so the S
// product of a group's next tile is issued as soon as the group has read S
// of its current one and runs during its softmax, and the P V product of one
// group runs during the other group's softmax.  Both groups accumulate into
// one O: every tile decides the row's reference maximum M in the order of the
// tiles (a chain through shared memory), keeping the previous M unless the
// row maximum grew by more than 2^16 (then O and the row sums are rescaled
// once, before the tile's P V product), and computes P = 2^(c (S - M)) with
// it, so every P V product adds terms of one common reference.
//
// CTA layout (576 threads, one CTA per SM, no register split):
//   warps 0-7   softmax group 0, warps 8-15 group 1: warp w reads TMEM lanes
//               32 (w % 4) .. (its 32 rows) and key columns 64 h .. 64 h + 63
//               with h = (w % 8) / 4; the two warps of a group that share rows
//               exchange row maxima through shared memory at a named
//               barrier; at the end of a unit the four warps that share rows
//               combine row sums and write O and the LSE
//   warp  16    TMA producer (lane 0): this CTA's Q tile into a double buffer,
//               its halves of K_j, V_j into a ring; the "full" barriers live
//               in CTA 0 and count both CTAs' bytes
//   warp  17    lane 0 of CTA 0: MMA issuer; warp 17 of both CTAs owns TMEM
// Units go to clusters round robin in the longest-first order of
// decode_unit (a static schedule: both CTAs of a pair walk the same list).
//
// TMEM (512 columns, allocated for the pair): S_g [128 g, 128 g + 128) for
// group g, O [256, 384), P_g [384 + 64 g, 448 + 64 g) (bf16 pairs).
//
// Every wait is bounded; on a timeout a CTA records the error word, stops
// issuing work, lets copies land, frees TMEM with its partner and returns.
// Nothing here uses TMA multicast.
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn {

constexpr int kPairSoftmaxWarps = 16;
constexpr int kPairGroupWarps = 8;
constexpr int kPairProducerWarp = 16;
constexpr int kPairMmaWarp = 17;
constexpr int kPairThreads = 32 * 18;
constexpr int kPairStages = 8;          // ring slots of 16 KB: a K half or a V half
constexpr int kPairHalfBytes = 16384;   // K: 64 keys x 128; V: 128 keys x 64 columns
constexpr int kPairKChunkBytes = 8192;  // 64 keys x 64 columns (128-byte rows)
constexpr int kPairQBytes = 2 * kChunkBytes;  // one 128 x 128 query tile
constexpr int kPairSmemBytes = 2 * kPairQBytes + kPairStages * kPairHalfBytes + 1024;
constexpr uint32_t kPairColO = 256;
constexpr uint32_t kPairColP = 384;
constexpr uint32_t kPairIdescS = make_idesc_bf16(256, kBN, false);
constexpr uint32_t kPairIdescPV = make_idesc_bf16(256, 128, true);
constexpr uint16_t kPairBoth = 3;       // cluster ranks 0 and 1

// Barrier slots in each CTA's shared memory (g: softmax group, b: Q buffer).
enum : int {
  kPBarQFull = 0,    // +b, CTA 0: both CTAs' Q tiles landed (TMA bytes of both)
  kPBarQEmpty = 2,   // +b, both CTAs: the unit's last S product finished (commit)
  kPBarSFull = 4,    // +g, both CTAs: S_g written (commit)
  kPBarSFree = 6,    // +g, CTA 0: group g of both CTAs read S_g (16 warps)
  kPBarPFull = 8,    // +g, CTA 0: group g of both CTAs wrote P_g (16 warps)
  kPBarPVDone = 10,  // +g, both CTAs: P_g V finished (commit)
  kPBarDec = 12,     // + 4 (tile % 2) + quadrant: the tile's row decisions written (1 warp)
  kPBarDrain = 20,   // both CTAs: every product finished (commit)
  kPBarKV = 21,      // full[s] = kPBarKV + s (CTA 0: both halves' bytes),
                     // empty[s] = kPBarKV + kPairStages + s (both CTAs)
};
constexpr int kPairBars = kPBarKV + 2 * kPairStages;

struct PairShared {
  uint64_t bars[kPairBars];
  uint32_t tmem_base;
  volatile int abort_flag;
  float row_max[2][2][2][kBM];  // [group][tile parity of the group][column half][row]
  float dec_m[2][kBM];          // [tile % 2][row]: the reference maximum after the tile
  float dec_alpha[2][kBM];      // [tile % 2][row]: the tile's rescale factor (1: none)
  float row_sum[2][2][2][kBM];  // [group][column half][l, l_fix][row]
};

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t pbar(PairShared& ps, int b) { return smem_u32(&ps.bars[b]); }

// Bounded wait on a barrier of this CTA.  kCluster: the phase completes by
// arrivals of the other CTA's threads, whose writes the waiter then uses.
template <bool kCluster>
__device__ __forceinline__ bool pair_wait(PairShared& ps, int bar, uint32_t parity,
                                          const FwdParams& p, int where) {
  const uint32_t a = pbar(ps, bar);
  auto try_once = [&]() { return kCluster ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity); };
  if (try_once()) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (try_once()) return true;
    if (ps.abort_flag) return false;
    if (globaltimer_ns() - t0 > p.timeout_ns) {
      ps.abort_flag = 1;
      atomicOr(p.err, kErrTimeout);
      atomicCAS(p.err + 1, 0, where);
      return false;
    }
  }
}

// The KV tiles of a cluster's units, one after the other (the static
// schedule): unit u = cluster, cluster + clusters, ...; j: tile of the unit.
struct TileStream {
  int u, ul, j, n;
  Unit un;
  bool ok;
  __device__ __forceinline__ void start(const FwdParams& p, int n_units) {
    u = (int)cluster_id_x();
    ul = 0;
    j = 0;
    ok = u < n_units;
    if (ok) {
      un = decode_unit<kModePlain>(p, u);
      n = un.nkv;
    }
  }
  __device__ __forceinline__ void next(const FwdParams& p, int n_units) {
    if (++j < n) return;
    j = 0;
    ++ul;
    u += (int)num_clusters_x();
    ok = u < n_units;
    if (ok) {
      un = decode_unit<kModePlain>(p, u);
      n = un.nkv;
    }
  }
};

// ------------------------------------------------------------ producer --
__device__ __forceinline__ void pair_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                              const CUtensorMap* tm_v, const FwdParams& p,
                                              PairShared& ps, uint8_t* sQ, uint8_t* sRing,
                                              uint32_t rank, int n_units) {
  uint32_t pos = 0;
  int ul = 0;
  bool injected = false;
  for (int u = (int)cluster_id_x(); u < n_units; u += (int)num_clusters_x(), ++ul) {
    const Unit un = decode_unit<kModePlain>(p, u);
    // Q into buffer ul % 2, once the S products of unit ul - 2 have finished
    const int qb = ul & 1;
    if (ul >= 2 && !pair_wait<false>(ps, kPBarQEmpty + qb, ((ul >> 1) - 1) & 1, p, 41)) return;
    const uint32_t qfull = pbar(ps, kPBarQFull + qb);
    if (rank == 0) mbar_arrive_expect_tx(qfull, 2 * kPairQBytes);
    const uint32_t qmb = rank == 0 ? qfull : map_cluster(qfull, 0);
    const int r0 = un.tok0 + q_tile_start(un, (int)rank);
    for (int c = 0; c < 2; ++c)
      tma_load_3d_pair(smem_u32(sQ + qb * kPairQBytes + c * kChunkBytes), tm_q, qmb, c * 64, un.h, r0);
    for (int j = 0; j < un.nkv; ++j) {
      const int b0 = un.k_tok0 + kv_tile_start(un, un.kv0 + j);
      for (int kind = 0; kind < 2; ++kind, ++pos) {
        const int slot = pos % kPairStages;
        const uint32_t n = pos / kPairStages;
        if (n > 0 && !pair_wait<false>(ps, kPBarKV + kPairStages + slot, (n - 1) & 1, p, 42)) return;
        const uint32_t full = pbar(ps, kPBarKV + slot);
        // CTA 0's barrier counts both halves; CTA 1's copies complete on it
        if (rank == 0) mbar_arrive_expect_tx(full, 2 * kPairHalfBytes);
        const uint32_t mb = rank == 0 ? full : map_cluster(full, 0);
        const uint32_t dst = smem_u32(sRing + slot * kPairHalfBytes);
        if (kind == 0) {
          if (p.fault_inject == 1 && blockIdx.x == 0 && !injected) {
            injected = true;  // test hook: these bytes never come, a bounded wait expires
            continue;
          }
          for (int c = 0; c < 2; ++c)
            tma_load_3d_pair(dst + c * kPairKChunkBytes, tm_k, mb, c * 64, un.h, b0 + 64 * (int)rank);
        } else {
          tma_load_3d_pair(dst, tm_v, mb, 64 * (int)rank, un.h, b0);
        }
      }
    }
  }
}

// ----------------------------------------------------------------- MMA --
// CTA 0 only.  Tile i of the stream: S into S_{i%2} once group i % 2 has read
// S of tile i - 2, P V once the group has written P of tile i.  Order:
// S_0 S_1, then per tile i: S of tile i + 2, P V of tile i.
__device__ __forceinline__ void pair_mma(const FwdParams& p, PairShared& ps, uint8_t* sQ,
                                         uint8_t* sRing, uint32_t tmem, int n_units) {
  auto slot_of = [&](uint32_t q) { return (int)(q % kPairStages); };
  auto wait_full = [&](uint32_t q) {
    return pair_wait<false>(ps, kPBarKV + slot_of(q), (q / kPairStages) & 1, p, 43);
  };
  auto release = [&](uint32_t q) { mma_commit_pair(pbar(ps, kPBarKV + kPairStages + slot_of(q)), kPairBoth); };
  TileStream sc, pc;
  sc.start(p, n_units);
  pc.start(p, n_units);
  uint32_t is = 0, ip = 0;  // stream indices of the next S and the next P V
  auto issue_s = [&]() -> bool {
    const uint32_t g = is & 1;
    if (is >= 2 && !pair_wait<true>(ps, kPBarSFree + (int)g, ((is - 2) >> 1) & 1, p, 44)) return false;
    const int qb = sc.ul & 1;
    if (sc.j == 0 && !pair_wait<false>(ps, kPBarQFull + qb, (sc.ul >> 1) & 1, p, 45)) return false;
    if (!wait_full(2 * is)) return false;
    tc_fence_after();
    const uint64_t qd = make_sdesc(smem_u32(sQ + qb * kPairQBytes), 16, 1024, kSwizzle128B);
    const uint64_t kd = make_sdesc(smem_u32(sRing + slot_of(2 * is) * kPairHalfBytes), 16, 1024, kSwizzle128B);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss_pair(tmem + 128u * g, qd + (uint64_t)(((kk / 4) * kChunkBytes + (kk % 4) * 32) >> 4),
                  kd + (uint64_t)(((kk / 4) * kPairKChunkBytes + (kk % 4) * 32) >> 4), kPairIdescS,
                  kk > 0 ? 1u : 0u);
    mma_commit_pair(pbar(ps, kPBarSFull + (int)g), kPairBoth);
    release(2 * is);
    // Q buffer free for the unit after next once the unit's last S has finished
    if (sc.j == sc.n - 1) mma_commit_pair(pbar(ps, kPBarQEmpty + qb), kPairBoth);
    sc.next(p, n_units);
    ++is;
    return true;
  };
  for (int k = 0; k < 2 && sc.ok; ++k)
    if (!issue_s()) return;
  while (pc.ok) {
    if (sc.ok && !issue_s()) return;
    const uint32_t g = ip & 1;
    if (!wait_full(2 * ip + 1)) return;
    if (!pair_wait<true>(ps, kPBarPFull + (int)g, (ip >> 1) & 1, p, 46)) return;
    tc_fence_after();
    const uint64_t vd = make_sdesc(smem_u32(sRing + slot_of(2 * ip + 1) * kPairHalfBytes), kChunkBytes,
                                   1024, kSwizzle128B);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts_pair(tmem + kPairColO, tmem + kPairColP + 64u * g + 8 * kk, vd + (uint64_t)((kk * 2048) >> 4),
                  kPairIdescPV, (pc.j > 0 || kk > 0) ? 1u : 0u);
    release(2 * ip + 1);
    mma_commit_pair(pbar(ps, kPBarPVDone + (int)g), kPairBoth);
    pc.next(p, n_units);
    ++ip;
  }
}

// ------------------------------------------------------------- softmax --
__device__ __forceinline__ void group_pair_sync(int g, int quadrant) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + g * 4 + quadrant) : "memory");
}
__device__ __forceinline__ void quad_sync(int quadrant) {
  asm volatile("bar.sync %0, 128;" ::"r"(9 + quadrant) : "memory");
}
// The four warps that share rows pass this at the end of every unit: each gets
// the OR of their failure flags, so all four leave at the same point.
__device__ __forceinline__ bool quad_sync_check(int quadrant, bool fail) {
  uint32_t any;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(any)
      : "r"(fail ? 1u : 0u), "r"(9 + quadrant)
      : "memory");
  return any != 0;
}

// O *= alpha for 64 columns of this thread's row (rare: a row maximum grew by
// more than 2^16); kept out of line so that its registers do not weigh on
// the softmax loop.
__device__ __noinline__ void pair_rescale_o(uint32_t taddr, float alpha) {
#pragma unroll
  for (int cc = 0; cc < 64; cc += 32) {
    uint32_t r[32];
    tmem_ld_x32(taddr + cc, r);
    tmem_ld_wait_x32(r);
#pragma unroll
    for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
    tmem_st_x32(taddr + cc, r);
  }
}

// Waits on PVDone_{t%2} name the phase of the P V product of stream tile t by
// its parity, which is exact only while that barrier has completed product
// t - 2 and not t + 2.  Product t + 2 cannot start before P of tile t + 1 is
// written, which each wait below precedes; product t - 2 is made certain by an
// earlier wait (products finish in order).
__device__ __forceinline__ void pair_softmax(const FwdParams& p, PairShared& ps, uint32_t tmem,
                                             uint32_t rank, int n_units) {
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int quadrant = warp % 4;
  const int g = warp / kPairGroupWarps;          // softmax group: tiles i with i % 2 == g
  const int half = (warp % kPairGroupWarps) / 4; // key columns 64 half .. 64 half + 63
  const int trow = quadrant * 32 + lane;         // row within the tile = TMEM lane
  const uint32_t lane_addr = tmem + ((uint32_t)(quadrant * 32) << 16);
  const float c2 = p.scale_log2;
  // arrivals on CTA 0's barriers: local there, through the cluster window from CTA 1
  const uint32_t sfree = rank == 0 ? pbar(ps, kPBarSFree + g) : map_cluster(pbar(ps, kPBarSFree + g), 0);
  const uint32_t pfull = rank == 0 ? pbar(ps, kPBarPFull + g) : map_cluster(pbar(ps, kPBarPFull + g), 0);
  auto arrive_leader = [&](uint32_t a) {
    if (rank == 0)
      mbar_arrive(a);
    else
      mbar_arrive_cluster(a);
  };
  // P V of stream tile t (group t % 2) has finished: phase t / 2 of PVDone_{t%2}
  auto pv_done = [&](uint32_t t, int where) {
    return pair_wait<false>(ps, kPBarPVDone + (int)(t & 1), (t >> 1) & 1, p, where);
  };
  // the row decisions of stream tile t are written: phase t / 2 of Dec_{t%2, quadrant}
  auto dec_ready = [&](uint32_t t, int where) {
    return pair_wait<false>(ps, kPBarDec + 4 * (int)(t & 1) + quadrant, (t >> 1) & 1, p, where);
  };
  int tokens_total = 0;
  if (p.cu_seqlens) tokens_total = p.cu_seqlens[p.B];

  bool fail = false;
  uint32_t i = 0;  // stream index of the unit's first tile
  for (int u = (int)cluster_id_x(); u < n_units; u += (int)num_clusters_x()) {
    const Unit un = decode_unit<kModePlain>(p, u);
    const int n = un.nkv;
    const int a0 = q_tile_start(un, (int)rank);
    const int row = a0 + trow;                    // sequence-relative row of this thread
    const int nominal0 = un.qb * kUnitRows + (int)rank * kBM;
    // tiles with a key visible to this CTA's rows (the lower tile of a causal
    // unit may see none of the last one: its P is then 0, no exponentials)
    const int n_mine = rank == 0 ? lower_tiles<kModePlain>(p, un) : n;
    float m_ref = -INFINITY;  // the row's reference maximum after the last decided tile
    float l = 0.f, l_fix = 0.f;
    for (int j = 0; j < n; ++j) {
      const uint32_t t = i + j;
      if ((int)(t & 1) != g) continue;
      const uint32_t gp = (t >> 1) & 1;  // phase of this group's barriers for tile t
      fail |= !__all_sync(0xffffffffu, pair_wait<false>(ps, kPBarSFull + g, gp, p, 47));
      tc_fence_after();
      const bool visible = j < n_mine;
      // This thread's 64 scores are read from TMEM twice, 32 at a time: for
      // the row maximum and then for the exponentials, so that at most 32
      // occupy registers (S_g is released after the second reading).
      // Mask: keys visited by the previous tile (pulled-back last tile) and,
      // when causal, keys after this row: visible columns [lo, hi] of the 64.
      const int jt = un.kv0 + j;
      const int b0 = kv_tile_start(un, jt);
      const bool need_mask = jt * kBN > b0 || b0 + kBN - 1 > (p.causal ? a0 : un.L - 1);
      const int lo = jt * kBN - b0 - kHalfCols * half;
      const int hi = min((p.causal ? row : un.L - 1) - b0, kBN - 1) - kHalfCols * half;
      auto load_chunk = [&](int k, float (&sc)[32]) {
        uint32_t r[32];
        tmem_ld_x32(lane_addr + 128u * g + 64u * half + 32u * k, r);
        tmem_ld_wait_x32(r);
        const int lo_k = lo - 32 * k, hi_k = hi - 32 * k;
        const bool none = hi_k < 0 || lo_k > 31 || hi_k < lo_k;
        const uint32_t vis = !need_mask ? 0xffffffffu
                             : none     ? 0u
                                        : (0xffffffffu >> (31 - min(hi_k, 31))) & (0xffffffffu << max(lo_k, 0));
#pragma unroll
        for (int c = 0; c < 32; ++c) sc[c] = (vis >> c) & 1u ? __uint_as_float(r[c]) : -INFINITY;
      };
      float mine = -INFINITY;
      if (visible) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          float sc[32];
          load_chunk(k, sc);
          float mx0 = fmaxf(sc[0], sc[1]), mx1 = fmaxf(sc[2], sc[3]);
          float mx2 = fmaxf(sc[4], sc[5]), mx3 = fmaxf(sc[6], sc[7]);
#pragma unroll
          for (int c = 8; c < 32; c += 8) {
            mx0 = max3(mx0, sc[c], sc[c + 1]);
            mx1 = max3(mx1, sc[c + 2], sc[c + 3]);
            mx2 = max3(mx2, sc[c + 4], sc[c + 5]);
            mx3 = max3(mx3, sc[c + 6], sc[c + 7]);
          }
          mine = fmaxf(mine, fmaxf(max3(mx0, mx1, mx2), mx3));
        }
      }
      // the previous tile's decision (the other group's, in the stream order;
      // a unit's first tile starts afresh but still waits, so that the slot
      // this tile writes below has been read by every reader)
      float alpha_prev = 1.0f;
      if (t > 0) {
        fail |= !__all_sync(0xffffffffu, dec_ready(t - 1, 48));
        if (j > 0) {
          m_ref = ps.dec_m[(t - 1) & 1][trow];
          alpha_prev = ps.dec_alpha[(t - 1) & 1][trow];
        }
      }
      l *= alpha_prev;
      l_fix *= alpha_prev;
      ps.row_max[g][gp][half][trow] = mine;
      // (also: both halves have read the previous decision before one of them
      // publishes this tile's, which releases the other group to overwrite it)
      group_pair_sync(g, quadrant);
      const float mx = fmaxf(mine, ps.row_max[g][gp][half ^ 1][trow]);
      const float m_new = fmaxf(m_ref, mx);
      float alpha = 1.0f;
      bool resc = false;
      if (m_ref == -INFINITY) {
        m_ref = m_new;  // nothing visible so far: O and l are 0 for this row
      } else if ((m_new - m_ref) * c2 > kRescaleLog2) {
        resc = true;
        alpha = ex2_approx((m_ref - m_new) * c2);
        m_ref = m_new;
      }
      // publish the decision of tile t (one warp per quadrant writes its rows)
      if (half == 0) {
        ps.dec_m[t & 1][trow] = m_ref;
        ps.dec_alpha[t & 1][trow] = alpha;
        __syncwarp();
        if (lane == 0) mbar_arrive(pbar(ps, kPBarDec + 4 * (int)(t & 1) + quadrant));
      }
      const bool rescale_warp = __any_sync(0xffffffffu, resc);
      // P_g is free once the P V product of tile t - 2 has finished (this
      // group waited for t - 4 at its previous tile); waited before the
      // exponentials, while P does not occupy registers yet
      if (t >= 2) {
        fail |= !__all_sync(0xffffffffu, pv_done(t - 2, 49));
        tc_fence_after();
      }
      // P in two halves of 32 keys, each stored to TMEM as soon as it is
      // packed (the P V product waits for the arrival below), so that at most
      // 16 packed words occupy registers beside the scores
      const uint32_t p_addr = lane_addr + kPairColP + 64u * g + 32u * half;
      if (visible) {
        const float neg = m_ref == -INFINITY ? 0.f : -m_ref * c2;
        // O's divisor carries the bf16 rounding change of the largest
        // probability of these 64 keys (same arithmetic as below)
        const float p_max = ex2_approx(fmaf(mine, c2, neg));
        const float fix = bf16_round_f32(p_max) - p_max;
        float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          float sc[32];
          load_chunk(k, sc);
          uint32_t pw[16];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            float x0, x1, x2, x3;
            fma2(x0, x1, sc[c], sc[c + 1], c2, neg);
            fma2(x2, x3, sc[c + 2], sc[c + 3], c2, neg);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            add2(sa0, sa1, p0, p1);
            add2(sb0, sb1, p2, p3);
            pw[c / 2] = pack_bf16x2(p0, p1);
            pw[c / 2 + 1] = pack_bf16x2(p2, p3);
          }
          tmem_st_x16(p_addr + 16u * k, pw);
        }
        l = l * alpha + ((sa0 + sa1) + (sb0 + sb1));
        l_fix = l_fix * alpha + fix;
      } else {
        uint32_t pw[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pw[c] = 0u;
        tmem_st_x16(p_addr, pw);
        tmem_st_x16(p_addr + 16u, pw);
      }
      // S_g is read: the S product of this group's next tile may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(sfree);
      if (rescale_warp) {
        // O *= alpha once every earlier product has finished (t - 3 has: t - 2
        // has); this thread: its row, d columns 64 half .. 64 half + 63
        if (t >= 1) {
          fail |= !pv_done(t - 1, 50);
          tc_fence_after();
        }
        pair_rescale_o(lane_addr + kPairColO + 64u * half, alpha);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(pfull);
    }
    // unit end: if the other group took the unit's last tile, its decision is
    // the row's final reference maximum and rescale
    const uint32_t t_last = i + (uint32_t)n - 1;
    const bool mine_last = (int)(t_last & 1) == g;
    if (!mine_last) {
      fail |= !__all_sync(0xffffffffu, dec_ready(t_last, 51));
      m_ref = ps.dec_m[t_last & 1][trow];
      const float a = ps.dec_alpha[t_last & 1][trow];
      l *= a;
      l_fix *= a;
    }
    // the four warps sharing rows combine their sums
    ps.row_sum[g][half][0][trow] = l;
    ps.row_sum[g][half][1][trow] = l_fix;
    quad_sync(quadrant);
    float l_all = 0.f, fix_all = 0.f;
#pragma unroll
    for (int gg = 0; gg < 2; ++gg)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        l_all += ps.row_sum[gg][hh][0][trow];
        fix_all += ps.row_sum[gg][hh][1][trow];
      }
    // (also: all four warps have read row_sum before the next unit writes it)
    if (quad_sync_check(quadrant, fail)) return;
    // the unit's last P V product; the other group first waits for its own
    // last one (tile t_last - 1), which makes t_last - 2 certain
    if (!mine_last && n > 1) {
      fail |= !__all_sync(0xffffffffu, pv_done(t_last - 1, 52));
    }
    fail |= !__all_sync(0xffffffffu, pv_done(t_last, 53));
    tc_fence_after();
    const float l_r = l_all + fix_all;
    const bool store = row >= nominal0 && row < un.L && row >= 0;
    const float inv_l = l_r > 0.f ? 1.0f / l_r : 0.f;
    const int part = 2 * g + half;  // this warp's 32 d columns of O
    {
      uint32_t r[32];
      tmem_ld_x32(lane_addr + kPairColO + 32u * part, r);
      tmem_ld_wait_x32(r);
      if (store) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)(un.tok0 + row) * p.H + un.h) * 128 + 32 * part);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(r[8 * k + 0]) * inv_l, __uint_as_float(r[8 * k + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv_l, __uint_as_float(r[8 * k + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv_l, __uint_as_float(r[8 * k + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv_l, __uint_as_float(r[8 * k + 7]) * inv_l);
          dst[k] = w;
        }
      }
    }
    if (store && part == 0) {
      const float lse = l_all > 0.f ? m_ref * p.scale + __log2f(l_all) * 0.69314718055994531f : -INFINITY;
      size_t idx;
      if (p.cu_seqlens)
        idx = (size_t)un.h * tokens_total + un.tok0 + row;
      else
        idx = ((size_t)un.seq * p.H + un.h) * p.N + row;
      p.lse[idx] = lse;
    }
    tc_fence_before();
    i += (uint32_t)n;
  }
}

// -------------------------------------------------------------- kernel --
// 576 threads: 96 registers each (two of the SM's four register-file quarters
// hold five warps).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ PairShared ps;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + 2 * kPairQBytes;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(pbar(ps, kPBarQFull + b), 1);
      mbar_init(pbar(ps, kPBarQEmpty + b), 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(pbar(ps, kPBarSFull + g), 1);
      mbar_init(pbar(ps, kPBarSFree + g), 2 * kPairGroupWarps);
      mbar_init(pbar(ps, kPBarPFull + g), 2 * kPairGroupWarps);
      mbar_init(pbar(ps, kPBarPVDone + g), 1);
    }
    for (int d = 0; d < 8; ++d) mbar_init(pbar(ps, kPBarDec + d), 1);
    mbar_init(pbar(ps, kPBarDrain), 1);
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(pbar(ps, kPBarKV + s), 1);
      mbar_init(pbar(ps, kPBarKV + kPairStages + s), 1);
    }
    ps.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kPairProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == kPairMmaWarp) {
    tmem_alloc_pair(smem_u32(&ps.tmem_base), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs' barriers are initialised before either CTA's commits, copies
  // or arrivals reach the other
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = ps.tmem_base;
  const int n_units = num_units<kModePlain>(p);

  if (warp == kPairProducerWarp) {
    if (lane == 0) pair_producer(&tm_q, &tm_k, &tm_v, p, ps, sQ, sRing, rank, n_units);
  } else if (warp == kPairMmaWarp) {
    if (lane == 0) {
      if (rank == 0) {
        pair_mma(p, ps, sQ, sRing, tmem, n_units);
        // every product has finished before either CTA frees TMEM
        mma_commit_pair(pbar(ps, kPBarDrain), kPairBoth);
      }
      if (!mbar_wait(pbar(ps, kPBarDrain), 0, 200000000ull)) ps.abort_flag = 1;
    }
  } else {
    pair_softmax(p, ps, tmem, rank, n_units);
  }
  __syncwarp();

  if (ps.abort_flag) {
    // copies issued before the abort may still be landing: give them 1 ms
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  // neither CTA frees TMEM or leaves while the other may still reach it
  cluster_sync();
  if (warp == kPairMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace attn
