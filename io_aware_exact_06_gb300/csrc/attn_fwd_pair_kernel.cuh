// Fused exact softmax-attention forward on a pair of SMs (sm_103a), d = 128,
// plain masks (causal or none), dense or packed batches.
//
// The same computation as attn_fwd_kernel (tiles of Q, K, V; running row max
// m and row sum l; S and P never reach HBM; O and the row LSE out), with the
// two devices the pages name for the shared-memory traffic of the tensor core
// on Blackwell: accumulators in TMEM and the 2-CTA MMA ("FlashAttention 1-4
// 演进速查" (argus-lessons), FlashAttention-4 items and the forward roofline
// table with the remedies under it).
//
// A cluster of two CTAs (ranks 0 and 1, on two SMs) takes a work unit
// (sequence, head, 256 query rows); CTA r holds query tile r (128 rows).  The
// even CTA issues every product as tcgen05.mma.cta_group::2 of M = 256 rows:
//   S_b = Q K_j^T   A = Q from each CTA's TMEM (its 128 rows), B = K_j split
//                   by keys (CTA r holds keys 64 r .. 64 r + 63 of the tile);
//   O  += P_j V_j   A = P_j from each CTA's TMEM, B = V_j split by columns
//                   (CTA r holds d columns 64 r .. 64 r + 63 of all 128 keys).
// So each SM reads 2 KB of shared memory per 64-cycle product and no query
// operand at all.  S is double-buffered: the product of tile j + 1 (issued
// when P_{j-1} was consumed) runs while the softmax warps work on tile j, and
// the P V product of tile j runs while they work on tile j + 1.
//
// CTA layout (576 threads, one CTA per SM, no register split):
//   warps 0-15  softmax: warp w reads TMEM lanes 32 (w % 4) .. (its 32 rows)
//               and key columns 32 (w / 4) .. + 31 of the tile; the four warps
//               of a row quadrant exchange row maxima and sums through shared
//               memory at a named barrier; they also copy the unit's Q tile
//               from shared memory into TMEM and write the O epilogue
//   warp  16    TMA producer (lane 0): this CTA's Q tile, then its halves of
//               K_j, V_j into a ring whose "full" barriers live in CTA 0 and
//               count both CTAs' bytes
//   warp  17    lane 0 of CTA 0: MMA issuer; warp 17 of both CTAs owns TMEM
// Units go to clusters round robin in the longest-first order of
// decode_unit (a static schedule: both CTAs of a pair walk the same list).
//
// TMEM (512 columns, allocated for the pair): S_0 [0, 128), S_1 [128, 256),
// O [256, 384), Q_u [384 + 64 u, 448 + 64 u) for unit parity u (bf16 pairs).
// P_j overwrites the first 64 columns of S_{j % 2} (bf16 pairs).
//
// Every wait is bounded; on a timeout a CTA records the error word, stops
// issuing work, lets copies land, frees TMEM with its partner and returns.
// Nothing here uses TMA multicast.
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn {

constexpr int kPairSoftmaxWarps = 16;
constexpr int kPairProducerWarp = 16;
constexpr int kPairMmaWarp = 17;
constexpr int kPairThreads = 32 * 18;
constexpr int kPairStages = 8;          // ring slots of 16 KB: a K half or a V half
constexpr int kPairHalfBytes = 16384;   // K: 64 keys x 128; V: 128 keys x 64 columns
constexpr int kPairKChunkBytes = 8192;  // 64 keys x 64 columns (128-byte rows)
constexpr int kPairQBytes = 2 * kChunkBytes;
constexpr int kPairSmemBytes = kPairQBytes + kPairStages * kPairHalfBytes + 1024;
constexpr uint32_t kPairColO = 256;
constexpr uint32_t kPairColQ = 384;
constexpr uint32_t kPairIdescS = make_idesc_bf16(256, kBN, false);
constexpr uint32_t kPairIdescPV = make_idesc_bf16(256, 128, true);
constexpr uint16_t kPairBoth = 3;       // cluster ranks 0 and 1

// Barrier slots in each CTA's shared memory.
enum : int {
  kPBarQFull = 0,    // this CTA's Q tile landed (TMA bytes)
  kPBarQEmpty = 1,   // this CTA's softmax warps copied Q to TMEM (16 warps)
  kPBarQReady = 2,   // CTA 0: both CTAs' Q is in TMEM (32 warps)
  kPBarSFull = 3,    // +b: S_b written (CTA 0's commit, both CTAs)
  kPBarPFull = 5,    // +(g % 2), CTA 0: both CTAs' P of tile g is in TMEM (32 warps)
  kPBarPVDone = 7,   // +(g % 2): P V product g finished (CTA 0's commit, both CTAs)
  kPBarDrain = 9,    // every product finished (CTA 0's commit, both CTAs)
  kPBarKV = 10,      // full[s] = kPBarKV + s (CTA 0: both halves' bytes),
                     // empty[s] = kPBarKV + kPairStages + s (both CTAs)
};
constexpr int kPairBars = kPBarKV + 2 * kPairStages;

struct PairShared {
  uint64_t bars[kPairBars];
  uint32_t tmem_base;
  volatile int abort_flag;
  float row_max[2][4][kBM];  // [tile parity][column quarter][row]
  float row_sum[4][2][kBM];  // [column quarter][l, l_fix][row]
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
    if (ul > 0 && !pair_wait<false>(ps, kPBarQEmpty, (ul - 1) & 1, p, 41)) return;
    mbar_arrive_expect_tx(pbar(ps, kPBarQFull), kPairQBytes);
    const int r0 = un.tok0 + q_tile_start(un, (int)rank);
    for (int c = 0; c < 2; ++c)
      tma_load_3d(smem_u32(sQ + c * kChunkBytes), tm_q, pbar(ps, kPBarQFull), c * 64, un.h, r0);
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
// CTA 0 only.  Per unit: S of tiles 0 and 1, then per tile j: P_j V_j and
// S of tile j + 2 into the buffer P_j leaves.
__device__ __forceinline__ void pair_mma(const FwdParams& p, PairShared& ps, uint8_t* sRing,
                                         uint32_t tmem, int n_units) {
  uint32_t pos = 0, t = 0, pvc = 0;
  int ul = 0;
  auto slot_of = [&](uint32_t q) { return (int)(q % kPairStages); };
  auto wait_full = [&](uint32_t q) {
    return pair_wait<false>(ps, kPBarKV + slot_of(q), (q / kPairStages) & 1, p, 43);
  };
  auto release = [&](uint32_t q) { mma_commit_pair(pbar(ps, kPBarKV + kPairStages + slot_of(q)), kPairBoth); };
  for (int u = (int)cluster_id_x(); u < n_units; u += (int)num_clusters_x(), ++ul) {
    const Unit un = decode_unit<kModePlain>(p, u);
    const int n = un.nkv;
    if (!pair_wait<true>(ps, kPBarQReady, ul & 1, p, 44)) return;
    tc_fence_after();
    const uint32_t qc = tmem + kPairColQ + 64u * (uint32_t)(ul & 1);
    auto issue_s = [&](int j) -> bool {
      const uint32_t kq = pos + 2 * j;
      if (!wait_full(kq)) return false;
      tc_fence_after();
      const uint32_t b = (t + j) & 1;
      const uint64_t kd = make_sdesc(smem_u32(sRing + slot_of(kq) * kPairHalfBytes), 16, 1024, kSwizzle128B);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts_pair(tmem + 128u * b, qc + 8 * kk,
                    kd + (uint64_t)(((kk / 4) * kPairKChunkBytes + (kk % 4) * 32) >> 4), kPairIdescS,
                    kk > 0 ? 1u : 0u);
      mma_commit_pair(pbar(ps, kPBarSFull + b), kPairBoth);
      release(kq);
      return true;
    };
    if (!issue_s(0)) return;
    if (n > 1 && !issue_s(1)) return;
    for (int j = 0; j < n; ++j) {
      const uint32_t vq = pos + 2 * j + 1;
      if (!wait_full(vq)) return;
      if (!pair_wait<true>(ps, kPBarPFull + (int)(pvc & 1), (pvc >> 1) & 1, p, 45)) return;
      tc_fence_after();
      const uint32_t b = (t + j) & 1;
      const uint64_t vd = make_sdesc(smem_u32(sRing + slot_of(vq) * kPairHalfBytes), kChunkBytes, 1024,
                                     kSwizzle128B);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts_pair(tmem + kPairColO, tmem + 128u * b + 8 * kk, vd + (uint64_t)((kk * 2048) >> 4),
                    kPairIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
      release(vq);
      mma_commit_pair(pbar(ps, kPBarPVDone + (pvc & 1)), kPairBoth);
      ++pvc;
      if (j + 2 < n && !issue_s(j + 2)) return;
    }
    t += n;
    pos += 2 * n;
  }
}

// ------------------------------------------------------------- softmax --
__device__ __forceinline__ void quad_sync(int quadrant) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + quadrant) : "memory");
}

// The four warps of a row quadrant pass this at the end of every unit: each
// gets the OR of their failure flags, so all four leave at the same point.
__device__ __forceinline__ bool quad_sync_check(int quadrant, bool fail) {
  uint32_t any;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(any)
      : "r"(fail ? 1u : 0u), "r"(1 + quadrant)
      : "memory");
  return any != 0;
}

__device__ __forceinline__ void pair_softmax(const FwdParams& p, PairShared& ps, const uint8_t* sQ,
                                             uint32_t tmem, uint32_t rank, int n_units) {
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int quadrant = warp % 4;
  const int w4 = warp / 4;                 // which 32 key columns (and d columns of O)
  const int trow = quadrant * 32 + lane;   // row within the tile = TMEM lane
  const uint32_t lane_addr = tmem + ((uint32_t)(quadrant * 32) << 16);
  const float c2 = p.scale_log2;
  // arrivals on CTA 0's barriers: local in CTA 0, through the cluster window in
  // CTA 1.  P of tile g goes to PFull + g % 2: S of tile g + 1 is issued before
  // P of tile g is consumed, so a warp may write P of tile g + 1 while another
  // still works on tile g (its arrival must not count for tile g), but not P
  // of tile g + 2 (S of tile g + 2 waits for the P V product of tile g).
  uint32_t pfull[2];
  for (int i = 0; i < 2; ++i)
    pfull[i] = rank == 0 ? pbar(ps, kPBarPFull + i) : map_cluster(pbar(ps, kPBarPFull + i), 0);
  const uint32_t qready = rank == 0 ? pbar(ps, kPBarQReady) : map_cluster(pbar(ps, kPBarQReady), 0);
  auto arrive_leader = [&](uint32_t a) {
    if (rank == 0)
      mbar_arrive(a);
    else
      mbar_arrive_cluster(a);
  };
  int tokens_total = 0;
  if (p.cu_seqlens) tokens_total = p.cu_seqlens[p.B];

  bool fail = false;
  // Q tile of unit ul: shared memory (128-byte swizzle) -> TMEM Q_{ul % 2};
  // this thread: its row, d columns 32 w4 .. 32 w4 + 31 (64 bytes)
  auto copy_q = [&](int ulq) {
    fail |= !__all_sync(0xffffffffu, pair_wait<false>(ps, kPBarQFull, ulq & 1, p, 46));
    const uint8_t* rowp = sQ + (w4 / 2) * kChunkBytes + trow * 128;
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int unit16 = (4 * (w4 % 2) + i) ^ (trow & 7);
      const uint4 x = *reinterpret_cast<const uint4*>(rowp + unit16 * 16);
      r[4 * i] = x.x;
      r[4 * i + 1] = x.y;
      r[4 * i + 2] = x.z;
      r[4 * i + 3] = x.w;
    }
    tmem_st_x16(lane_addr + kPairColQ + 64u * (uint32_t)(ulq & 1) + 16u * w4, r);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(pbar(ps, kPBarQEmpty));
      arrive_leader(qready);
    }
  };

  uint32_t t = 0;
  uint32_t pv0 = 0;  // P V products of the units before this one
  auto pv_done = [&](uint32_t g, int where) {
    return pair_wait<false>(ps, kPBarPVDone + (int)(g & 1), (g >> 1) & 1, p, where);
  };
  int ul = 0;
  const int u0 = (int)cluster_id_x(), ustep = (int)num_clusters_x();
  if (u0 < n_units) copy_q(0);
  for (int u = u0; u < n_units; u += ustep, ++ul) {
    const Unit un = decode_unit<kModePlain>(p, u);
    const int n = un.nkv;
    const int a0 = q_tile_start(un, (int)rank);
    const int row = a0 + trow;                    // sequence-relative row of this thread
    const int nominal0 = un.qb * kUnitRows + (int)rank * kBM;
    // tiles with a key visible to this CTA's rows (the lower tile of a causal
    // unit may see none of the last one: its P is then 0, no exponentials)
    const int n_mine = rank == 0 ? lower_tiles<kModePlain>(p, un) : n;
    float m_used = -INFINITY;
    float l = 0.f, l_fix = 0.f;
    for (int j = 0; j < n; ++j) {
      const uint32_t b = t & 1;  // S buffer and P barrier of global tile t
      fail |= !__all_sync(0xffffffffu, pair_wait<false>(ps, kPBarSFull + b, (t >> 1) & 1, p, 47));
      ++t;
      tc_fence_after();
      uint32_t pw[16];
      float alpha = 1.0f;
      bool rescale_warp = false;
      if (j < n_mine) {
        float s[32];
        {
          uint32_t r[32];
          tmem_ld_x32(lane_addr + 128u * b + 32u * w4, r);
          tmem_ld_wait_x32(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(r[i]);
        }
        // mask: keys visited by the previous tile (pulled-back last tile) and,
        // when causal, keys after this row; decided per CTA, applied per row
        const int jt = un.kv0 + j;
        const int b0 = kv_tile_start(un, jt);
        const int min_khi = p.causal ? a0 : un.L - 1;
        if (jt * kBN > b0 || b0 + kBN - 1 > min_khi) {
          const int khi = p.causal ? row : un.L - 1;
          const int lo = jt * kBN - b0 - 32 * w4;
          const int hi = min(khi - b0, kBN - 1) - 32 * w4;
          const bool none = hi < 0 || lo > 31 || hi < lo;
          const uint32_t vis = none ? 0u : (0xffffffffu >> (31 - min(hi, 31))) & (0xffffffffu << max(lo, 0));
#pragma unroll
          for (int i = 0; i < 32; ++i) s[i] = (vis >> i) & 1u ? s[i] : -INFINITY;
        }
        float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
        float mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
        for (int c = 8; c < 32; c += 8) {
          mx0 = max3(mx0, s[c], s[c + 1]);
          mx1 = max3(mx1, s[c + 2], s[c + 3]);
          mx2 = max3(mx2, s[c + 4], s[c + 5]);
          mx3 = max3(mx3, s[c + 6], s[c + 7]);
        }
        const float mine = fmaxf(max3(mx0, mx1, mx2), mx3);
        ps.row_max[j & 1][w4][trow] = mine;
        // (also orders the four warps' S loads before any P store)
        quad_sync(quadrant);
        const float mx = fmaxf(max3(ps.row_max[j & 1][0][trow], ps.row_max[j & 1][1][trow],
                                    ps.row_max[j & 1][2][trow]),
                               ps.row_max[j & 1][3][trow]);
        const float m_new = fmaxf(m_used, mx);
        bool resc = false;
        if (m_used == -INFINITY) {
          m_used = m_new;
        } else if ((m_new - m_used) * c2 > kRescaleLog2) {
          resc = true;
          alpha = ex2_approx((m_used - m_new) * c2);
          m_used = m_new;
        }
        rescale_warp = __any_sync(0xffffffffu, resc);
        const float neg = m_used == -INFINITY ? 0.f : -m_used * c2;
        // O's divisor carries the bf16 rounding change of the largest
        // probability of these 32 keys (same arithmetic as below)
        const float p_max = ex2_approx(fmaf(mine, c2, neg));
        const float fix = bf16_round_f32(p_max) - p_max;
        float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
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
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) pw[i] = 0u;
      }
      // O is rescaled only after P V of tile j - 1 has finished, and the wait
      // is taken only then.  Product g completes phase g / 2 of barrier
      // PVDone + g % 2: when S of tile j has arrived, product g - 2 (same
      // barrier) has finished (S of tile j was issued after it, or it
      // belongs to a unit whose last product was waited for), and product
      // g + 2 cannot start before this P is written, so the parity names the
      // phase exactly although most phases are never waited for.
      if (rescale_warp && j > 0) {
        fail |= !pv_done(pv0 + j - 1, 48);
        tc_fence_after();
      }
      if (rescale_warp) {
        uint32_t r[32];
        tmem_ld_x32(lane_addr + kPairColO + 32u * w4, r);
        tmem_ld_wait_x32(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st_x32(lane_addr + kPairColO + 32u * w4, r);
      }
      tmem_st_x16(lane_addr + 128u * b + 16u * w4, pw);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(pfull[b]);
    }
    // the next unit's Q goes to the other TMEM buffer while this unit's last
    // products run (its S products have all finished: S of this unit's tiles
    // was waited for, and the MMA thread issues in order)
    if (!fail && u + ustep < n_units) copy_q(ul + 1);
    ps.row_sum[w4][0][trow] = l;
    ps.row_sum[w4][1][trow] = l_fix;
    quad_sync(quadrant);
    float l_all = 0.f, fix_all = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      l_all += ps.row_sum[k][0][trow];
      fix_all += ps.row_sum[k][1][trow];
    }
    // (also: all four warps have read row_sum before the next unit writes it)
    if (quad_sync_check(quadrant, fail)) return;
    // the unit's last P V product (the next one waits for this unit's P)
    fail |= !__all_sync(0xffffffffu, pv_done(pv0 + n - 1, 49));
    pv0 += n;
    tc_fence_after();
    const float l_r = l_all + fix_all;
    const bool store = row >= nominal0 && row < un.L && row >= 0;
    const float inv_l = l_r > 0.f ? 1.0f / l_r : 0.f;
    {
      uint32_t r[32];
      tmem_ld_x32(lane_addr + kPairColO + 32u * w4, r);
      tmem_ld_wait_x32(r);
      if (store) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)(un.tok0 + row) * p.H + un.h) * 128 + 32 * w4);
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
    if (store && w4 == 0) {
      const float lse = l_all > 0.f ? m_used * p.scale + __log2f(l_all) * 0.69314718055994531f : -INFINITY;
      size_t idx;
      if (p.cu_seqlens)
        idx = (size_t)un.h * tokens_total + un.tok0 + row;
      else
        idx = ((size_t)un.seq * p.H + un.h) * p.N + row;
      p.lse[idx] = lse;
    }
    tc_fence_before();
  }
}

// -------------------------------------------------------------- kernel --
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ PairShared ps;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + kPairQBytes;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    mbar_init(pbar(ps, kPBarQFull), 1);
    mbar_init(pbar(ps, kPBarQEmpty), kPairSoftmaxWarps);
    mbar_init(pbar(ps, kPBarQReady), 2 * kPairSoftmaxWarps);
    for (int b = 0; b < 2; ++b) mbar_init(pbar(ps, kPBarSFull + b), 1);
    for (int g = 0; g < 2; ++g) mbar_init(pbar(ps, kPBarPFull + g), 2 * kPairSoftmaxWarps);
    for (int g = 0; g < 2; ++g) mbar_init(pbar(ps, kPBarPVDone + g), 1);
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
        pair_mma(p, ps, sRing, tmem, n_units);
        // every product has finished before either CTA frees TMEM
        mma_commit_pair(pbar(ps, kPBarDrain), kPairBoth);
      }
      if (!mbar_wait(pbar(ps, kPBarDrain), 0, 200000000ull)) ps.abort_flag = 1;
    }
  } else {
    pair_softmax(p, ps, sQ, tmem, rank, n_units);
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
