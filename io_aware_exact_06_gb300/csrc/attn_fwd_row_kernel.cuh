// Fused exact softmax-attention forward for sm_103a with one softmax thread
// per query row (plain and sliding-window masks, d = 64 or 128, dense or
// packed batches).
//
// The work units and the TMA producer are those of attn_fwd_kernel (see
// there), and so, at d = 128, are the MMA issuer, the TMEM layout and the
// ping-pong of two query tiles; at d = 64 P has TMEM columns of its own and
// two threads issue the products (RowCfg, mma_s_loop, mma_pv_loop).  The
// softmax differs throughout.  Each query tile has four softmax warps, one per TMEM
// row quadrant, and each thread owns one row and all 128 key columns of the
// tile: the row maximum, the exponentials, the row sums and the O epilogue
// of a row stay in one thread, with no exchange between warps (the layout of
// the FA-4 softmax: "FlashAttention 1-4 演进速查" (argus-lessons),
// FlashAttention-4 items).  The scores of a row take 128 registers, so the
// softmax warps get 184 registers each and the control warps 120 (setmaxnreg).
//
// CTA layout (384 threads = 3 warpgroups, one CTA per SM, persistent):
//   warps 0-3   softmax group 0 (query tile 0 of the unit), warps 4-7 group
//               1: warp w reads TMEM lanes 32 (w % 4) .. (its 32 rows)
//   warp  8     TMA producer (lane 0)
//   warp  9     MMA issuer (lane 0; at d = 64 of the S products) and TMEM owner
//   warp  10    at d = 64: issuer of the P V products (lane 0); else idle
//   warp  11    idle
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn {

constexpr int kRowGroupWarps = 4;
constexpr int kRowSoftmaxWarps = kQTiles * kRowGroupWarps;
constexpr int kRowProducerWarp = kRowSoftmaxWarps;
constexpr int kRowMmaWarp = kRowSoftmaxWarps + 1;
constexpr int kRowPvWarp = kRowSoftmaxWarps + 2;
constexpr int kRowThreads = 32 * (kRowSoftmaxWarps + 4);
constexpr int kRowLaunchRegs = 168;   // 65536 / 384, rounded down to 8
constexpr int kRowSoftmaxRegs = 184;
constexpr int kRowControlRegs = 120;
static_assert(kRowThreads == 384, "three warpgroups");
static_assert(kRowSoftmaxWarps * 32 * kRowSoftmaxRegs + 128 * kRowControlRegs <= kRowThreads * kRowLaunchRegs,
              "register split exceeds the launch allotment");
// each of the SM's four register-file quarters holds two softmax warps and
// one control warp
static_assert(2 * 32 * kRowSoftmaxRegs + 32 * kRowControlRegs <= 16384, "register-file quarter");

// Shared memory of the kernel: Q tiles, the K/V ring, an O staging tile of
// 32 rows x 64 columns per softmax warp (the epilogue writes 64 columns of
// the warp's 32 rows there and stores them with one TMA store, two rounds at
// d = 128), and, at d = 64, where it fits, a second Q buffer (the next
// unit's Q tiles load while the current unit runs).
//
// At d = 64 TMEM also has room for P apart from S (S_g [128 g, +128), O_g
// [256 + 64 g, +64), P_g [384 + 64 g, +64)), so a group's next S product is
// issued as soon as its softmax has read S and runs during that softmax
// (mma_s_loop, mma_pv_loop); at d = 128 P takes the first 64 columns of S_g.
template <int D>
struct RowCfg {
  using C = FwdCfg<D>;
  static constexpr int kQBufs = D == 64 ? 2 : 1;
  static constexpr int kStageWarpBytes = 32 * 128;               // 32 rows x 64 bf16
  static constexpr int kStageGroupBytes = 4 * kStageWarpBytes;   // a query tile's 4 warps
  static constexpr bool kSPre = D == 64;
  __host__ __device__ static constexpr uint32_t col_p(int g) {
    return kSPre ? 384u + 64u * (uint32_t)g : C::col_s(g);
  }
  static constexpr int kSmemStage = kQTiles * kStageGroupBytes;
  static constexpr int kSmemBytes = kQBufs * C::kSmemQ + C::kSmemRing + kSmemStage + 1024;
};
static_assert(RowCfg<64>::kSmemBytes + 1024 <= 227 * 1024, "shared memory of the d = 64 kernel");
// Readers of each published unit index: the MMA thread(s) and every softmax warp.
template <int D>
__host__ __device__ constexpr int row_unit_consumers() {
  return (RowCfg<D>::kSPre ? 2 : 1) + kRowSoftmaxWarps;
}
static_assert(RowCfg<128>::kSmemBytes + 1024 <= 227 * 1024, "shared memory of the d = 128 kernel");

// MMA issuers of the d = 64 layout (P apart from S): two threads, so that
// neither stream of products waits behind the other's issue (an issuing
// thread returns from tcgen05.mma only as the tensor pipe takes it).
//   mma_s_loop   S_g of every tile: after the group's softmax has read its
//                previous S (SFree); K slots released here; runs on into the
//                next unit (its Q tiles in the other Q buffer).
//   mma_pv_loop  O_g += P_g V of every tile: after P_g (PFull); each product
//                signals PFree, the unit's last one OFull; V slots released here.
// Ring positions follow the producer's order, K_0, V_0, K_1, V_1, ... per unit.
template <int D, int kMode>
__device__ __forceinline__ void mma_s_loop(const FwdParams& p, SharedState& ss, uint8_t* sQ,
                                           uint8_t* sRing, uint32_t tmem) {
  using C = FwdCfg<D>;
  using R = RowCfg<D>;
  static_assert(R::kSPre && R::kQBufs == 2, "layout with P apart from S and two Q buffers");
  uint32_t sfree[2] = {0, 0};
  bool first[2] = {true, true};
  uint32_t uslot = 0, base = 0;
  for (int ux = 0;; ++ux) {
    int u;
    Unit un;
    if (!next_unit(ss, p, uslot, false, u, &un) || u < 0) return;
    // group 0 may skip the unit's last tile (lower_tiles); group 1 visits all
    const int n[2] = {lower_tiles<kMode>(p, un), un.nkv};
    const int qb = ux % R::kQBufs;
    if (!wait_bar(ss, bar_qfull(qb), (ux / R::kQBufs) & 1, p, 11)) return;
    for (int j = 0; j < un.nkv; ++j) {
      const uint32_t posK = base + 2 * j;
      if (!wait_bar(ss, kBarKV + posK % C::kStages, (posK / C::kStages) & 1, p, 10)) return;
      tc_fence_after();
      for (int g = 0; g < kQTiles; ++g) {
        if (j >= n[g]) continue;
        if (!first[g]) {
          if (!wait_bar(ss, kBarSFree + g, sfree[g] & 1, p, 18 + g)) return;
          ++sfree[g];
          tc_fence_after();
        }
        first[g] = false;
        issue_qk<D>(tmem + C::col_s(g), smem_u32(sQ + qb * C::kSmemQ + g * C::kTileBytes),
                    smem_u32(sRing + (posK % C::kStages) * C::kTileBytes));
        mma_commit(bar_addr(ss, kBarSFull + g));
      }
      mma_commit(bar_addr(ss, kBarKV + C::kStages + posK % C::kStages));
      // Q is free for a later unit's copy once the unit's last S product is done
      if (j == un.nkv - 1) mma_commit(bar_addr(ss, bar_qempty(qb)));
    }
    base += 2 * un.nkv;
  }
}

template <int D, int kMode>
__device__ __forceinline__ void mma_pv_loop(const FwdParams& p, SharedState& ss, uint8_t* sRing,
                                            uint32_t tmem) {
  using C = FwdCfg<D>;
  using R = RowCfg<D>;
  uint32_t pfull[2] = {0, 0};
  uint32_t uslot = 0, base = 0;
  for (;;) {
    int u;
    Unit un;
    if (!next_unit(ss, p, uslot, false, u, &un) || u < 0) return;
    const int n[2] = {lower_tiles<kMode>(p, un), un.nkv};
    for (int j = 0; j < un.nkv; ++j) {
      const uint32_t posV = base + 2 * j + 1;
      if (!wait_bar(ss, kBarKV + posV % C::kStages, (posV / C::kStages) & 1, p, 10)) return;
      tc_fence_after();
      for (int g = 0; g < kQTiles; ++g) {
        if (j >= n[g]) continue;
        if (!wait_bar(ss, kBarPFull + g, pfull[g] & 1, p, 12 + g)) return;
        ++pfull[g];
        tc_fence_after();
        issue_pv<D>(tmem + C::col_o(g), tmem + R::col_p(g),
                    smem_u32(sRing + (posV % C::kStages) * C::kTileBytes), j > 0);
        mma_commit(bar_addr(ss, kBarPFree + g));
        if (j == n[g] - 1) mma_commit(bar_addr(ss, kBarOFull + g));
      }
      mma_commit(bar_addr(ss, kBarKV + C::kStages + posV % C::kStages));
    }
    base += 2 * un.nkv;
  }
}

// The softmax of query tile g of every unit, one thread per row.
template <int D, int kMode>
__device__ __forceinline__ void softmax_rows(const FwdParams& p, SharedState& ss, uint32_t tmem,
                                             int g, int n_units, uint8_t* sStage,
                                             const CUtensorMap* tm_o) {
  using C = FwdCfg<D>;
  using R = RowCfg<D>;
  static_assert(kMode == kModePlain || kMode == kModeWindow, "plain and window masks");
  constexpr bool kWindow = kMode == kModeWindow;
  constexpr bool kSPre = R::kSPre;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int quadrant = warp % 4;
  const int trow = quadrant * 32 + lane;       // row within the tile = TMEM lane
  const uint32_t lane_addr = tmem + ((uint32_t)(quadrant * 32) << 16);
  const uint32_t colS = C::col_s(g);
  const uint32_t colO = C::col_o(g);
  const uint32_t colP = R::col_p(g);
  const float c2 = p.scale_log2;
  uint32_t scount = 0;
  uint32_t pfree = 0;     // P V products of this group waited for (P apart from S)
  bool first_tile = true; // no P V product of this group before this tile
  int units_done = 0;
  int tokens_total = 0;
  if (p.cu_seqlens) tokens_total = p.cu_seqlens[p.B];

  uint32_t uslot = 0;
  int u = -1;
  Unit un_cur{};
  if (!next_unit(ss, p, uslot, true, u, &un_cur)) return;
  while (u >= 0) {
    const Unit un = un_cur;
    const int a0 = q_tile_start(un, g);
    const int row = a0 + trow;                       // sequence-relative row of this thread
    const int nominal0 = un.qb * kUnitRows + g * kBM;
    const int n_tiles = g == 0 ? lower_tiles<kMode>(p, un) : un.nkv;
    float m_used = -INFINITY;
    float l = 0.f;     // sum of the fp32 probabilities: the LSE
    float l_fix = 0.f; // rounding change of each half tile's largest probability
    for (int j = 0; j < n_tiles; ++j) {
      if (!__all_sync(0xffffffffu, wait_bar(ss, kBarSFull + g, scount & 1, p, 60 + g))) return;
      ++scount;
      tc_fence_after();
      // Mask: keys already visited by the previous tile (pulled-back last
      // tile), keys after this row when causal, keys outside the sliding
      // window.  Decided per group, applied per row: this row's visible
      // columns [lo, hi] form one range, masked from a bit mask per 32
      // columns.  The decision comes before the scores are read, and each
      // side reads them and takes the row maxima in straight-line code (a
      // branch between the reads and the maxima kept the two apart: 6-7 %
      // on the d = 64 workloads)
      const int jt = un.kv0 + j;
      const int b0 = kv_tile_start(un, jt);
      const int max_klo = (kWindow && p.wl >= 0) ? max(0, a0 + kBM - 1 - p.wl) : 0;
      int min_khi = p.causal ? a0 : un.L - 1;
      if (kWindow && p.wr >= 0) min_khi = min(min_khi, a0 + p.wr);
      const bool masked = jt * kBN > b0 || b0 < max_klo || b0 + kBN - 1 > min_khi;
      float s[kBN];
      // the row maximum of each 64-key half (four 3-input max chains each)
      float mine[2];
      auto read_scores = [&]() {
#pragma unroll
        for (int k = 0; k < kBN / 32; ++k) {
          uint32_t r[32];
          tmem_ld_x32(lane_addr + colS + 32 * k, r);
          tmem_ld_wait_x32(r);
#pragma unroll
          for (int c = 0; c < 32; ++c) s[32 * k + c] = __uint_as_float(r[c]);
        }
        if constexpr (kSPre) {
          // S_g is read: the group's next S product may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_addr(ss, kBarSFree + g));
        }
      };
      auto row_maxima = [&]() {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float* sh = s + 64 * h;
          float mx0 = fmaxf(sh[0], sh[1]), mx1 = fmaxf(sh[2], sh[3]);
          float mx2 = fmaxf(sh[4], sh[5]), mx3 = fmaxf(sh[6], sh[7]);
#pragma unroll
          for (int c = 8; c < 64; c += 8) {
            mx0 = max3(mx0, sh[c], sh[c + 1]);
            mx1 = max3(mx1, sh[c + 2], sh[c + 3]);
            mx2 = max3(mx2, sh[c + 4], sh[c + 5]);
            mx3 = max3(mx3, sh[c + 6], sh[c + 7]);
          }
          mine[h] = fmaxf(max3(mx0, mx1, mx2), mx3);
        }
      };
      if (!masked) {
        read_scores();
        row_maxima();
      } else {
        read_scores();
        int klo = (kWindow && p.wl >= 0) ? max(0, row - p.wl) : 0;
        int khi = p.causal ? row : un.L - 1;
        if (kWindow && p.wr >= 0) khi = min(khi, row + p.wr);
        klo = max(klo, jt * kBN);
        const int lo = klo - b0;
        const int hi = min(khi - b0, kBN - 1);
#pragma unroll
        for (int k = 0; k < kBN / 32; ++k) {
          const int lo_k = lo - 32 * k, hi_k = hi - 32 * k;
          const bool none = hi_k < 0 || lo_k > 31 || hi_k < lo_k;
          const uint32_t vis =
              none ? 0u : (0xffffffffu >> (31 - min(hi_k, 31))) & (0xffffffffu << max(lo_k, 0));
#pragma unroll
          for (int c = 0; c < 32; ++c) s[32 * k + c] = (vis >> c) & 1u ? s[32 * k + c] : -INFINITY;
        }
        row_maxima();
      }
      const float m_new = fmaxf(m_used, fmaxf(mine[0], mine[1]));
      // O correction decision: only when the row max grew by more than 2^16
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
      // probability of each 64-key half tile (same arithmetic as below, so
      // each p_max is bit-identical to the value written to P)
      float fix = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float p_max = ex2_approx(fmaf(mine[h], c2, neg));
        fix += bf16_round_f32(p_max) - p_max;
      }
      // p = 2^(c2 s - c2 m): packed fp32x2 FMA, MUFU ex2, packed sums; P goes
      // to TMEM 32 keys at a time (bf16 pairs over the first 64 columns of
      // S_g, whose scores this thread already holds)
      // (P apart from S: all of P in registers first; its TMEM columns are
      // written once the group's previous P V product has finished)
      float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
      uint32_t pw[kBN / 32][16];
#pragma unroll
      for (int k = 0; k < kBN / 32; ++k) {
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          float x0, x1, x2, x3;
          fma2(x0, x1, s[32 * k + c], s[32 * k + c + 1], c2, neg);
          fma2(x2, x3, s[32 * k + c + 2], s[32 * k + c + 3], c2, neg);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
          add2(sa0, sa1, p0, p1);
          add2(sb0, sb1, p2, p3);
          pw[k][c / 2] = pack_bf16x2(p0, p1);
          pw[k][c / 2 + 1] = pack_bf16x2(p2, p3);
        }
        if (!kSPre) tmem_st_x16(lane_addr + colP + 16 * k, pw[k]);
      }
      if constexpr (kSPre) {
        if (!first_tile) {
          if (!__all_sync(0xffffffffu, wait_bar(ss, kBarPFree + g, pfree & 1, p, 64 + g))) return;
          ++pfree;
          tc_fence_after();
        }
#pragma unroll
        for (int k = 0; k < kBN / 32; ++k) tmem_st_x16(lane_addr + colP + 16 * k, pw[k]);
      }
      first_tile = false;
      l = l * alpha + ((sa0 + sa1) + (sb0 + sb1));
      l_fix = l_fix * alpha + fix;
      // O *= alpha before this tile's P V product (the previous one has
      // finished: S of this tile was issued after it, or, with P apart from
      // S, PFree was waited for above)
      if (rescale_warp) {
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t r[32];
          tmem_ld_x32(lane_addr + colO + cc, r);
          tmem_ld_wait_x32(r);
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
          tmem_st_x32(lane_addr + colO + cc, r);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_addr(ss, kBarPFull + g));
    }
    // Epilogue: O / l_r -> bf16 (this thread: its row, all D columns), LSE =
    // scale * m + ln(l).  Rows before the nominal tile start (recomputed) and
    // rows past the sequence are not stored.  The next unit's index is taken
    // first (the producer published it long ago).
    const int cur_seq = un.seq, cur_h = un.h, cur_tok0 = un.tok0, cur_L = un.L;
    int u_next = -1;
    if (!next_unit(ss, p, uslot, true, u_next, &un_cur)) return;
    if (!__all_sync(0xffffffffu, wait_bar(ss, kBarOFull + g, units_done & 1, p, 62 + g))) return;
    tc_fence_after();
    const float l_r = l + l_fix;
    const bool store = row >= nominal0 && row < cur_L && row >= 0;
    const float inv_l = l_r > 0.f ? 1.0f / l_r : 0.f;
    {
      // This warp's 32 rows through its staging tile, 64 columns at a time:
      // the thread writes its row's 64 columns (16-byte chunk c of row r at
      // r * 128 + 16 (c ^ (r % 8)), no bank conflicts; the 128-byte swizzle
      // of the tensor map), then one TMA store of the 32 rows x 64 columns;
      // where the tile starts before its nominal rows (pulled back at the
      // sequence end) or before the buffer, lane l stores chunk l % 8 of rows
      // 4 i + l / 8 instead, four 128-byte row pieces per instruction.
      uint8_t* stage = sStage + g * RowCfg<D>::kStageGroupBytes + quadrant * RowCfg<D>::kStageWarpBytes;
      const bool whole = a0 == nominal0 && a0 >= 0;
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh) {
        // the previous TMA store from this tile has read it
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < 64; cc += 32) {
          uint32_t r[32];
          tmem_ld_x32(lane_addr + colO + 64 * hh + cc, r);
          tmem_ld_wait_x32(r);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l);
            const int c = cc / 8 + i;
            *reinterpret_cast<uint4*>(stage + lane * 128 + ((c ^ (lane & 7)) << 4)) = w;
          }
        }
        if (whole) {
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(tm_o, smem_u32(stage), 64 * hh, cur_h, cur_tok0 + a0 + quadrant * 32);
            bulk_commit();
          }
        } else {
          __syncwarp();
          const int c = lane & 7;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3);
            const uint4 w = *reinterpret_cast<const uint4*>(stage + rr * 128 + ((c ^ (rr & 7)) << 4));
            const int row_r = a0 + quadrant * 32 + rr;
            if (row_r >= nominal0 && row_r < cur_L && row_r >= 0)
              *reinterpret_cast<uint4*>(p.o + ((size_t)(cur_tok0 + row_r) * p.H + cur_h) * D + 64 * hh +
                                        8 * c) = w;
          }
          __syncwarp();   // every lane has read the tile before it is written again
        }
      }
    }
    if (store) {
      const float lse = l > 0.f ? m_used * p.scale + __log2f(l) * 0.69314718055994531f : -INFINITY;
      size_t idx;
      if (p.cu_seqlens)
        idx = (size_t)cur_h * tokens_total + cur_tok0 + row;
      else
        idx = ((size_t)cur_seq * p.H + cur_h) * p.N + row;
      p.lse[idx] = lse;
    }
    tc_fence_before();
    ++units_done;
    u = u_next;
  }
  // the TMA stores of O have completed before the kernel's shared memory goes
  if ((threadIdx.x & 31) == 0) bulk_wait_all();
}

template <int D, int kMode>
__global__ void __launch_bounds__(kRowThreads, 1)
attn_fwd_row_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p) {
  using C = FwdCfg<D>;
  using R = RowCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ SharedState ss;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + R::kQBufs * C::kSmemQ;
  uint8_t* sStage = sRing + C::kSmemRing;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // the next call on the stream may start its CTAs (and their set-up) on the
  // SMs this grid leaves; it reads nothing before this grid has completed
  if (threadIdx.x == 0) grid_dep_launch();

  if (threadIdx.x == 0) {
    for (int b = 0; b < R::kQBufs; ++b) {
      mbar_init(bar_addr(ss, bar_qfull(b)), 1);
      mbar_init(bar_addr(ss, bar_qempty(b)), 1);
    }
    for (int g = 0; g < kQTiles; ++g) {
      mbar_init(bar_addr(ss, kBarSFull + g), 1);
      mbar_init(bar_addr(ss, kBarPFull + g), 32 * kRowGroupWarps);
      mbar_init(bar_addr(ss, kBarSFree + g), kRowGroupWarps);
      mbar_init(bar_addr(ss, kBarPFree + g), 1);
      mbar_init(bar_addr(ss, kBarOFull + g), 1);
    }
    mbar_init(bar_addr(ss, kBarDrain), 1);
    mbar_init(bar_addr(ss, kBarDrain1), 1);
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(bar_addr(ss, kBarUnitFull + i), 1);
      mbar_init(bar_addr(ss, kBarUnitEmpty + i), row_unit_consumers<D>());
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_addr(ss, kBarKV + s), 1);
      mbar_init(bar_addr(ss, kBarKV + C::kStages + s), 1);
    }
    ss.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kRowProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == kRowMmaWarp) {
    tmem_alloc(smem_u32(&ss.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ss.tmem_base;
  // every global access below waits for the grids this one depends on (the
  // previous call on the stream, when launched as its dependent)
  grid_dep_wait();
  const int n_units = num_units<kMode>(p);

  if (warp >= kRowSoftmaxWarps) {
    setmaxnreg_dec<kRowControlRegs>();
    if (warp == kRowProducerWarp) {
      if (lane == 0)
        producer_loop<D, kMode, C::kStages, R::kQBufs>(&tm_q, &tm_k, &tm_v, p, ss, sQ, sRing, n_units);
    } else if (warp == kRowMmaWarp) {
      if (lane == 0) {
        if constexpr (R::kSPre)
          mma_s_loop<D, kMode>(p, ss, sQ, sRing, tmem);
        else
          mma_loop<D, kMode, R::kQBufs>(p, ss, sQ, sRing, tmem, n_units);
        // every MMA issued by this thread has finished before TMEM is freed
        mma_commit(bar_addr(ss, kBarDrain));
        mbar_wait(bar_addr(ss, kBarDrain), 0, 100000000ull);
      }
    } else if (R::kSPre && warp == kRowPvWarp) {
      if (lane == 0) {
        mma_pv_loop<D, kMode>(p, ss, sRing, tmem);
        mma_commit(bar_addr(ss, kBarDrain1));
        mbar_wait(bar_addr(ss, kBarDrain1), 0, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    setmaxnreg_inc<kRowSoftmaxRegs>();
    softmax_rows<D, kMode>(p, ss, tmem, warp / kRowGroupWarps, n_units, sStage, &tm_o);
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
  if (warp == kRowMmaWarp) {
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

}  // namespace attn
