// FP8 (e4m3) attention forward with one softmax thread per query row
// (sm_103a, d = 64 or 128, dense or packed batches).
//
// The computation, the quantised operands, the unit order, the TMA producer
// and the MMA issuer are those of attn_fp8_kernel (see attn_fp8_kernel.cuh);
// the softmax differs, as in attn_fwd_row_kernel: each query tile has four
// softmax warps, one per TMEM row quadrant, and each thread owns one row and
// all 128 key columns of a tile, so the row maximum, the exponentials, the
// row sum and the epilogue of a row stay in one thread, with no exchange
// between warps ("FlashAttention 1-4 演进速查" (argus-lessons),
// FlashAttention-4 items).  P of a row, 128 e4m3 codes, is one 32-column
// TMEM store over the first columns of its S.
//
// CTA layout (384 threads, one CTA per SM, persistent): warps 0-3 softmax of
// query tile 0 of the unit, warps 4-7 of query tile 1, warp 8 TMA producer,
// warp 9 MMA issuer and TMEM owner, warps 10-11 idle; registers split 184 /
// 120 by setmaxnreg (the three warpgroups of the one-thread-per-row layout).
#pragma once

#include "attn_fp8_kernel.cuh"
#include "attn_fwd_row_kernel.cuh"

namespace attn {

constexpr int kFp8RowUnitConsumers = 1 + kRowSoftmaxWarps;  // the MMA thread and every softmax warp

template <int D>
__device__ __forceinline__ void fp8_softmax_rows(const Fp8Params& p, SharedState& ss, uint32_t tmem,
                                                 int g, uint8_t* sStage, const CUtensorMap* tm_o) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quadrant = warp % 4;
  const int trow = quadrant * 32 + lane;              // row of the tile = TMEM lane
  const uint32_t lane_addr = tmem + ((uint32_t)(quadrant * 32) << 16);
  const uint32_t colS = 128u * g;
  const uint32_t colP = 128u * g;                     // 128 e4m3 = 32 columns over S
  const uint32_t colO = fp8_col_o<D>(g);
  uint32_t scount = 0, uslot = 0;
  int units_done = 0;
  int u = -1;
  if (!fp8_next_unit(ss, p, uslot, true, u)) return;
  while (u >= 0) {
    const Fp8Unit un = fp8_unit(p, u);
    const int bh = un.b * p.H + un.h;
    const int a0 = fp8_q_start(un, g);
    const int row = a0 + trow;
    const int nominal0 = un.qb * kUnitRows + g * kBM;
    // the quantisation block of this query tile (the pulled-back last block
    // when the tile is pulled back; rows it shares with the block before it
    // are recomputed with the wrong scale here but never stored)
    const int t_last = (un.L + kBM - 1) / kBM - 1;
    const float qfac = p.logit_log2 * p.sq[(size_t)bh * p.T + min(nominal0 / kBM, t_last)];
    const int khi = p.causal ? min(row, un.L - 1) : un.L - 1;  // this row's last visible key
    const int tile_khi = p.causal ? min(a0 + kBM - 1, un.L - 1) : un.L - 1;  // any row's
    float m_used = -INFINITY;  // running max of the log2-scaled logits (moved by > 0.75 only)
    float l = 0.f;             // sum of the fp32 probabilities (of 2^8 P)
    float sk_next = p.sk[(size_t)bh * p.T];
    for (int j = 0; j < un.nkv; ++j) {
      const float sk = sk_next;
      if (j + 1 < un.nkv) sk_next = p.sk[(size_t)bh * p.T + j + 1];
      if (!__all_sync(0xffffffffu, fp8_wait(ss, kBarSFull + g, scount & 1, p, 240 + g))) return;
      ++scount;
      tc_fence_after();
      float s[kBN];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld_x32(lane_addr + colS, r0);
        tmem_ld_x32(lane_addr + colS + 32, r1);
        tmem_ld_x32(lane_addr + colS + 64, r2);
        tmem_ld_x32(lane_addr + colS + 96, r3);
        tmem_ld_wait_x32(r0);
        tmem_ld_wait_x32(r1);
        tmem_ld_wait_x32(r2);
        tmem_ld_wait_x32(r3);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(r0[c]);
          s[32 + c] = __uint_as_float(r1[c]);
          s[64 + c] = __uint_as_float(r2[c]);
          s[96 + c] = __uint_as_float(r3[c]);
        }
      }
      // keys past the sequence (K tiles are not pulled back) and, when
      // causal, after the row: this row's visible columns are 0 .. hi,
      // masked from a bit mask per 32 columns on the tiles that need it
      if (j * kBN + kBN - 1 > tile_khi || (p.causal && j * kBN + kBN - 1 > a0)) {
        const int hi = khi - j * kBN;
#pragma unroll
        for (int k = 0; k < kBN / 32; ++k) {
          const int hi_k = hi - 32 * k;
          const uint32_t vis = hi_k < 0 ? 0u : (0xffffffffu >> (31 - min(hi_k, 31)));
#pragma unroll
          for (int c = 0; c < 32; ++c) s[32 * k + c] = (vis >> c) & 1u ? s[32 * k + c] : -INFINITY;
        }
      }
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
      float mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int c = 8; c < kBN; c += 8) {
        mx0 = max3(mx0, s[c], s[c + 1]);
        mx1 = max3(mx1, s[c + 2], s[c + 3]);
        mx2 = max3(mx2, s[c + 4], s[c + 5]);
        mx3 = max3(mx3, s[c + 6], s[c + 7]);
      }
      const float raw = fmaxf(max3(mx0, mx1, mx2), mx3);
      // log2 units per raw S unit, at least the smallest normal float so that a
      // masked (-inf) logit stays -inf (a zero scale, or tiny block scales,
      // would give -inf * 0 = NaN)
      const float c2t = fmaxf(qfac * sk, FLT_MIN);
      const float m_new = fmaxf(m_used, raw == -INFINITY ? -INFINITY : raw * c2t);
      float alpha = 1.0f;
      bool resc = false;
      if (m_used == -INFINITY) {
        m_used = m_new;
      } else if (m_new - m_used > kFp8RescaleLog2) {
        resc = true;
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      const bool rescale_warp = __any_sync(0xffffffffu, resc);
      // 2^8 P = 2^(x - m + 8): the e4m3 scale of P is folded into the exponent
      const float neg = (m_used == -INFINITY ? 0.f : -m_used) + kFp8PLog2;
      float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
      uint32_t pw[32];
#pragma unroll
      for (int c = 0; c < kBN; c += 4) {
        float x0, x1, x2, x3;
        fma2(x0, x1, s[c], s[c + 1], c2t, neg);
        fma2(x2, x3, s[c + 2], s[c + 3], c2t, neg);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
        add2(sa0, sa1, p0, p1);
        add2(sb0, sb1, p2, p3);
        pw[c / 4] = e4m3x4(p0, p1, p2, p3);
      }
      l = l * alpha + ((sa0 + sa1) + (sb0 + sb1));
      // O *= alpha before this tile's P V product (the previous one has
      // finished: S of this tile was issued after it)
      if (rescale_warp) {
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
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
    // epilogue (l sums 2^8 P): O = O_acc * s_v / l -> bf16; LSE = ln 2 (m + log2 l - 8)
    int u_next = -1;
    if (!fp8_next_unit(ss, p, uslot, true, u_next)) return;
    if (!__all_sync(0xffffffffu, fp8_wait(ss, kBarOFull + g, units_done & 1, p, 242 + g))) return;
    tc_fence_after();
    const bool store = row >= nominal0 && row < un.L && row >= 0;
    const float ofac = l > 0.f ? p.sv[bh] / l : 0.f;
    // O of the warp's 32 rows through its staging tiles (64 channels each:
    // 16-byte chunk c of row r at r * 128 + 16 (c ^ (r % 8)), the 128-byte
    // swizzle of the tensor map), then one TMA store per 64 channels; where
    // the tile starts before its nominal rows (pulled back at the sequence
    // end) or before the buffer, lane l stores chunk l % 8 of rows 4 i + l / 8
    // instead, four 128-byte row pieces per instruction
    uint8_t* stage = sStage + (g * 4 + quadrant) * kFp8StageWarpBytes;
    // the previous unit's TMA stores from these tiles have read them
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int cc = 0; cc < D; cc += 32) {
      uint32_t r[32];
      tmem_ld_x32(lane_addr + colO + cc, r);
      tmem_ld_wait_x32(r);
      uint8_t* st = stage + (cc / 64) * (32 * 128);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]) * ofac, __uint_as_float(r[8 * i + 1]) * ofac);
        w.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]) * ofac, __uint_as_float(r[8 * i + 3]) * ofac);
        w.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]) * ofac, __uint_as_float(r[8 * i + 5]) * ofac);
        w.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]) * ofac, __uint_as_float(r[8 * i + 7]) * ofac);
        const int c = (cc % 64) / 8 + i;
        *reinterpret_cast<uint4*>(st + lane * 128 + ((c ^ (lane & 7)) << 4)) = w;
      }
    }
    if (a0 == nominal0 && a0 >= 0) {
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh)
          tma_store_3d(tm_o, smem_u32(stage + hh * (32 * 128)), 64 * hh, un.h,
                       un.tok0 + a0 + quadrant * 32);
        bulk_commit();
      }
    } else {
      __syncwarp();
      const int c = lane & 7;
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = 4 * i + (lane >> 3);
          const uint4 w =
              *reinterpret_cast<const uint4*>(stage + hh * (32 * 128) + rr * 128 + ((c ^ (rr & 7)) << 4));
          const int row_r = a0 + quadrant * 32 + rr;
          if (row_r >= nominal0 && row_r < un.L && row_r >= 0)
            *reinterpret_cast<uint4*>(p.o + ((size_t)(un.tok0 + row_r) * p.H + un.h) * D + 64 * hh +
                                      8 * c) = w;
        }
      }
      __syncwarp();   // every lane has read the tiles before they are written again
    }
    if (store)
      p.lse[p.cu_seqlens ? (size_t)un.h * p.cu_seqlens[p.B] + un.tok0 + row : (size_t)bh * p.N + row] =
          l > 0.f ? (m_used + (__log2f(l) - kFp8PLog2)) * 0.69314718055994531f : -INFINITY;
    tc_fence_before();
    ++units_done;
    u = u_next;
  }
  // the TMA stores of O have completed before the kernel's shared memory goes
  if (lane == 0) bulk_wait_all();
}

template <int D>
__global__ void __launch_bounds__(kRowThreads, 1)
attn_fp8_row_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_vt, const __grid_constant__ CUtensorMap tm_o,
                    const Fp8Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ SharedState ss;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + kQTiles * kFp8TileBytes;
  uint8_t* sStage = sRing + kFp8Stages * kFp8TileBytes;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // the next call on the stream may start its CTAs (and their set-up) on the
  // SMs this grid leaves; it reads nothing before this grid has completed
  if (threadIdx.x == 0) grid_dep_launch();

  if (threadIdx.x == 0) {
    mbar_init(bar_addr(ss, kBarQFull), 1);
    mbar_init(bar_addr(ss, kBarQEmpty), 1);
    for (int g = 0; g < kQTiles; ++g) {
      mbar_init(bar_addr(ss, kBarSFull + g), 1);
      mbar_init(bar_addr(ss, kBarPFull + g), 32 * kRowGroupWarps);
      mbar_init(bar_addr(ss, kBarOFull + g), 1);
    }
    mbar_init(bar_addr(ss, kBarDrain), 1);
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(bar_addr(ss, kBarUnitFull + i), 1);
      mbar_init(bar_addr(ss, kBarUnitEmpty + i), kFp8RowUnitConsumers);
    }
    for (int s = 0; s < kFp8Stages; ++s) {
      mbar_init(bar_addr(ss, kBarKV + s), 1);
      mbar_init(bar_addr(ss, kBarKV + kFp8Stages + s), 1);
    }
    ss.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kRowProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_vt);
  }
  if (warp == kRowMmaWarp) {
    tmem_alloc(smem_u32(&ss.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ss.tmem_base;
  // launched as a dependent of the V quantiser: every global access below
  // waits for that grid (and so for the whole quantisation) to complete
  grid_dep_wait();
  const int n_units = fp8_num_units(p);

  if (warp >= kRowSoftmaxWarps) {
    setmaxnreg_dec<kRowControlRegs>();
    if (warp == kRowProducerWarp) {
      if (lane == 0) fp8_producer<D>(&tm_q, &tm_k, &tm_vt, p, ss, sQ, sRing, n_units);
    } else if (warp == kRowMmaWarp) {
      if (lane == 0) {
        fp8_mma_loop<D>(p, ss, sQ, sRing, tmem);
        // every MMA issued by this thread has finished before TMEM is freed
        mma_commit(bar_addr(ss, kBarDrain));
        mbar_wait(bar_addr(ss, kBarDrain), 0, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    setmaxnreg_inc<kRowSoftmaxRegs>();
    fp8_softmax_rows<D>(p, ss, tmem, warp / kRowGroupWarps, sStage, &tm_o);
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
    tmem_dealloc(tmem, 512);
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
