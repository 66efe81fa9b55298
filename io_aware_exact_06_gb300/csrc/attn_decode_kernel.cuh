// Split-KV attention forward for one query row against a long key sequence
// (decoding one token), on CUDA cores.
//
// With one query row the work is a matrix-vector product per (sequence,
// head): 4 d flops for every 4 d bytes of K and V, one flop per byte, so HBM
// bounds it; a tensor-core tile of 128 query rows would compute 127 rows of
// padding.  The key sequence is cut into ranges processed by separate work
// items, and their partial results are merged by attn_combine_kernel with the
// two-segment merge identity ("flash-attention-evolution" (letsgetai),
// FlashAttention "核心机制"); the ranges themselves are the FlashDecoding split
// of "FlashAttention" (compassingai), section 5.  (With two or more query
// rows the per-key arithmetic grows with the rows and the tensor-core split
// kernel is faster: measured 1754 GB/s here at four rows against about 4600.)
//
// Layout of a work item (sequence b, head h, key range s = keys [s*chunk,
// min(Nk, (s+1)*chunk))): 8 warps; a key row of d bf16 is read by d/8 lanes,
// 16 bytes each (one coalesced 16-byte load per lane), so a warp covers
// 32/(d/8) keys per step; warp w takes steps w, w + 8, ... in groups of four
// steps, the loads of the next group issued before the current one is used
// (two groups of K and V rows in registers), and keeps, per key of its step,
// its own running max m, sum l and d/8-wide slice of the output sum.  At the
// end the key groups of a warp merge through shuffles and the warps through
// shared memory, and the item writes O_s = f / l (fp32) and LSE_s = scale m +
// ln l.
//
// The running max moves only when a score exceeds it by more than 2^8 in
// log2 units (the probabilities against a stale max stay below 2^8, far
// inside fp32), as in the forward kernel.  Probabilities stay in fp32.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "attn_fwd_kernel.cuh"

namespace attn {
namespace decode {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kUnroll = 4;           // steps per group of loads
constexpr float kLazyLog2 = 8.0f;

__device__ __forceinline__ float dex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint4 ld_stream(const __nv_bfloat16* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void widen(const uint4& w, float (&f)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
}

// (m, l, o) of one key group merged with another's: the result refers to the
// larger max; a group that saw no key has m = -inf and weight 0.
__device__ __forceinline__ void merge(float& m, float& l, float (&o)[8], float m2, float l2,
                                      const float (&o2)[8], float c) {
  const float mm = fmaxf(m, m2);
  const float w1 = m == -INFINITY ? 0.f : dex2((m - mm) * c);
  const float w2 = m2 == -INFINITY ? 0.f : dex2((m2 - mm) * c);
  l = l * w1 + l2 * w2;
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = o[i] * w1 + o2[i] * w2;
  m = mm;
}

// q: [B, 1, H, D] bf16.  Dense keys (cu_k null): k, v [B, Nk, H, D], key
// range s of every sequence = keys [s*chunk, min(Nk, (s+1)*chunk)).  Packed
// keys: k, v [cu_k[B], H, D], sequence b's keys at tokens cu_k[b] ..
// cu_k[b+1]-1, cut into S ranges of ceil(L_b / S) keys; *valid (written by
// decode_check_kernel) is 0 when cu_k is invalid, and then nothing is read or
// written.  o_part [S][B][H][D] fp32, lse_part [S][B][H].  Items (b, h, s),
// b-major; persistent CTAs stride over them.  c = scale * log2(e) (at least
// the smallest normal float).  The one query is the newest position of its
// sequence, so causal attention sees every key: there is no mask.
template <int D>
__global__ void __launch_bounds__(kThreads)
attn_decode_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                   const __nv_bfloat16* __restrict__ v, float* __restrict__ o_part,
                   float* __restrict__ lse_part, int B, int H, int Nk, int S, int chunk,
                   float scale, float c, const int* __restrict__ cu_k,
                   const int* __restrict__ valid) {
  constexpr int kLpk = D / 8;        // lanes per key row
  constexpr int kKps = 32 / kLpk;    // keys per warp step
  constexpr int kStride = kWarps * kKps;
  constexpr int kGroup = kStride * kUnroll;  // keys between a warp's groups
  __shared__ float sm_m[kWarps];
  __shared__ float sm_l[kWarps];
  __shared__ __align__(16) float sm_o[kWarps][D];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int grp = lane / kLpk;       // key of the step
  const int slice = lane % kLpk;     // elements 8*slice .. 8*slice+7 of the row
  const size_t row_stride = (size_t)H * D;
  const int n_items = B * H * S;
  if (cu_k && *valid == 0) return;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int s = item % S;
    const int bh = item / S;
    const int b = bh / H, h = bh % H;
    int kbase = b * Nk, Lk = Nk, ch = chunk;  // first key token, keys, keys per range
    if (cu_k) {
      kbase = cu_k[b];
      Lk = cu_k[b + 1] - kbase;
      ch = (Lk + S - 1) / S;
    }
    const int k_lo = s * ch;
    const int k_hi = min(Lk, k_lo + ch);
    float qf[8];
    widen(*reinterpret_cast<const uint4*>(q + (size_t)b * row_stride + (size_t)h * D + 8 * slice),
          qf);
    float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    const __nv_bfloat16* kb = k + (size_t)kbase * row_stride + (size_t)h * D + 8 * slice;
    const __nv_bfloat16* vb = v + (size_t)kbase * row_stride + (size_t)h * D + 8 * slice;
    // keys past the range read the range's last key (in bounds) and are skipped
    auto load_group = [&](int base, uint4 (&kw)[kUnroll], uint4 (&vw)[kUnroll]) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int key = min(base + u * kStride + grp, k_hi - 1);
        kw[u] = ld_stream(kb + (size_t)key * row_stride);
        vw[u] = ld_stream(vb + (size_t)key * row_stride);
      }
    };
    auto use_group = [&](int base, const uint4 (&kw)[kUnroll], const uint4 (&vw)[kUnroll]) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        float kf[8], vf[8];
        widen(kw[u], kf);
        widen(vw[u], vf);
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) dot = fmaf(qf[i], kf[i], dot);
#pragma unroll
        for (int off = 1; off < kLpk; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        if (base + u * kStride + grp < k_hi) {
          if (m == -INFINITY) {
            m = dot;
          } else if ((dot - m) * c > kLazyLog2) {
            const float alpha = dex2((m - dot) * c);
            l *= alpha;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] *= alpha;
            m = dot;
          }
          const float p = dex2((dot - m) * c);
          l += p;
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vf[i], acc[i]);
        }
      }
    };
    uint4 ka[kUnroll], va[kUnroll], kn[kUnroll], vn[kUnroll];
    int base = k_lo + warp * kKps;
    if (base < k_hi) load_group(base, ka, va);
    while (base < k_hi) {
      const int b1 = base + kGroup;
      if (b1 < k_hi) load_group(b1, kn, vn);
      use_group(base, ka, va);
      if (b1 >= k_hi) break;
      const int b2 = b1 + kGroup;
      if (b2 < k_hi) load_group(b2, ka, va);
      use_group(b1, kn, vn);
      base = b2;
    }
    // merge the key groups of the warp (lanes kLpk, 2 kLpk, ... apart)
#pragma unroll
    for (int off = kLpk; off < 32; off <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
      const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
      float o2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o2[i] = __shfl_xor_sync(0xffffffffu, acc[i], off);
      merge(m, l, acc, m2, l2, o2, c);
    }
    if (lane == 0) {
      sm_m[warp] = m;
      sm_l[warp] = l;
    }
    if (grp == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) sm_o[warp][8 * slice + i] = acc[i];
    }
    __syncthreads();
    // merge the warps: thread t handles column t
    for (int col = threadIdx.x; col < D; col += kThreads) {
      float mm = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, sm_m[w]);
      float lsum = 0.f, osum = 0.f;
      if (mm != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float mw = sm_m[w];
          const float wt = mw == -INFINITY ? 0.f : dex2((mw - mm) * c);
          lsum = fmaf(sm_l[w], wt, lsum);
          osum = fmaf(sm_o[w][col], wt, osum);
        }
      }
      const size_t orow = ((size_t)s * B + b) * H + h;
      o_part[orow * D + col] = lsum > 0.f ? osum / lsum : 0.f;
      if (col == 0)
        lse_part[orow] = lsum > 0.f ? mm * scale + __log2f(lsum) * 0.69314718055994531f : -INFINITY;
    }
    __syncthreads();  // shared memory is reused by the next item
  }
}

// Packed keys: cu_k must start at 0 and hold B lengths in [0, max_len]; then
// every key a decode item reads lies in [0, cu_k[B]).  *valid = 1 if so, else
// 0 with kErrSeqlens in the error word.  One CTA.
__global__ void __launch_bounds__(256)
decode_check_kernel(const int* cu_k, int B, int max_len, int* valid, int* err) {
  __shared__ int bad;
  if (threadIdx.x == 0) bad = cu_k[0] != 0;
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int L = cu_k[b + 1] - cu_k[b];
    if (L < 0 || L > max_len) bad = 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    *valid = bad ? 0 : 1;
    if (bad) atomicOr(err, kErrSeqlens);
  }
}

}  // namespace decode
}  // namespace attn
