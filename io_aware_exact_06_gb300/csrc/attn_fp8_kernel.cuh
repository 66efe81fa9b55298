// FP8 (e4m3) fused attention forward for sm_103a, d = 64 or 128, dense or
// packed variable-length batches.  The attention kernel keeps Q and K codes
// in rows of 128 bytes (d = 64: channels 64..127 zero), so both head
// dimensions share the 128-byte-swizzled S product; the P V product has N = d.
//
// The pages name the FP8 path's two devices without formulas: block
// quantisation and incoherent processing ("flash-attention-evolution"
// (letsgetai), FlashAttention-3 section, item 3; "FlashAttention 1-4 演进速查"
// (argus-lessons), FlashAttention-3 items).  This build reads them as:
//   - incoherent processing: Q and K are multiplied along d by the same
//     orthogonal matrix diag(signs) H_d / sqrt(d) (H_d Sylvester-Hadamard), so
//     Q K^T is unchanged while outliers of single channels spread over all d;
//     the transform is applied unnormalised (fp32 butterflies) and its 1/d
//     goes into the logit scale;
//   - block quantisation: one scale per 128-row tile and head for Q and K (the
//     tiles the tensor core multiplies), one per sequence and head for V (its
//     scale then factors out of the P V sum); a block's max |x| maps to 448,
//     the largest finite e4m3 value.
// P = 2^(x - m) <= 2^0.75 is stored as e4m3 of 256 P (the normal e4m3 range
// then reaches 2^-14), the running max moving whenever it grows by more than
// 0.75 (log2 units), so 256 P <= 431 stays below 448.
//
// Kernels:
//   fp8_quant_stage1_kernel  rotation + block quantisation of Q and of K, and
//                         in the same launch the max |V| of every 128-row
//                         block of V (its fp32 bit pattern, one word a block):
//                         persistent CTAs take one (sequence, head, 128-row
//                         block) at a time, its rows arriving by TMA in a
//                         shared-memory double buffer while the block before
//                         is quantised from registers
//   fp8_quant_v_kernel    the max |V| per (sequence, head) over its blocks'
//                         maxima, then V codes, stored transposed per
//                         (sequence, head):
//                         [d][keys padded to 128] (keys contiguous), so both
//                         products of the attention kernel take K-major
//                         operands
//   attn_fp8_row_kernel   the forward pass (attn_fp8_row_kernel.cuh): the
//                         bf16 kernel's schedule and warp roles (persistent
//                         CTAs, longest-first units of two 128-row query
//                         tiles, producer / MMA / one softmax thread per query
//                         row, P in TMEM over its S), with this file's producer
//                         and MMA issuer: tcgen05.mma of kind::f8f6f4, K tiles
//                         not pulled back (keys past the sequence are masked).
// Packed batches (cu_seqlens, every length <= N) keep the dense layouts of the
// scales and of the transposed V codes, indexed by sequence with N the length
// bound: blocks and key tiles past a sequence's end are neither written nor
// read.  The quantisers run after the bf16 path's worklist kernel, which
// validates cu_seqlens; they do nothing when it found no work (an invalid
// cu_seqlens among the reasons), so no block reads outside [0, cu_seqlens[B]).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cfloat>
#include <cstdint>

#include "attn_fwd_kernel.cuh"

namespace attn {

constexpr int kFp8D = 128;  // bytes of a Q / K code row in the attention kernel (channels, padded)
constexpr int kFp8TileBytes = kBM * kFp8D;   // 128 rows x 128 e4m3 = one 128-byte swizzle span
constexpr int kFp8Stages = 8;                // K / V ring slots
// O staging: per softmax warp its 32 rows of bf16 O, one 32 x 64 tile (4 KB,
// 128-byte swizzle) per 64 channels, stored by TMA
constexpr int kFp8StageWarpBytes = 2 * 32 * 128;
constexpr int kFp8SmemStage = kQTiles * 4 * kFp8StageWarpBytes;
constexpr int kFp8SmemBytes =
    kQTiles * kFp8TileBytes + kFp8Stages * kFp8TileBytes + kFp8SmemStage + 1024;
static_assert(kFp8SmemBytes + 1024 <= 227 * 1024, "shared memory of the FP8 kernel");
constexpr float kFp8Max = 448.0f;
constexpr float kFp8PLog2 = 8.0f;            // P is stored as e4m3(2^8 P)
constexpr float kFp8RescaleLog2 = 0.75f;

// Instruction descriptor of tcgen05.mma kind::f8f6f4, e4m3 A and B, fp32 D,
// both operands K-major: [4,6) D format (1 = f32), [7,10) A format (0 =
// e4m3), [10,13) B format (0 = e4m3), [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_e4m3(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
constexpr uint32_t kIdescFp8 = make_idesc_e4m3(kBM, kBN);
// TMEM columns of the attention kernel: S_g at 128 g (P_g over its first 32
// columns), O_g at 256 + D g.
template <int D>
__host__ __device__ constexpr uint32_t fp8_col_o(int g) { return 256u + (uint32_t)D * g; }

__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct Fp8Params {
  __nv_bfloat16* o;     // [tokens, H, d]
  float* lse;           // dense [B, H, N]; packed [H, cu_seqlens[B]]
  const float* sq;      // [B*H][T]: Q block scales
  const float* sk;      // [B*H][T]: K block scales
  const float* sv;      // [B*H]: V scale
  const int* cu_seqlens;   // null: dense batch of B sequences of length N
  const int* work;         // packed: longest-first (sequence, q-block) pairs
  const int* num_entries;  // packed: number of pairs in `work`
  int* err;
  int* sched;
  int B, H, N, T;          // N: the length (packed: the length bound); T = ceil(N / 128)
  int causal;
  float logit_log2;     // scale * log2(e) / d (the transform's 1/d folded in)
  float scale;
  unsigned long long timeout_ns;
  int head_group;       // packed: heads per group of the unit order (0: one group)
};

// Sign vector of the transform, one bit per channel (1: negate).
struct Fp8Signs {
  uint32_t bits[4];
};

// ----------------------------------------------------------- quantisers --
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// The first quantisation stage: one thread per row of a 128-row block, the
// row's D channels in registers.  A block's rows arrive by TMA in a
// shared-memory buffer (64-channel chunks of [128 rows][128 bytes], 128-byte
// swizzle: row r's 16-byte unit u at (u ^ (r mod 8)) * 16, so the 32 rows a
// warp reads at once spread over all banks), the next block's rows landing
// in the other buffer meanwhile.  The last block of a sequence (tokens
// [tok0, tok0 + L)) is pulled back to end at L, so no copy leaves the
// sequence, and leaves the rows it shares with the block before it to that
// block; rows before the sequence count as zero.
template <int D>
struct QuantCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kBlockBytes = kBM * D * 2;
  static constexpr int kSmemBytes = 2 * kBlockBytes + 1024;
  // resident CTAs per SM: at d = 128 a row's 128 channels and the butterflies
  // need about 225 registers (two CTAs: no spills; three spilled 24 bytes and
  // were slower); at d = 64, three
  static constexpr int kCtasPerSm = D == 128 ? 2 : 3;
};
constexpr int kQuantThreads = kBM;  // one per row of a block

// x H_D of one row held by one thread, unnormalised, fp32: butterflies over
// strides 1, 2, 4, ..., D/2, each pair (i, i + s) with bit s of i clear
// becoming (a + b, a - b), each rounded once.
// From stride 2 on, the butterflies of channels i and i + 1 (both with bit
// s clear) run as one packed fp32x2 addition and one subtraction, each lane
// rounded once like the scalar operations.
__device__ __forceinline__ void butterfly2(float& a0, float& a1, float& b0, float& b1) {
  asm("{\n .reg .b64 a, b, s, d;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n"
      " add.rn.f32x2 s, a, b;\n sub.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, s;\n mov.b64 {%2, %3}, d;\n}"
      : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

template <int D>
__device__ __forceinline__ void fwht_row(float (&v)[D]) {
#pragma unroll
  for (int i = 0; i < D; i += 2) {
    const float a = v[i], b = v[i + 1];
    v[i] = a + b;
    v[i + 1] = a - b;
  }
#pragma unroll
  for (int s = 2; s < D; s <<= 1) {
#pragma unroll
    for (int i = 0; i < D; i += 2) {
      if (i & s) continue;
      butterfly2(v[i], v[i + 1], v[i + s], v[i + s + 1]);
    }
  }
}

// Row r of the staged block (bf16) as fp32, the sign bits of the channels
// whose sign is -1 flipped first (exact); flips: one 32-bit mask per pair of
// channels (bit 15: the even channel, bit 31: the odd one).
template <int D>
__device__ __forceinline__ void fp8_load_row(const uint8_t* stage, int r, const uint32_t* flips,
                                             float (&v)[D]) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 w = *reinterpret_cast<const uint4*>(stage + c * kBM * 128 + r * 128 + ((u ^ (r & 7)) << 4));
      const uint4 f = *reinterpret_cast<const uint4*>(flips + 32 * c + 4 * u);
      const uint32_t x[4] = {w.x ^ f.x, w.y ^ f.y, w.z ^ f.z, w.w ^ f.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[64 * c + 8 * u + 2 * q] = __uint_as_float(x[q] << 16);
        v[64 * c + 8 * u + 2 * q + 1] = __uint_as_float(x[q] & 0xffff0000u);
      }
    }
  }
}

// max over the 128 threads of the words b (every thread gets it); red: 4
// words of shared memory, free on entry.  For the bit patterns of
// non-negative floats this is the float maximum.
__device__ __forceinline__ uint32_t block_max128_bits(uint32_t b, uint32_t* red) {
  b = __reduce_max_sync(0xffffffffu, b);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = b;
  __syncthreads();
  return max(max(red[0], red[1]), max(red[2], red[3]));
}

// Tokens [tok0, tok0 + L) of sequence b; false when block t lies past its end
// or when the worklist kernel found no work (packed only).
__device__ __forceinline__ bool fp8_seq_block(const int* cu_seqlens, const int* num_entries,
                                              int b, int t, int N, int& tok0, int& L) {
  if (!cu_seqlens) {
    tok0 = b * N;
    L = N;
    return true;
  }
  if (*num_entries == 0) return false;
  tok0 = cu_seqlens[b];
  L = cu_seqlens[b + 1] - tok0;
  return t * kBM < L;
}


// One launch for the first quantisation stage over blocks block0 + i, i in
// [0, n_blocks): blocks [0, nb) quantise Q, [nb, 2 nb) quantise K, [2 nb,
// 3 nb) write the max |V| of each 128-row block of V (its fp32 bit pattern,
// amax_v[block]); nb = B * H * T, block = (b * H + h) * T + t.
// tm_q, tm_k, tm_v: [tokens][H][D] bf16, box 64 channels x 1 head x 128 rows,
// 128-byte swizzle (a map of an absent input is never used).  Codes go to
// rows of code_stride bytes (D, or 128 for the attention kernel's padded
// rows).  Persistent CTAs of 128 threads, QuantCfg<D>::kCtasPerSm per SM.
template <int D>
__global__ void __launch_bounds__(kQuantThreads, QuantCfg<D>::kCtasPerSm)
fp8_quant_stage1_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, uint8_t* q8, uint8_t* k8,
                        float* sq, float* sk, unsigned int* amax_v, int B, int H, int N, int T,
                        Fp8Signs signs, int rotate, int block0, int n_blocks,
                        const int* cu_seqlens, const int* num_entries, int* err, int code_stride) {
  using QC = QuantCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t full[2];
  __shared__ __align__(16) uint32_t flips[D / 2];
  __shared__ uint32_t red[2][kQuantThreads / 32];
  const int nb = B * H * T;
  const int r = threadIdx.x;  // the row of the block this thread takes
  // launched as a programmatic dependent of the stream's previous kernel:
  // nothing global is touched before that grid has completed; the V
  // quantiser, this grid's dependent, may take the SM resources left free
  // meanwhile (it waits in turn for this grid's completion)
  grid_dep_wait();
  if (r == 0) grid_dep_launch();
  // block i of this launch: segment, index within it, head, sequence tokens, first staged row
  auto locate = [&](int i, int& seg, int& idx, int& h, int& tok0, int& t, int& r0) {
    const int gidx = i + block0;
    seg = gidx / nb;
    idx = gidx - seg * nb;
    t = idx % T;
    const int bh = idx / T;
    const int b = bh / H;
    h = bh - b * H;
    int L;
    if (!fp8_seq_block(cu_seqlens, num_entries, b, t, N, tok0, L)) return false;
    r0 = min(t * kBM, L - kBM);
    return true;
  };
  auto issue = [&](int i, int buf) {  // one thread
    int seg, idx, h, tok0, t, r0;
    if (i >= n_blocks || !locate(i, seg, idx, h, tok0, t, r0)) return;
    const CUtensorMap* tm = seg == 0 ? &tm_q : (seg == 1 ? &tm_k : &tm_v);
    const uint32_t bar = smem_u32(&full[buf]);
    mbar_arrive_expect_tx(bar, QC::kBlockBytes);
#pragma unroll
    for (int c = 0; c < QC::kChunks; ++c)
      tma_load_3d(smem_u32(stage + buf * QC::kBlockBytes + c * kBM * 128), tm, bar, 64 * c, h, tok0 + r0);
  };
  // sign masks of the channel pairs (negation is exact)
  if (threadIdx.x < D / 2) {
    const int c0 = 2 * threadIdx.x;
    uint32_t f = 0u;
    if (rotate) {
      if ((signs.bits[c0 / 32] >> (c0 % 32)) & 1u) f |= 0x8000u;
      if ((signs.bits[(c0 + 1) / 32] >> ((c0 + 1) % 32)) & 1u) f |= 0x80000000u;
    }
    flips[threadIdx.x] = f;
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&full[0]), 1);
    mbar_init(smem_u32(&full[1]), 1);
    fence_mbar_init();
    issue(blockIdx.x, 0);
    issue(blockIdx.x + gridDim.x, 1);
  }
  __syncthreads();
  uint32_t used0 = 0u, used1 = 0u;  // copies consumed per buffer
  int k = 0;
  bool failed = false;
  for (int i = blockIdx.x; i < n_blocks; i += gridDim.x, ++k) {
    const int buf = k & 1;
    int seg, idx, h, tok0, t, r0;
    const bool valid = locate(i, seg, idx, h, tok0, t, r0);  // the same in every thread
    float v[D];
    float m = 0.f;  // max |x| of this thread's row: never NaN (max.f32 drops NaN inputs)
    bool ok = true;
    if (valid) {
      ok = mbar_wait(smem_u32(&full[buf]), (buf ? used1 : used0) & 1, 2000000000ull);
      if (buf)
        ++used1;
      else
        ++used0;
    }
    if (valid && ok) {
      const uint8_t* st = stage + buf * QC::kBlockBytes;
      if (seg < 2) {
        if (r0 + r >= 0) {
          fp8_load_row<D>(st, r, flips, v);
          if (rotate) fwht_row<D>(v);
        } else {
#pragma unroll
          for (int c = 0; c < D; ++c) v[c] = 0.f;
        }
#pragma unroll
        for (int c = 0; c < D; c += 2) m = max3(m, fabsf(v[c]), fabsf(v[c + 1]));
      } else if (r0 + r >= t * kBM) {  // V: the rows of this block only
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 w = *reinterpret_cast<const uint4*>(st + c * kBM * 128 + r * 128 + ((u ^ (r & 7)) << 4));
            const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
              m = max3(m, fabsf(__uint_as_float(x[q] << 16)), fabsf(__uint_as_float(x[q] & 0xffff0000u)));
          }
        }
      }
    }
    // every read of this buffer is done once all threads have the block max;
    // a thread whose copy wait gave up contributes all-ones, above the bits
    // of every non-negative float, so that all threads leave together
    const uint32_t mbits = block_max128_bits(ok ? __float_as_uint(m) : 0xffffffffu, red[k & 1]);
    if (mbits == 0xffffffffu) {
      failed = true;
      break;
    }
    const float amax = __uint_as_float(mbits);
    if (threadIdx.x == 0) {
      // (the generic-proxy reads above before the copy that overwrites them)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(i + 2 * gridDim.x, buf);
    }
    if (!valid) continue;
    if (seg < 2) {
      uint8_t* codes = seg == 0 ? q8 : k8;
      float* scale_out = (seg == 0 ? sq : sk) + idx;
      const float inv = amax > 0.f ? __fdiv_rn(kFp8Max, amax) : 1.0f;
      if (threadIdx.x == 0) *scale_out = amax > 0.f ? __fdiv_rn(amax, kFp8Max) : 1.0f;
      const int row = r0 + r;
      if (row >= t * kBM) {  // (rows before it are the previous block's)
        uint4* dst = reinterpret_cast<uint4*>(codes + ((size_t)(tok0 + row) * H + h) * code_stride);
#pragma unroll
        for (int q = 0; q < D / 16; ++q) {
          uint4 w;
          w.x = e4m3x4(__fmul_rn(v[16 * q + 0], inv), __fmul_rn(v[16 * q + 1], inv),
                       __fmul_rn(v[16 * q + 2], inv), __fmul_rn(v[16 * q + 3], inv));
          w.y = e4m3x4(__fmul_rn(v[16 * q + 4], inv), __fmul_rn(v[16 * q + 5], inv),
                       __fmul_rn(v[16 * q + 6], inv), __fmul_rn(v[16 * q + 7], inv));
          w.z = e4m3x4(__fmul_rn(v[16 * q + 8], inv), __fmul_rn(v[16 * q + 9], inv),
                       __fmul_rn(v[16 * q + 10], inv), __fmul_rn(v[16 * q + 11], inv));
          w.w = e4m3x4(__fmul_rn(v[16 * q + 12], inv), __fmul_rn(v[16 * q + 13], inv),
                       __fmul_rn(v[16 * q + 14], inv), __fmul_rn(v[16 * q + 15], inv));
          dst[q] = w;
        }
        for (int q = D / 16; q < code_stride / 16; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
      }
    } else if (threadIdx.x == 0) {
      amax_v[idx] = __float_as_uint(amax);
    }
  }
  if (failed) {
    if (threadIdx.x == 0) atomicOr(err, kErrTimeout);
    // a copy issued for a later block may still be landing
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
}

// V codes, transposed: vt[(b*H + h) * 128 + c][key] for keys padded to Np
// (a multiple of 128; padding keys of the sequence's last tile get code 0,
// tiles past its end are not written).  The scale is max |V| over the
// sequence's blocks (amax_bits[(b*H + h) * T + t], the first stage's block
// maxima); the first tile's CTA writes it to sv.
// One CTA per (sequence, head, 128 keys); warp w takes keys 16 w .. 16 w + 15
// and lane l channels 4 l .. 4 l + 3 (one 8-byte load per key, a warp reading
// whole rows), so a thread holds a 16-key x 4-channel block of codes: four
// 4 x 4 byte transposes (byte permutes) turn it into 16 keys of each of its
// channels, one 16-byte store per channel.
template <int D>
__global__ void __launch_bounds__(256)
fp8_quant_v_kernel(const __nv_bfloat16* v, const unsigned int* amax_bits, float* sv, uint8_t* vt,
                   int B, int H, int N, int Np, const int* cu_seqlens, const int* num_entries) {
  static_assert(kBN == 8 * 16, "8 warps of 16 keys");
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // launched as a dependent of the first stage: nothing global is read before
  // that grid (the maxima of |V|) has completed; the attention kernel, this
  // grid's dependent, waits in turn for this one
  grid_dep_wait();
  if (threadIdx.x == 0) grid_dep_launch();
  const int T = Np / kBN;
  const int t = blockIdx.x % T;
  const int bh = blockIdx.x / T;
  const int b = bh / H, h = bh % H;
  int tok0, L;
  if (!fp8_seq_block(cu_seqlens, num_entries, b, t, N, tok0, L)) return;  // uniform in the CTA
  // this thread's 16 keys, all loads in flight together (issued before the
  // scale is known: they overlap its reduction)
  const bool active = lane < D / 4;
  const int key0 = t * kBN + 16 * warp;
  uint2 raw[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    raw[i] = active && key0 + i < L
                 ? *reinterpret_cast<const uint2*>(v + ((size_t)(tok0 + key0 + i) * H + h) * D + 4 * lane)
                 : make_uint2(0u, 0u);
  // max |V| of the sequence, by every warp on its own (a few words, in L2;
  // no block barrier): the bit patterns of non-negative floats order as the
  // floats do
  unsigned int mb = 0u;
  const int nblk = (L + kBM - 1) / kBM;
  for (int i = lane; i < nblk; i += 32) mb = max(mb, amax_bits[(size_t)bh * T + i]);
  mb = __reduce_max_sync(0xffffffffu, mb);
  const float amax = __uint_as_float(mb);
  const float inv = amax > 0.f ? __fdiv_rn(kFp8Max, amax) : 1.0f;
  if (t == 0 && threadIdx.x == 0) sv[bh] = amax > 0.f ? __fdiv_rn(amax, kFp8Max) : 1.0f;
  if (!active) return;
  // codes of key i, channels 4 l + j in byte j
  uint32_t cw[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float f0 = __uint_as_float(raw[i].x << 16), f1 = __uint_as_float(raw[i].x & 0xffff0000u);
    const float f2 = __uint_as_float(raw[i].y << 16), f3 = __uint_as_float(raw[i].y & 0xffff0000u);
    cw[i] = e4m3x4(__fmul_rn(f0, inv), __fmul_rn(f1, inv), __fmul_rn(f2, inv), __fmul_rn(f3, inv));
  }
  // out[j][m]: channel 4 l + j, keys 4 m .. 4 m + 3 (key 4 m + i in byte i)
  uint32_t out[4][4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t a0 = cw[4 * m], a1 = cw[4 * m + 1], a2 = cw[4 * m + 2], a3 = cw[4 * m + 3];
    const uint32_t lo01 = __byte_perm(a0, a1, 0x5140), lo23 = __byte_perm(a2, a3, 0x5140);
    const uint32_t hi01 = __byte_perm(a0, a1, 0x7362), hi23 = __byte_perm(a2, a3, 0x7362);
    out[0][m] = __byte_perm(lo01, lo23, 0x5410);
    out[1][m] = __byte_perm(lo01, lo23, 0x7632);
    out[2][m] = __byte_perm(hi01, hi23, 0x5410);
    out[3][m] = __byte_perm(hi01, hi23, 0x7632);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(vt + ((size_t)bh * D + 4 * lane + j) * Np + key0) =
        make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]);
}

// ------------------------------------------------------------ attention --
// S = Q K^T over 4 k-steps of 32 e4m3: both operands K-major, 128-byte
// swizzle, one 128-byte span per row; a k-step advances the start by 32 bytes.
__device__ __forceinline__ void issue_qk_fp8(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  const uint64_t a0 = make_sdesc(q_smem, 16, 1024, kSwizzle128B);
  const uint64_t b0 = make_sdesc(k_smem, 16, 1024, kSwizzle128B);
#pragma unroll
  for (int kk = 0; kk < kFp8D / 32; ++kk)
    mma_f8_ss(d_tmem, a0 + (uint64_t)(kk * 2), b0 + (uint64_t)(kk * 2), kIdescFp8, kk > 0 ? 1u : 0u);
}

// O (+)= P V over 4 k-steps of 32 keys: P (e4m3, four per TMEM column, keys
// 32 kk.. in columns 8 kk..) and V^T (D channels x 128 keys, K-major).
template <int D>
__device__ __forceinline__ void issue_pv_fp8(uint32_t d_tmem, uint32_t p_tmem, uint32_t vt_smem,
                                             bool accumulate) {
  constexpr uint32_t kIdescPV = make_idesc_e4m3(kBM, D);
  const uint64_t b0 = make_sdesc(vt_smem, 16, 1024, kSwizzle128B);
  const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
  for (int kk = 0; kk < kBN / 32; ++kk)
    mma_f8_ts(d_tmem, p_tmem + 8 * kk, b0 + (uint64_t)(kk * 2), kIdescPV, kk > 0 ? 1u : acc0);
}

__device__ __forceinline__ bool fp8_wait(SharedState& ss, int bar, uint32_t parity,
                                         const Fp8Params& p, int where) {
  const uint32_t a = bar_addr(ss, bar);
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

// Unit u: rows [256 qb, +256) of head h of sequence b (tokens [tok0, tok0 +
// L)); KV tiles [0, nkv).  Dense: q-blocks in decreasing cost, then batch,
// then head; packed: the worklist kernel's longest-first pairs, then head.
struct Fp8Unit {
  int b, h, qb, nkv, tok0, L;
};

__device__ __forceinline__ int fp8_num_units(const Fp8Params& p) {
  if (p.cu_seqlens) return *p.num_entries * p.H;
  return p.B * p.H * ((p.N + kUnitRows - 1) / kUnitRows);
}

__device__ __forceinline__ Fp8Unit fp8_unit(const Fp8Params& p, int u) {
  Fp8Unit un;
  int e = u / p.H;
  un.h = u - e * p.H;
  if (p.cu_seqlens && p.head_group > 0 && p.head_group < p.H) {
    // heads in groups of p.head_group, one group after the other; within a
    // group the sorted list, then head (their codes stay in L2 meanwhile)
    const int E = *p.num_entries;
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
    un.h = gi * G + (r - e * ng);
  }
  if (p.cu_seqlens) {
    un.b = p.work[2 * e];
    un.qb = p.work[2 * e + 1];
    un.tok0 = p.cu_seqlens[un.b];
    un.L = p.cu_seqlens[un.b + 1] - un.tok0;
  } else {
    const int nqb = (p.N + kUnitRows - 1) / kUnitRows;
    const int rank = e / p.B;
    un.b = e - rank * p.B;
    un.qb = nqb - 1 - rank;
    un.tok0 = un.b * p.N;
    un.L = p.N;
  }
  const int r_hi = min(un.qb * kUnitRows + kUnitRows, un.L) - 1;
  un.nkv = (p.causal ? r_hi : un.L - 1) / kBN + 1;
  return un;
}

// First row (sequence-relative) loaded for query tile g, pulled back so the
// tile ends at the sequence end at the latest.
__device__ __forceinline__ int fp8_q_start(const Fp8Unit& un, int g) {
  return min(un.qb * kUnitRows + g * kBM, un.L - kBM);
}

template <int D>
__device__ __forceinline__ void fp8_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                             const CUtensorMap* tm_vt, const Fp8Params& p,
                                             SharedState& ss, uint8_t* sQ, uint8_t* sRing,
                                             int n_units) {
  uint32_t ring = 0, uslot = 0;
  int units_done = 0;
  int u = blockIdx.x;
  for (;;) {
    if (u >= n_units) u = -1;
    {
      const int slot = uslot % kUnitSlots;
      const uint32_t n = uslot / kUnitSlots;
      if (n > 0 && !fp8_wait(ss, kBarUnitEmpty + slot, (n - 1) & 1, p, 203)) return;
      ss.unit_ring[slot] = u;
      mbar_arrive(bar_addr(ss, kBarUnitFull + slot));
      ++uslot;
    }
    if (u < 0) return;
    const int next_u = (int)gridDim.x + atomicAdd(p.sched, 1);
    const Fp8Unit un = fp8_unit(p, u);
    if (units_done > 0 && !fp8_wait(ss, kBarQEmpty, (units_done - 1) & 1, p, 201)) return;
    mbar_arrive_expect_tx(bar_addr(ss, kBarQFull), kQTiles * kFp8TileBytes);
    for (int g = 0; g < kQTiles; ++g)
      tma_load_3d(smem_u32(sQ + g * kFp8TileBytes), tm_q, bar_addr(ss, kBarQFull), 0, un.h,
                  un.tok0 + fp8_q_start(un, g));
    for (int j = 0; j < un.nkv; ++j) {
      for (int kind = 0; kind < 2; ++kind) {
        const int slot = ring % kFp8Stages;
        const uint32_t n = ring / kFp8Stages;
        if (n > 0 && !fp8_wait(ss, kBarKV + kFp8Stages + slot, (n - 1) & 1, p, 202)) return;
        const uint32_t full = bar_addr(ss, kBarKV + slot);
        // K: 128 keys x 128 code bytes; V^T: D channels x 128 keys
        mbar_arrive_expect_tx(full, kind == 0 ? kFp8TileBytes : D * kBN);
        const uint32_t dst = smem_u32(sRing + slot * kFp8TileBytes);
        if (kind == 0)
          tma_load_3d(dst, tm_k, full, 0, un.h, un.tok0 + j * kBN);
        else
          tma_load_3d(dst, tm_vt, full, j * kBN, 0, un.b * p.H + un.h);
        ++ring;
      }
    }
    ++units_done;
    u = next_u;
  }
}

__device__ __forceinline__ bool fp8_next_unit(SharedState& ss, const Fp8Params& p,
                                              uint32_t& uslot, bool whole_warp, int& u) {
  const int slot = uslot % kUnitSlots;
  bool ok = fp8_wait(ss, kBarUnitFull + slot, (uslot / kUnitSlots) & 1, p, 230);
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

template <int D>
__device__ __forceinline__ void fp8_mma_loop(const Fp8Params& p, SharedState& ss, uint8_t* sQ,
                                             uint8_t* sRing, uint32_t tmem) {
  uint32_t ring = 0;
  uint32_t pcount[2] = {0, 0};
  int units_done = 0;
  const uint32_t q_smem[2] = {smem_u32(sQ), smem_u32(sQ + kFp8TileBytes)};
  auto slot_smem = [&](uint32_t pos) { return smem_u32(sRing + (pos % kFp8Stages) * kFp8TileBytes); };
  auto wait_full = [&](uint32_t pos) {
    return fp8_wait(ss, kBarKV + pos % kFp8Stages, (pos / kFp8Stages) & 1, p, 210);
  };
  auto release = [&](uint32_t pos) { mma_commit(bar_addr(ss, kBarKV + kFp8Stages + pos % kFp8Stages)); };
  // TMEM: S_g at 128 g (P_g over its first 32 columns), O_g at 256 + D g
  uint32_t uslot = 0;
  for (;;) {
    int u;
    if (!fp8_next_unit(ss, p, uslot, false, u) || u < 0) return;
    const Fp8Unit un = fp8_unit(p, u);
    if (!fp8_wait(ss, kBarQFull, units_done & 1, p, 211)) return;
    tc_fence_after();
    uint32_t posK = ring, posV = ring + 1;
    ring += 2;
    if (!wait_full(posK)) return;
    tc_fence_after();
    for (int g = 0; g < kQTiles; ++g) {
      issue_qk_fp8(tmem + 128u * g, q_smem[g], slot_smem(posK));
      mma_commit(bar_addr(ss, kBarSFull + g));
    }
    release(posK);
    if (un.nkv == 1) mma_commit(bar_addr(ss, kBarQEmpty));
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
      for (int g = 0; g < kQTiles; ++g) {
        if (!fp8_wait(ss, kBarPFull + g, pcount[g] & 1, p, 212 + g)) return;
        ++pcount[g];
        tc_fence_after();
        issue_pv_fp8<D>(tmem + fp8_col_o<D>(g), tmem + 128u * g, slot_smem(posV), j > 1);
        if (g == kQTiles - 1) release(posV);
        if (more) {
          issue_qk_fp8(tmem + 128u * g, q_smem[g], slot_smem(nextK));
          mma_commit(bar_addr(ss, kBarSFull + g));
        } else {
          mma_commit(bar_addr(ss, kBarOFull + g));
        }
      }
      if (more) {
        release(nextK);
        if (j == un.nkv - 1) mma_commit(bar_addr(ss, kBarQEmpty));
        posV = nextV;
      }
    }
    ++units_done;
  }
}

}  // namespace attn
