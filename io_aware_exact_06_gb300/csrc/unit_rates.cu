// Per-SM unit rates of the running GPU, for the rooflines of the attention
// forward: MUFU exp2 (ex2.approx.ftz.f32) results per clock per SM, and
// tcgen05 bf16 MMA flops per clock per SM.  Standalone program; prints one
// JSON object.  Every wait is bounded.
#include <cuda_runtime.h>

#include <cstdio>
#include <vector>

#include "sm100_ptx.cuh"

using namespace attn;

namespace {

constexpr int kChains = 8;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 1024 threads per SM, kChains independent ex2 chains per thread.
__global__ void __launch_bounds__(1024, 1) ex2_rate(float* out, long long* cycles, int iters) {
  float x[kChains];
  for (int j = 0; j < kChains; ++j) x[j] = (threadIdx.x & 7) * 0.01f - 0.3f * j;
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) x[j] = fmaf(ex2(x[j]), -0.5f, 0.25f);
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
  for (int j = 0; j < kChains; ++j) s += x[j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// One thread per SM issues n back-to-back 128 x N x 16 bf16 MMAs into TMEM,
// A from shared memory (ts = 0) or from TMEM (ts = 1), B from shared memory;
// operands K-major with the 128-byte swizzle.
__global__ void __launch_bounds__(128, 1) mma_rate(long long* cycles, int n, int N, int ts,
                                                   int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid / 32;
  for (int i = tid; i < 65536 / 4; i += 128) reinterpret_cast<uint32_t*>(smem)[i] = 0;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    const uint32_t id = make_idesc_bf16(128, N, false);
    const uint64_t a = make_sdesc(smem_u32(smem), 16, 1024, kSwizzle128B);
    const uint64_t b = make_sdesc(smem_u32(smem + 16384), 16, 1024, kSwizzle128B);
    const long long t0 = clock64();
    if (ts) {
      for (int i = 0; i < n; ++i) mma_ts(tmem, tmem + 256, b, id, i > 0);  // A: columns 256..263
    } else {
      for (int i = 0; i < n; ++i) mma_ss(tmem, a, b, id, i > 0);
    }
    mma_commit(smem_u32(&bar));
    if (!mbar_wait(smem_u32(&bar), 0, 1000000000ull)) atomicOr(err, 1);
    cycles[blockIdx.x] = clock64() - t0;
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The operand forms of the attention kernels: products of 128 x N x 16
// cycling through the eight k-steps of a 128-deep tile, issued as the kernels
// issue them (eight products with compile-time descriptor offsets per loop
// step): A from shared memory (TS = 0, K-major) or from TMEM (TS = 1); B
// K-major (BMN = 0: S = Q K^T) or MN-major (BMN = 1: P V, dS K, P^T dO, dS^T
// Q).  With contend = 1, warps 4-7 load and store TMEM columns the products do
// not use, back to back, while warp 0 issues (the softmax and gradient warps'
// traffic).  N = 256: TMEM D [0, 256), A [256, 320), traffic [384, 448).
template <int TS, int BMN, int N>
__global__ void __launch_bounds__(256, 1) mma_form_rate(long long* cycles, int n, int contend,
                                                        int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid / 32;
  for (int i = tid; i < 98304 / 4; i += 256) reinterpret_cast<uint32_t*>(smem)[i] = 0;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  // B K-major: 64-column chunks of N rows (N * 128 bytes apart); MN-major: N/64
  // chunks of 128 keys (16 KB apart), 16 keys per k-step (2048 bytes)
  constexpr uint32_t kBChunk = BMN ? 16384u : (uint32_t)N * 128u;
  if (tid == 0) {
    const uint32_t id = make_idesc_bf16(128, N, BMN != 0);
    const uint64_t a0 = make_sdesc(smem_u32(smem), 16, 1024, kSwizzle128B);
    const uint64_t b0 = BMN ? make_sdesc(smem_u32(smem + 32768), 16384, 1024, kSwizzle128B)
                            : make_sdesc(smem_u32(smem + 32768), 16, 1024, kSwizzle128B);
    const long long t0 = clock64();
    for (int i = 0; i < n; i += 8) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t aoff = (uint64_t)(((kk / 4) * 16384 + (kk % 4) * 32) >> 4);
        const uint64_t boff = BMN ? (uint64_t)((kk * 2048) >> 4)
                                  : (uint64_t)(((kk / 4) * kBChunk + (kk % 4) * 32) >> 4);
        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
        if (TS)
          mma_ts(tmem, tmem + 256 + 8 * kk, b0 + boff, id, acc);
        else
          mma_ss(tmem, a0 + aoff, b0 + boff, id, acc);
      }
    }
    mma_commit(smem_u32(&bar));
    if (!mbar_wait(smem_u32(&bar), 0, 1000000000ull)) atomicOr(err, 1);
    cycles[blockIdx.x] = clock64() - t0;
  } else if (contend && warp >= 4) {
    // bounded: a fixed number of load / store pairs (longer than the products)
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp % 4)) << 16);
    uint32_t r[32];
    for (int it = 0; it < 4 * n; ++it) {
      tmem_ld_x32(lane_addr + 384, r);
      tmem_ld_wait_x32(r);
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] += 1u;
      tmem_st_x32(lane_addr + 416, r);
      tmem_st_wait();
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// A pair of SMs (a cluster of two CTAs) sharing each product: the even CTA
// issues n products of 256 x 128 x 16 (cta_group::2) stepping through the
// k-slices of a 128-deep tile as a paired attention kernel does (eight
// products with compile-time offsets per loop step).  A is each
// CTA's own 128 rows, from shared memory (TS = 0, K-major) or from TMEM
// (TS = 1); B is 64 of the 128 columns from each CTA's shared memory, K-major
// (BMN = 0: S = Q K^T with 64 keys per CTA) or MN-major (bmn = 1: P V with 64
// of the d columns per CTA; BMN = 1).  contend = 1: warps 4-7 of both CTAs load and
// store TMEM columns the products do not use.  256 TMEM columns per CTA:
// D [0, 128), A [128, 192), traffic [192, 256).
template <int TS, int BMN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    mma_pair_rate(long long* cycles, int n, int contend, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid / 32;
  const uint32_t rank = cluster_ctarank();
  for (int i = tid; i < 65536 / 4; i += 256) reinterpret_cast<uint32_t*>(smem)[i] = 0;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
    tmem_alloc_pair(smem_u32(&tmem_base), 256);
    tmem_relinquish_pair();
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    const long long t0 = clock64();
    if (rank == 0) {
      const uint32_t id = make_idesc_bf16(256, 128, BMN != 0);
      const uint64_t a0 = make_sdesc(smem_u32(smem), 16, 1024, kSwizzle128B);
      const uint64_t b0 = BMN ? make_sdesc(smem_u32(smem + 32768), 16384, 1024, kSwizzle128B)
                              : make_sdesc(smem_u32(smem + 32768), 16, 1024, kSwizzle128B);
      for (int i = 0; i < n; i += 8) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t aoff = (uint64_t)(((kk / 4) * 16384 + (kk % 4) * 32) >> 4);
          // B: 64 rows per 64-column chunk when K-major (8 KB chunks), 16 keys
          // (2048 bytes) per k-step when MN-major
          const uint64_t boff = BMN ? (uint64_t)((kk * 2048) >> 4)
                                    : (uint64_t)(((kk / 4) * 8192 + (kk % 4) * 32) >> 4);
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          if (TS)
            mma_ts_pair(tmem, tmem + 128 + 8 * kk, b0 + boff, id, acc);
          else
            mma_ss_pair(tmem, a0 + aoff, b0 + boff, id, acc);
        }
      }
      mma_commit_pair(smem_u32(&bar), 3);
    }
    // both CTAs: every product has finished writing this CTA's TMEM
    if (!mbar_wait(smem_u32(&bar), 0, 1000000000ull)) atomicOr(err, 1);
    cycles[blockIdx.x] = clock64() - t0;
  } else if (contend && warp >= 4) {
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp % 4)) << 16);
    uint32_t r[32];
    for (int it = 0; it < 2 * n; ++it) {
      tmem_ld_x32(lane_addr + 192, r);
      tmem_ld_wait_x32(r);
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] += 1u;
      tmem_st_x32(lane_addr + 224, r);
      tmem_st_wait();
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 0) tmem_dealloc_pair(tmem, 256);
}

bool check(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    printf("{\"error\": \"%s: %s\"}\n", what, cudaGetErrorString(e));
    return false;
  }
  return true;
}

}  // namespace

int main() {
  int sms = 0, clk_khz = 0, major = 0, minor = 0;
  if (!check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0), "attr")) return 1;
  cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, 0);
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, 0);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, 0);
  float* out = nullptr;
  long long* cyc = nullptr;
  int* err = nullptr;
  if (!check(cudaMalloc(&out, (size_t)sms * 1024 * sizeof(float)), "malloc")) return 1;
  if (!check(cudaMalloc(&cyc, sms * sizeof(long long)), "malloc")) return 1;
  if (!check(cudaMalloc(&err, sizeof(int)), "malloc")) return 1;
  cudaMemset(err, 0, sizeof(int));
  std::vector<long long> h(sms);

  const int iters = 4096;
  ex2_rate<<<sms, 1024>>>(out, cyc, 64);
  ex2_rate<<<sms, 1024>>>(out, cyc, iters);
  if (!check(cudaDeviceSynchronize(), "ex2_rate")) return 1;
  cudaMemcpy(h.data(), cyc, sms * sizeof(long long), cudaMemcpyDeviceToHost);
  double mean = 0;
  for (long long c : h) mean += (double)c / sms;
  const double ex2_per_clk = 1024.0 * kChains * iters / mean;

  const int n = 4096;
  // 120 KB of shared memory keeps one CTA per SM (each allocates all of TMEM)
  const size_t smem = 120 * 1024 + 1024;
  cudaFuncSetAttribute(mma_rate, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  // flops per clock per SM of 128 x N x 16 products: {N, A from TMEM}
  const int shapes[5][2] = {{256, 0}, {128, 0}, {64, 0}, {128, 1}, {64, 1}};
  double rate[5];
  for (int s = 0; s < 5; ++s) {
    mma_rate<<<sms, 128, smem>>>(cyc, 64, shapes[s][0], shapes[s][1], err);
    mma_rate<<<sms, 128, smem>>>(cyc, n, shapes[s][0], shapes[s][1], err);
    if (!check(cudaDeviceSynchronize(), "mma_rate")) return 1;
    cudaMemcpy(h.data(), cyc, sms * sizeof(long long), cudaMemcpyDeviceToHost);
    mean = 0;
    for (long long c : h) mean += (double)c / sms;
    rate[s] = 2.0 * 128 * shapes[s][0] * 16 * n / mean;
  }
  // the attention kernels' operand forms, issued unrolled
  const size_t smem_f = 96 * 1024 + 1024;
  typedef void (*FormFn)(long long*, int, int, int*);
  struct Form { FormFn fn; int N, contend; };
  const Form forms[8] = {{mma_form_rate<0, 0, 128>, 128, 0}, {mma_form_rate<1, 0, 128>, 128, 0},
                         {mma_form_rate<0, 1, 128>, 128, 0}, {mma_form_rate<1, 1, 128>, 128, 0},
                         {mma_form_rate<1, 0, 128>, 128, 1}, {mma_form_rate<1, 1, 128>, 128, 1},
                         {mma_form_rate<0, 0, 256>, 256, 0}, {mma_form_rate<1, 0, 256>, 256, 0}};
  double form_rate[8];
  for (int s = 0; s < 8; ++s) {
    cudaFuncSetAttribute(forms[s].fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_f);
    forms[s].fn<<<sms, 256, smem_f>>>(cyc, 64, forms[s].contend, err);
    forms[s].fn<<<sms, 256, smem_f>>>(cyc, n, forms[s].contend, err);
    if (!check(cudaDeviceSynchronize(), "mma_form_rate")) return 1;
    cudaMemcpy(h.data(), cyc, sms * sizeof(long long), cudaMemcpyDeviceToHost);
    mean = 0;
    for (long long c : h) mean += (double)c / sms;
    form_rate[s] = 2.0 * 128 * forms[s].N * 16 * n / mean;
  }
  // the pair of SMs: flops per clock per SM (half of a 256-row product per
  // SM), cycles of the even CTA
  typedef void (*PairFn)(long long*, int, int, int*);
  struct PForm { PairFn fn; int contend; };
  const PForm pforms[5] = {{mma_pair_rate<0, 0>, 0}, {mma_pair_rate<1, 0>, 0}, {mma_pair_rate<1, 1>, 0},
                           {mma_pair_rate<1, 0>, 1}, {mma_pair_rate<1, 1>, 1}};
  double pair_rate[5];
  const int pgrid = sms & ~1;
  for (int s = 0; s < 5; ++s) {
    cudaFuncSetAttribute(pforms[s].fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    pforms[s].fn<<<pgrid, 256, smem>>>(cyc, 64, pforms[s].contend, err);
    pforms[s].fn<<<pgrid, 256, smem>>>(cyc, n, pforms[s].contend, err);
    if (!check(cudaDeviceSynchronize(), "mma_pair_rate")) return 1;
    cudaMemcpy(h.data(), cyc, sms * sizeof(long long), cudaMemcpyDeviceToHost);
    mean = 0;
    for (int b = 0; b < pgrid; b += 2) mean += (double)h[b] / (pgrid / 2);
    pair_rate[s] = 2.0 * 256 * 128 * 16 * n / 2 / mean;
  }
  int herr = 0;
  cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost);
  printf("{\"sm_count\": %d, \"sm\": \"%d.%d\", \"max_clock_mhz\": %.0f, \"ex2_per_clk_per_sm\": %.2f, "
         "\"mma_bf16_flop_per_clk_per_sm\": %.1f, \"mma_ss_n128\": %.1f, \"mma_ss_n64\": %.1f, "
         "\"mma_ts_n128\": %.1f, \"mma_ts_n64\": %.1f, \"ksteps_ss_kmajor\": %.1f, "
         "\"ksteps_ts_kmajor\": %.1f, \"ksteps_ss_b_mnmajor\": %.1f, \"ksteps_ts_b_mnmajor\": %.1f, "
         "\"ksteps_ts_kmajor_tmem_traffic\": %.1f, \"ksteps_ts_b_mnmajor_tmem_traffic\": %.1f, "
         "\"ksteps_ss_n256\": %.1f, \"ksteps_ts_n256\": %.1f, "
         "\"pair_ksteps_ss_kmajor\": %.1f, \"pair_ksteps_ts_kmajor\": %.1f, "
         "\"pair_ksteps_ts_b_mnmajor\": %.1f, \"pair_ksteps_ts_kmajor_tmem_traffic\": %.1f, "
         "\"pair_ksteps_ts_b_mnmajor_tmem_traffic\": %.1f, "
         "\"mma_wait_error\": %d}\n",
         sms, major, minor, clk_khz / 1000.0, ex2_per_clk, rate[0], rate[1], rate[2], rate[3], rate[4],
         form_rate[0], form_rate[1], form_rate[2], form_rate[3], form_rate[4], form_rate[5],
         form_rate[6], form_rate[7],
         pair_rate[0], pair_rate[1], pair_rate[2], pair_rate[3], pair_rate[4], herr);
  return herr ? 2 : 0;
}
