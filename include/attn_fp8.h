/*
 * C ABI of the GB300 (sm_103a) FP8 attention forward (e4m3, d = 64 or 128).
 *
 * The FP8 path of the pages ("flash-attention-evolution" (letsgetai),
 * FlashAttention-3 section, item 3; "FlashAttention 1-4 演进速查"
 * (argus-lessons), FlashAttention-3 items) quantises the operands to 8-bit
 * floats and controls the error with block quantisation and incoherent
 * processing.  Read here as:
 *   - incoherent processing: Q and K are multiplied along d by the same
 *     orthogonal matrix diag(signs) H_d / sqrt(d) (H_d Sylvester-Hadamard,
 *     signs a caller-supplied +-1 vector), which leaves Q K^T unchanged;
 *   - block quantisation: e4m3 codes (round to nearest even, saturating at
 *     448), one fp32 scale per block: per 128-row tile and head for Q and K,
 *     per sequence and head for V; a block's max |x| maps to 448.
 * P is quantised as e4m3(256 P) before the P V product; fp32 accumulation.
 * This is an approximation of the exact attention of attn_fwd.h.
 *
 * Layouts as in attn_fwd.h.  Dense (cu_seqlens == NULL): q, k, v, o
 * [B, N, H, d] bf16, lse [B, H, N] fp32.  Packed (cu_seqlens int32[B+1] on
 * the device, lengths <= N, checked on the device like attn_fwd's): q, k, v, o
 * [total, H, d], lse [H, total], total = cu_seqlens[B].  The per-sequence
 * outputs of the quantisers keep their dense shapes with N as the length
 * bound: a sequence of length L has blocks [0, ceil(L / 128)) written, the
 * rest of its rows untouched.  Same conventions as attn_fwd.h (device
 * pointers, asynchronous on stream, status codes, error word); d other than
 * 64 or 128 returns ATTN_ERR_HEADDIM.
 */
#ifndef IO_AWARE_EXACT_06_ATTN_FP8_H
#define IO_AWARE_EXACT_06_ATTN_FP8_H

#include <stdint.h>

#include "attn_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_fp8_quantize_qk: the Q or K quantisation step.  x [B, N, H, d] bf16
 * (packed: [total, H, d]); codes e4m3 (uint8) of the same shape; scales
 * [B, H, T] fp32, T = ceil(N / 128): block t holds rows [128 t, 128 t + 128)
 * of a sequence (of length L) and head, the last block pulled back to end at L
 * (the rows it shares with block t - 1 keep that block's codes; rows before
 * the sequence count as zero).  cu_seqlens: NULL (dense) or as above.  signs:
 * host array of d int8 (+1 / -1) for the rotation, or NULL for no rotation.
 */
int attn_fp8_quantize_qk(const void *x, uint8_t *codes, float *scales, int B, int H, int N,
                         int d, const int32_t *cu_seqlens, const int8_t *signs,
                         attn_stream_t stream);

/*
 * attn_fp8_quantize_v: the V quantisation step.  v [B, N, H, d] bf16
 * (packed: [total, H, d]); codes_t [B, H, d, Np] e4m3 with
 * Np = 128 * ceil(N / 128): the codes transposed per sequence and head (keys
 * contiguous), keys L .. 128 ceil(L / 128) - 1 zero for a sequence of length
 * L; scale [B, H] fp32 (max |V| / 448 of the sequence and head; 1 when that
 * max is 0; not written for an empty sequence).  cu_seqlens: NULL or as above.
 */
int attn_fp8_quantize_v(const void *v, uint8_t *codes_t, float *scale, int B, int H, int N,
                        int d, const int32_t *cu_seqlens, attn_stream_t stream);

/*
 * attn_fwd_fp8: O = softmax(scale * Q K^T) V and the LSE through the FP8 path
 * above (quantisation kernels, then the FP8 attention kernel).  scale: finite
 * and >= 0; causal and cu_seqlens as in attn_fwd (an invalid cu_seqlens sets
 * ATTN_ERR_SEQLENS in the error word and nothing is computed).  signs: as for
 * attn_fp8_quantize_qk.  The library keeps a per-(device, stream) workspace
 * for the codes and scales (about 4 * B * N * H * 128 bytes), grown on demand.
 */
int attn_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                 int N, int d, float scale, int causal, const int32_t *cu_seqlens,
                 const int8_t *signs, attn_stream_t stream);

/*
 * attn_fwd_fp8_codes: the FP8 attention step of attn_fwd_fp8 alone, on codes
 * and scales the caller made with attn_fp8_quantize_qk and
 * attn_fp8_quantize_v, so that keys and values quantised once (a key/value
 * cache) serve many query batches.  d must be 128 (the quantisers' code rows
 * are then the 128-byte rows the attention kernel reads; d = 64 returns
 * ATTN_ERR_HEADDIM).  q8, k8: [B, N, H, 128] e4m3 (packed [total, H, 128]);
 * sq, sk: [B, H, T] fp32; vt: [B, H, 128, Np] e4m3; sv: [B, H] fp32 (the
 * quantisers' layouts).  rotated: nonzero when Q and K were quantised with
 * the same signs (the rotated logits carry the factor d of the unnormalised
 * rotation, divided out here); zero when both were quantised without.
 * o, lse, scale, causal, cu_seqlens: as for attn_fwd_fp8.  Alignment: q8,
 * k8, vt, o 16 bytes; the scales and lse 4 bytes.  Same ordering, errors
 * and worklist workspace as attn_fwd_fp8; O and the LSE equal attn_fwd_fp8's
 * on the same inputs bit for bit.
 */
int attn_fwd_fp8_codes(const uint8_t *q8, const float *sq, const uint8_t *k8, const float *sk,
                       const uint8_t *vt, const float *sv, void *o, float *lse, int B, int H,
                       int N, int d, float scale, int causal, int rotated,
                       const int32_t *cu_seqlens, attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* IO_AWARE_EXACT_06_ATTN_FP8_H */
