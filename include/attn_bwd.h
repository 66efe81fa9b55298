/*
 * C ABI of the GB300 (sm_103a) fused exact attention backward.
 *
 * Given the forward's inputs Q, K, V, its outputs O and LSE (from attn_fwd)
 * and the gradient dO of a loss with respect to O, computes
 *     dV_j = sum_i P_ij dO_i
 *     dK_j = scale * sum_i dS_ij q_i
 *     dQ_i = scale * sum_j dS_ij k_j
 * with P_ij = exp(scale q_i.k_j - LSE_i), dS_ij = P_ij (dO_i.v_j - dO_i.O_i),
 * over the visible (i, j) pairs (all, or j <= i when causal), rebuilding the
 * score and probability tiles from Q, K, V and the LSE instead of reading
 * stored ones ("flash-attention-evolution" (letsgetai), FlashAttention
 * "核心机制", recomputation paragraph; "FlashAttention 1-4 演进速查"
 * (argus-lessons), FlashAttention-1 items).  The LSE output of the forward is
 * taken to carry no gradient of its own.
 *
 * Numerics: bf16 inputs, fp32 accumulation; P and dS rounded to bf16 before
 * their products; dQ, dK, dV written as bf16 (round to nearest even).  D_i =
 * dO_i.O_i uses the forward's bf16 O, so on a row where one key carries
 * nearly all of P, dS = P (dP - D) is a difference of nearly equal terms and
 * keeps the bf16 rounding of O (about 2^-9 |dO_i| |v_j|): dQ_i and dK_j of
 * such rows have that absolute error where their exact values are near 0.
 *
 * Only sm_103 devices; device pointers; asynchronous on `stream`; argument
 * errors are reported synchronously before anything is launched.  Status
 * codes are those of attn_fwd.h.
 */
#ifndef IO_AWARE_EXACT_06_ATTN_BWD_H
#define IO_AWARE_EXACT_06_ATTN_BWD_H

#include <stdint.h>

#include "attn_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_bwd: dQ, dK, dV of attn_fwd.
 *
 * Layouts as for attn_fwd, with dout, dq, dk, dv laid out like q:
 *   dense (cu_seqlens == NULL): q, k, v, o, dout, dq, dk, dv [B, N, H, d]
 *   bf16, lse [B, H, N] fp32; packed (cu_seqlens != NULL, device int32
 *   [B+1], validated on the device): [total, H, d] and lse [H, total], N >=
 *   every length, at most 8192 tiles of 128 rows per sequence.  lse is the
 *   one attn_fwd wrote for the same q, k, v, scale and causal flag.
 * q, k, v, o, dout, lse: read only.  dq, dk, dv: every element of every
 *   sequence written.
 * d: 64 or 128.  scale and causal: those of the forward call.
 * Alignment: the bf16 tensors 16-byte aligned; lse 4-byte aligned.
 * Ownership: the caller owns every buffer.  The library keeps a cached
 *   per-(device, stream) workspace of 2 * B * H * ceil(N / 128) * 128 floats
 *   (each row's D = <dO, O> and LSE * log2(e)) and, for packed batches, its
 *   scheduling lists, grown on demand; device-side errors (an expired bounded
 *   wait, invalid cu_seqlens) are latched in the same error word as the
 *   forward's and read by attn_last_device_error.
 * B == 0, N == 0 or H == 0 is a no-op returning ATTN_OK.
 * Returns ATTN_OK or a negative attn_status; nothing is launched on error.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
             const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
             float scale, int causal, const int32_t *cu_seqlens, attn_stream_t stream);

/*
 * attn_bwd_window: attn_bwd for attn_fwd_window's sliding window: key j is
 * visible to query i iff i - window_left <= j <= i + window_right (-1: no
 * bound on that side), within the sequence and j <= i when causal; the
 * window and lse must be those of the forward call.  Tiles no query and key
 * of the window pair up in are skipped.  A window value below -1 returns
 * ATTN_ERR_SHAPE; otherwise as attn_bwd ((-1, -1) is attn_bwd).
 */
int attn_bwd_window(const void *q, const void *k, const void *v, const void *o, const void *dout,
                    const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                    float scale, int causal, int window_left, int window_right,
                    const int32_t *cu_seqlens, attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* IO_AWARE_EXACT_06_ATTN_BWD_H */
