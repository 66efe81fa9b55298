/*
 * C ABI of the GB300 (sm_103a) fused exact attention forward.
 *
 * Computes, for every sequence s, head h and query row i,
 *     O_i   = sum_j softmax_j(scale * q_i . k_j) v_j
 *     LSE_i = log sum_j exp(scale * q_i . k_j)        (natural log)
 * over the visible keys j (all keys of the sequence, or j <= i when causal),
 * in one kernel that never writes the score or probability matrices to device
 * memory: tiles of Q, K and V with a running row max and running row sum
 * ("flash-attention-evolution" (letsgetai), FlashAttention section "核心机制";
 * "FlashAttention" (compassingai), section 3 "技術原理").
 *
 * Numerics: bf16 inputs, fp32 accumulation, P rounded to bf16 before the PV
 * product, O written as bf16 (round to nearest even), LSE as fp32.
 *
 * Only sm_103 devices are supported (the kernels are built for sm_103a only).
 * All pointers are device pointers unless stated otherwise.  Every call is
 * asynchronous on `stream` like any CUDA kernel launch; argument errors are
 * reported synchronously, before anything is launched.
 */
#ifndef IO_AWARE_EXACT_06_ATTN_FWD_H
#define IO_AWARE_EXACT_06_ATTN_FWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = -1,           /* a required pointer is NULL */
    ATTN_ERR_SHAPE = -2,          /* B, H or N negative or too large */
    ATTN_ERR_HEADDIM = -3,        /* d is not 64 or 128 */
    ATTN_ERR_ALIGN = -4,          /* q/k/v/o not 16-byte or lse not 4-byte aligned */
    ATTN_ERR_SCALE = -5,          /* scale is negative or not finite */
    ATTN_ERR_CUDA = -6,           /* a CUDA runtime call or launch failed */
    ATTN_ERR_DEVICE_TIMEOUT = -7, /* a bounded device-side wait expired */
    ATTN_ERR_SEQLENS = -8,        /* cu_seqlens not increasing from 0, or a length > N */
    ATTN_ERR_ARCH = -9,           /* current device is not sm_103 */
    ATTN_ERR_SCRATCH = -10        /* attn_fwd_noalloc: problem larger than its fixed scratch */
} attn_status;

/*
 * attn_fwd: O = softmax(scale * Q K^T) V and the per-row LSE.
 *
 * Layout, dense (cu_seqlens == NULL): q, k, v, o are contiguous [B, N, H, d]
 *   bf16 (token-major, heads interleaved); lse is [B, H, N] fp32.
 * Layout, packed variable length (cu_seqlens != NULL): q, k, v, o are
 *   [total, H, d] with total = cu_seqlens[B]; sequence s occupies tokens
 *   cu_seqlens[s] .. cu_seqlens[s+1]-1; lse is [H, total].  N must be >= every
 *   sequence length (it bounds the work list); cu_seqlens is int32[B+1] in
 *   device memory and is validated on the device (see attn_last_device_error).
 *   Zero-length sequences are allowed.
 * q, k, v: read only.  o, lse: written for every valid row, nothing else.
 * d: 64 or 128.  scale: finite and >= 0 (1/sqrt(d) for the usual attention).
 * causal: nonzero means key j is visible to query i iff j <= i (within each
 *   sequence); zero means every key of the sequence is visible.
 * Alignment: q, k, v, o 16-byte aligned; lse 4-byte aligned.
 * Ownership: the caller owns every buffer and keeps it alive until the stream
 *   work has finished.  The library keeps a small cached device workspace per
 *   (device, stream) pair (the scheduling list) and an error word per device,
 *   allocated on first use.  Calls on one stream are ordered; calls on
 *   different streams may run concurrently.
 * B == 0, N == 0 or H == 0 is a no-op returning ATTN_OK.
 * Returns ATTN_OK or a negative attn_status; nothing is launched on error.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int H, int N, int d, float scale, int causal,
             const int32_t *cu_seqlens, attn_stream_t stream);

/*
 * attn_fwd_window: attn_fwd with a sliding window.  Key j is visible to query
 * i iff i - window_left <= j <= i + window_right (within the sequence, and
 * j <= i when causal); -1 leaves that side unbounded, so (-1, -1) is attn_fwd.
 * Tiles outside every row's window are skipped, so the cost grows with the
 * window, not with the sequence.  Sliding-window masks over the same tiled
 * kernel: "FlashAttention" (compassingai), section 5, FlexAttention item.
 * Same layouts, ownership and errors as attn_fwd; a window value below -1
 * returns ATTN_ERR_SHAPE.
 */
int attn_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse,
                    int B, int H, int N, int d, float scale, int causal,
                    int window_left, int window_right, const int32_t *cu_seqlens,
                    attn_stream_t stream);

/*
 * attn_fwd_kvsplit: queries and keys of different lengths, the keys of every
 * query block processed in num_splits ranges by separate work units whose
 * partial results (O / l and LSE per range, fp32) are merged afterwards by
 * the two-segment merge identity ("flash-attention-evolution" (letsgetai),
 * FlashAttention "核心机制"); parallelising over the key sequence for
 * inference is the pages' FlashDecoding item ("FlashAttention" (compassingai),
 * section 5).
 * Layout (dense): q, o [B, Nq, H, d]; k, v [B, Nk, H, d]; lse [B, H, Nq].
 * causal: query row r sits at key position Nk - Nq + r (the queries are the
 *   last Nq positions of the key sequence) and sees keys j <= Nk - Nq + r;
 *   requires Nq <= Nk.  Non-causal: every key is visible.
 * Nq == 1 (decoding one token) runs on CUDA cores: a matrix-vector product
 *   per (sequence, head), bound by reading K and V; Nq > 1 runs on the tensor
 *   cores in 256-row query blocks, and with Nq <= 128 (one 128-row query tile)
 *   the two halves of a unit take the tile against two key ranges each.
 * num_splits: 1..256 ranges, or 0 to choose (Nq == 1: about 16 (sequence,
 *   head, range) items per SM, ranges of at least 64 keys; else the count
 *   with the shortest estimated makespan over the SMs, at most 64).  With
 *   2 <= Nq <= 128 an odd count is raised by one.
 * Ownership: like attn_fwd; in addition the library keeps a per-(device,
 *   stream) fp32 workspace for the partial results, grown on demand.
 * Errors: like attn_fwd; Nk == 0, num_splits outside [0, 256] or causal with
 *   Nq > Nk return ATTN_ERR_SHAPE.
 */
int attn_fwd_kvsplit(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H, int Nq, int Nk, int d, float scale, int causal,
                     int num_splits, attn_stream_t stream);

/*
 * attn_fwd_decode: one query per sequence (the newest token) against the
 * sequence's packed keys, which differ in length from sequence to sequence
 * (a key/value cache): O_b = softmax(scale q_b K_b^T) V_b over every key of
 * sequence b, computed as attn_fwd_kvsplit computes Nq == 1 (key ranges on
 * CUDA cores, merged by the two-segment merge identity).
 * Layout: q, o [B, H, d] bf16; k, v [total, H, d] bf16 with total =
 *   cu_seqlens_k[B], sequence b's keys at tokens cu_seqlens_k[b] ..
 *   cu_seqlens_k[b+1]-1; lse [B, H] fp32.  cu_seqlens_k: device int32[B+1].
 * max_seqlen_k >= every key length (sizes the ranges; checked on the device).
 * A sequence with no key gets O = 0 and LSE = -inf.
 * num_splits: ranges per sequence, 1..256, or 0 to choose (about 16
 *   (sequence, head, range) items per SM, ranges of at least 64 keys of the
 *   longest sequence).
 * Ownership: like attn_fwd_kvsplit.
 * Errors: like attn_fwd; cu_seqlens_k not starting at 0, decreasing, or with
 *   a length above max_seqlen_k: ATTN_ERR_SEQLENS in the error word and
 *   nothing is read past the check or written.
 */
int attn_fwd_decode(const void *q, const void *k, const void *v, void *o, float *lse,
                    int B, int H, int d, float scale, const int32_t *cu_seqlens_k,
                    int max_seqlen_k, int num_splits, attn_stream_t stream);

/*
 * attn_fwd_host: attn_fwd on HOST buffers.  The call copies Q, K, V to the
 * device, computes O and the LSE with attn_fwd's kernels, and copies them
 * back, in groups of heads so that the copies of one group overlap the
 * attention of the next: group g + 1 is copied in on one internal stream
 * while group g is computed on `stream` and group g - 1 is copied out on
 * another.  Every row is computed exactly as by attn_fwd, so O and the LSE
 * are bit-identical to attn_fwd's on the same inputs.  This is plumbing
 * around the pages' kernel, which assumes its inputs already sit in HBM
 * ("flash-attention-evolution" (letsgetai), FlashAttention "核心机制").
 * Arguments and layouts: those of attn_fwd, with every buffer (cu_seqlens
 *   included) in host (or any) memory: dense q, k, v, o [B, N, H, d] bf16 and
 *   lse [B, H, N] fp32; packed [total, H, d] and lse [H, total] with total =
 *   cu_seqlens[B].  Page-locked host memory lets the copies run
 *   asynchronously and overlap; with pageable memory the call still works,
 *   its copies serialise with the host.
 * Ordering: the call is asynchronous like attn_fwd.  Its work starts after
 *   the work queued on `stream` before it, and the work queued on `stream`
 *   after it starts once o and lse are written; synchronise `stream` before
 *   reading them.  The caller keeps the host buffers alive and unchanged
 *   until then.
 * Ownership: the library keeps, per (device, stream), two internal copy
 *   streams, their events and a device workspace for two head groups (four
 *   [tokens, hg, d] tiles, the group's LSE and a copy of cu_seqlens each),
 *   grown on demand.
 * Errors: like attn_fwd (no alignment requirement on the host buffers).
 *   cu_seqlens is checked on the host before anything is copied: not
 *   starting at 0, decreasing, or with a length above N returns
 *   ATTN_ERR_SEQLENS.  A failed copy returns ATTN_ERR_CUDA; device-side
 *   errors are read with attn_last_device_error(stream).
 */
int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int H, int N, int d, float scale, int causal,
                  const int32_t *cu_seqlens, attn_stream_t stream);

/* Options of attn_fwd_ex.  Zero-initialise and set what is needed. */
typedef struct {
    uint64_t wait_timeout_ns; /* bound on each device-side wait; 0 = 2 s */
    int fault_inject;         /* 0 = none; 1 = CTA 0 never issues its first K copy,
                                 so a bounded wait must expire (tests only) */
    int max_ctas;             /* 0 = one persistent CTA per SM; else at most this many */
    int kernel;               /* 0 = the library's choice (3); 1 = one CTA per unit,
                                 two softmax threads per query row; 3 = one CTA per
                                 unit, one softmax thread per row; 2 = the pair-of-SMs
                                 kernel (two SMs share each product; d = 128 without a
                                 window only, else ATTN_ERR_SHAPE; ATTN_ERR_CUDA if the
                                 device cannot run it) */
} attn_fwd_options;

/* attn_fwd with options (opts may be NULL).  Same arguments and errors. */
int attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                int B, int H, int N, int d, float scale, int causal,
                const int32_t *cu_seqlens, attn_stream_t stream,
                const attn_fwd_options *opts);

/*
 * Synchronises `stream`, then returns and clears the device-side error word
 * of the current device: ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT (a bounded wait
 * expired; the kernel stopped early and its outputs are incomplete) or
 * ATTN_ERR_SEQLENS (invalid cu_seqlens; nothing was computed).  Returns
 * ATTN_ERR_CUDA if the synchronisation itself fails.
 */
int attn_last_device_error(attn_stream_t stream);

/* Identifier of the wait that expired, as read by the last
 * attn_last_device_error call (0 if none); for diagnostics. */
int attn_last_error_site(void);

/* The cudaError_t behind the last ATTN_ERR_CUDA of this thread (0 if none). */
int attn_last_cuda_error(void);

/*
 * attn_fwd_noalloc: attn_fwd for callers that must not allocate device memory.
 *
 * The pages have no counterpart to this entry point.  It exists for callers
 * that cannot call cudaMalloc: code that runs inside another framework whose
 * memory pool owns all device memory, or a runtime that forbids device
 * allocation after start-up because an allocation may synchronise the device
 * or fail at an arbitrary point of a latency-critical loop.  attn_fwd
 * allocates a small workspace on its first call per device and stream; this
 * variant allocates nothing: its scratch (the error word and
 * the scheduling list of packed batches) is a fixed array of 8 + 2 * 65536
 * int32 (about 512 KB) in the library's own device memory, which every GPU
 * that loads the library holds until the process exits.
 *
 * Same arguments, layouts and results as attn_fwd.  Differences:
 *   - Packed batches (cu_seqlens given): B * ceil(N / 256) must not exceed
 *     65536 (the number of (sequence, 256-row block) pairs the scratch
 *     holds); larger ones return ATTN_ERR_SCRATCH before anything is
 *     launched.  Dense batches keep no list there and have no such limit.
 *   - The first call on a device does the set-up for that device (kernel
 *     attributes and the device address of the scratch array); make that
 *     first call before any stream capture.  No call allocates device memory.
 *   - Every call clears the words that must start at zero (with an
 *     asynchronous memset on `stream`) and then shares the same scratch:
 *     calls whose work overlaps on the GPU (different streams, or different
 *     host threads without ordering) race on it and must be serialised by
 *     the caller.  The array keeps the last call's contents.
 *   - Device-side errors of this variant (an expired bounded wait, invalid
 *     cu_seqlens) are recorded in its scratch, not in the error word read by
 *     attn_last_device_error; read them with
 *     attn_fwd_noalloc_last_device_error.  The outputs of such a call are
 *     incomplete (with invalid cu_seqlens nothing is written).
 */
int attn_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H, int N, int d, float scale, int causal,
                     const int32_t *cu_seqlens, attn_stream_t stream);

/* attn_fwd_noalloc with the options of attn_fwd_ex (opts may be NULL): the
 * bound on each device-side wait, the test hook that makes one wait expire,
 * a cap on the CTAs.  Allocates nothing either; same arguments and errors. */
int attn_fwd_noalloc_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                        int B, int H, int N, int d, float scale, int causal,
                        const int32_t *cu_seqlens, attn_stream_t stream,
                        const attn_fwd_options *opts);

/*
 * The device-side error status of the attn_fwd_noalloc calls on the current
 * device since the last one started (each call clears it when it starts):
 * synchronises `stream`, reads the error words of the fixed scratch with
 * plain copies (no allocation), clears them and returns ATTN_OK,
 * ATTN_ERR_DEVICE_TIMEOUT (a bounded wait expired; that call's outputs are
 * incomplete), ATTN_ERR_SEQLENS (invalid cu_seqlens; nothing was computed)
 * or ATTN_ERR_SHAPE; ATTN_ERR_CUDA if the synchronisation or a copy fails.
 * The site of an expired wait is then read with attn_last_error_site.  Like
 * the calls it reports on, it races with attn_fwd_noalloc work of another
 * stream that overlaps it on the GPU.  The pages have no counterpart to it.
 */
int attn_fwd_noalloc_last_device_error(attn_stream_t stream);

/* Bytes of device memory the library currently holds in its own workspaces
 * (error words, scheduling lists, split-KV partial results, attn_fwd_host's
 * slots, the backward's and the FP8 path's buffers), over all devices.
 * attn_fwd_noalloc adds nothing to it.  For diagnostics; not on the pages. */
size_t attn_device_bytes(void);

/* A static, human-readable name of a status code. */
const char *attn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* IO_AWARE_EXACT_06_ATTN_FWD_H */
