/*
 * fp64 CPU oracle for exact softmax attention: forward pass and its gradients.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path, and nothing in the CUDA path may
 * call it.
 *
 * What it computes (the plain definition, for one sequence s, head h, row i):
 *
 *   S_ij  = scale * sum_k q_ik k_jk        for every visible key j
 *   m_i   = max_j S_ij
 *   l_i   = sum_j exp(S_ij - m_i)
 *   P_ij  = exp(S_ij - m_i) / l_i
 *   O_i   = sum_j P_ij v_j
 *   LSE_i = m_i + log(l_i)                 (natural log, scaled-logit units)
 *
 * Sources on the pages:
 *   - the attention formula softmax(Q K^T / sqrt(d)) V: "flash-attention-evolution"
 *     (letsgetai), section "为什么 attention 慢", display equation;
 *   - materialise S, then P = softmax(S), then O = P V: "FlashAttention"
 *     (compassingai), section 3 "技術原理", the three-step listing of standard
 *     attention (read for what it computes);
 *   - normalise by l once at the end: "flash-attention-evolution", section
 *     FlashAttention "核心机制", the two-segment merge equations (softmax = f / l).
 *
 * Readings where the pages are silent: "visible" is every key j < L_s, or
 * j <= i when causal (lower-triangular mask within each sequence); the LSE is
 * the natural log of sum_j exp(S_ij) in units of the scaled logits.
 * Sliding windows ("FlashAttention" (compassingai), section 5, FlexAttention
 * item: sliding-window masks over the same tiled kernel) narrow the visible
 * keys further to i - wl <= j <= i + wr (wl, wr < 0: no bound on that side).
 *
 * Inputs are bf16 bit patterns (uint16) in the packed layout
 * [tokens, H, d]; sequence s occupies tokens cu_seqlens[s] .. cu_seqlens[s+1]-1.
 * Every bf16 value widens exactly to fp64 here; nothing is rounded afterwards.
 *
 * Backward (oracle_attn_bwd).  The pages say only that the backward pass
 * rebuilds S and P from Q, K, V (and the saved row statistics) instead of
 * storing them ("flash-attention-evolution" (letsgetai), FlashAttention
 * "核心机制", the recomputation paragraph; "FlashAttention 1-4 演进速查"
 * (argus-lessons), FlashAttention-1 items).  What the backward computes is
 * then the derivative of the definition above, given the gradient dO of a
 * scalar loss with respect to O (and none with respect to the LSE): by the
 * chain rule through O_i = sum_j P_ij v_j and the row softmax,
 *
 *   dV_j   = sum_i P_ij dO_i
 *   dP_ij  = <dO_i, v_j>
 *   D_i    = sum_j P_ij dP_ij
 *   dS_ij  = P_ij (dP_ij - D_i)
 *   dQ_i   = scale * sum_j dS_ij k_j
 *   dK_j   = scale * sum_i dS_ij q_i
 *
 * over the same visible (i, j) pairs as the forward (with a sliding window:
 * oracle_attn_bwd_window).
 *
 * FP8 (oracle_fp8_quantize, oracle_attn_rows_f64).  The pages name the FP8
 * forward's two devices without formulas: block quantisation and incoherent
 * processing ("flash-attention-evolution" (letsgetai), FlashAttention-3
 * section, item 3; "FlashAttention 1-4 演进速查" (argus-lessons),
 * FlashAttention-3 items).  Readings taken here:
 *   - incoherent processing multiplies Q and K along d by the same orthogonal
 *     matrix, diag(signs) H_d / sqrt(d) with H_d the Sylvester-Hadamard
 *     matrix, so Q K^T is unchanged; the transform is computed unnormalised
 *     (butterflies in fp32) and the 1/d it leaves in Q K^T goes into the
 *     logit scale;
 *   - block quantisation gives every block its own scale: the block's largest
 *     |x| maps to 448, the largest finite e4m3 value; codes are e4m3, rounded
 *     to nearest even, saturating.
 * Because a quantised code is an integer decided by floating point, this
 * oracle takes each step in fp32 in the kernel's order (the butterfly
 * stages, the max, 448 / amax, x * (448 / amax), the rounding), so codes and
 * scales are reproduced bit for bit.  The attention of the dequantised values
 * is then the plain definition again, in fp64 (oracle_attn_rows_f64).
 *
 * Besides the definition, two more routines restate the pages' own incremental
 * formulations so the tests can pin one against the other:
 *   - oracle_softmax_merge: the two-segment (m, l, f) merge identity;
 *   - oracle_attn_online:   the block-by-block running-max / running-sum loop
 *     ("FlashAttention", compassingai, section 3, online softmax listing),
 *     finished with the division by l that the merge equations add.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Number of CPUs in this process's affinity mask (at least 1). */
int oracle_cpu_count(void)
{
    cpu_set_t set;
    CPU_ZERO(&set);
    if (sched_getaffinity(0, sizeof set, &set) == 0) {
        int n = CPU_COUNT(&set);
        if (n > 0)
            return n;
    }
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

typedef struct {
    const uint16_t *q, *k, *v;
    const int64_t *cu;
    int64_t nseq;
    int H, d;
    double scale;
    int causal;
    int64_t wl, wr;      /* window: i - wl <= j <= i + wr; negative = unbounded */
    const int64_t *rows; /* [nrows][3] = (seq, head, row) */
    int64_t nrows;
    double *o;   /* [nrows][d] */
    double *lse; /* [nrows] */
    int64_t begin, end;
    int status;
} rows_job;

/* Checks one requested row and returns its sequence bounds. */
static int row_bounds(const rows_job *jb, int64_t r, int64_t *base, int64_t *L,
                      int64_t *i, int *h)
{
    int64_t s = jb->rows[3 * r + 0];
    int64_t hh = jb->rows[3 * r + 1];
    int64_t ii = jb->rows[3 * r + 2];
    if (s < 0 || s >= jb->nseq || hh < 0 || hh >= jb->H)
        return ORACLE_EINVAL;
    *base = jb->cu[s];
    *L = jb->cu[s + 1] - jb->cu[s];
    if (ii < 0 || ii >= *L)
        return ORACLE_EINVAL;
    *i = ii;
    *h = (int)hh;
    return ORACLE_OK;
}

static void *rows_worker(void *arg)
{
    rows_job *jb = (rows_job *)arg;
    const int H = jb->H, d = jb->d;
    int64_t maxL = 0;
    for (int64_t s = 0; s < jb->nseq; ++s)
        if (jb->cu[s + 1] - jb->cu[s] > maxL)
            maxL = jb->cu[s + 1] - jb->cu[s];
    double *srow = (double *)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1));
    double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
    if (!srow || !qrow) {
        free(srow);
        free(qrow);
        jb->status = ORACLE_ENOMEM;
        return NULL;
    }
    for (int64_t r = jb->begin; r < jb->end; ++r) {
        int64_t base, L, i;
        int h;
        if (row_bounds(jb, r, &base, &L, &i, &h) != ORACLE_OK) {
            jb->status = ORACLE_EINVAL;
            break;
        }
        /* visible keys [jlo, jhi): the whole sequence, or j <= i when causal,
           narrowed by the window to i - wl <= j <= i + wr */
        int64_t jlo = 0, jhi = jb->causal ? i + 1 : L;
        if (jb->wl >= 0 && i - jb->wl > jlo)
            jlo = i - jb->wl;
        if (jb->wr >= 0 && i + jb->wr + 1 < jhi)
            jhi = i + jb->wr + 1;
        const int64_t nvis = jhi > jlo ? jhi - jlo : 0;
        const uint16_t *qi = jb->q + ((base + i) * H + h) * (int64_t)d;
        for (int c = 0; c < d; ++c)
            qrow[c] = widen_bf16(qi[c]);
        /* S_ij = scale * <q_i, k_j> for every visible key, materialised */
        for (int64_t j = jlo; j < jhi; ++j) {
            const uint16_t *kj = jb->k + ((base + j) * H + h) * (int64_t)d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += qrow[c] * widen_bf16(kj[c]);
            srow[j - jlo] = jb->scale * dot;
        }
        /* m_i = max_j S_ij */
        double m = -INFINITY;
        for (int64_t j = 0; j < nvis; ++j)
            if (srow[j] > m)
                m = srow[j];
        /* l_i = sum_j exp(S_ij - m_i) */
        double l = 0.0;
        for (int64_t j = 0; j < nvis; ++j)
            l += exp(srow[j] - m);
        /* P_ij = exp(S_ij - m_i) / l_i ;  O_i = sum_j P_ij v_j */
        double *oi = jb->o + r * (int64_t)d;
        for (int c = 0; c < d; ++c)
            oi[c] = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            const double p = exp(srow[j] - m) / l;
            const uint16_t *vj = jb->v + ((base + jlo + j) * H + h) * (int64_t)d;
            for (int c = 0; c < d; ++c)
                oi[c] += p * widen_bf16(vj[c]);
        }
        /* LSE_i = m_i + log(l_i) */
        jb->lse[r] = nvis > 0 ? m + log(l) : -INFINITY;
    }
    free(srow);
    free(qrow);
    return NULL;
}

static int check_common(const void *q, const void *k, const void *v, const int64_t *cu,
                        int64_t nseq, int H, int d, double scale)
{
    if (!q || !k || !v || !cu || nseq < 0 || H <= 0 || d <= 0 || !isfinite(scale))
        return ORACLE_EINVAL;
    if (cu[0] != 0)
        return ORACLE_EINVAL;
    for (int64_t s = 0; s < nseq; ++s)
        if (cu[s + 1] < cu[s])
            return ORACLE_EINVAL;
    return ORACLE_OK;
}

/*
 * O and LSE of the requested rows, by the plain definition above, with the
 * visible keys of row i narrowed to i - wl <= j <= i + wr (wl, wr < 0: no
 * bound on that side).  nthreads <= 0 uses every CPU of the affinity mask; *threads_used (if not
 * NULL) receives the number of threads that ran.  Returns 0, or a negative
 * code for a bad argument (row outside its sequence, decreasing cu_seqlens...).
 */
int oracle_attn_rows_window(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const int64_t *cu_seqlens, int64_t nseq, int H, int d,
                            double scale, int causal, int64_t wl, int64_t wr,
                            const int64_t *rows, int64_t nrows, double *o, double *lse,
                            int nthreads, int *threads_used)
{
    int st = check_common(q, k, v, cu_seqlens, nseq, H, d, scale);
    if (st != ORACLE_OK || nrows < 0 || (nrows > 0 && (!rows || !o || !lse)))
        return ORACLE_EINVAL;
    int nt = nthreads > 0 ? nthreads : oracle_cpu_count();
    if (nt > nrows)
        nt = nrows > 0 ? (int)nrows : 1;
    rows_job *jobs = (rows_job *)calloc((size_t)nt, sizeof(rows_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return ORACLE_ENOMEM;
    }
    int started = 0;
    for (int t = 0; t < nt; ++t) {
        rows_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v;
        jb->cu = cu_seqlens; jb->nseq = nseq;
        jb->H = H; jb->d = d; jb->scale = scale; jb->causal = causal;
        jb->wl = wl; jb->wr = wr;
        jb->rows = rows; jb->nrows = nrows; jb->o = o; jb->lse = lse;
        jb->begin = nrows * t / nt;
        jb->end = nrows * (t + 1) / nt;
        jb->status = ORACLE_OK;
    }
    if (nt == 1) {
        rows_worker(&jobs[0]);
        started = 1;
    } else {
        for (int t = 0; t < nt; ++t) {
            if (pthread_create(&tid[t], NULL, rows_worker, &jobs[t]) != 0)
                break;
            ++started;
        }
        /* rows of threads that failed to start run on this thread */
        for (int t = started; t < nt; ++t)
            rows_worker(&jobs[t]);
        for (int t = 0; t < started; ++t)
            pthread_join(tid[t], NULL);
    }
    for (int t = 0; t < nt; ++t)
        if (jobs[t].status != ORACLE_OK)
            st = jobs[t].status;
    if (threads_used)
        *threads_used = nt == 1 ? 1 : (started > 0 ? started : 1);
    free(jobs);
    free(tid);
    return st;
}

/* O and LSE of the requested rows without a window (every visible key). */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const int64_t *cu_seqlens, int64_t nseq, int H, int d,
                     double scale, int causal, const int64_t *rows, int64_t nrows,
                     double *o, double *lse, int nthreads, int *threads_used)
{
    return oracle_attn_rows_window(q, k, v, cu_seqlens, nseq, H, d, scale, causal, -1, -1, rows,
                                   nrows, o, lse, nthreads, threads_used);
}

/*
 * The probability row P_i (length nvis: L_s, or i+1 when causal) of one query
 * row, by the plain definition.  p must hold L_s doubles.  Returns the number
 * of visible keys written, or a negative code.
 */
int64_t oracle_attn_probs(const uint16_t *q, const uint16_t *k,
                          const int64_t *cu_seqlens, int64_t nseq, int H, int d,
                          double scale, int causal, int64_t seq, int h, int64_t i,
                          double *p)
{
    static const uint16_t dummy = 0;
    int st = check_common(q, k, &dummy, cu_seqlens, nseq, H, d, scale);
    if (st != ORACLE_OK || !p || seq < 0 || seq >= nseq || h < 0 || h >= H)
        return ORACLE_EINVAL;
    const int64_t base = cu_seqlens[seq];
    const int64_t L = cu_seqlens[seq + 1] - base;
    if (i < 0 || i >= L)
        return ORACLE_EINVAL;
    const int64_t nvis = causal ? i + 1 : L;
    const uint16_t *qi = q + ((base + i) * H + h) * (int64_t)d;
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        const uint16_t *kj = k + ((base + j) * H + h) * (int64_t)d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += widen_bf16(qi[c]) * widen_bf16(kj[c]);
        p[j] = scale * dot;
        if (p[j] > m)
            m = p[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j)
        l += exp(p[j] - m);
    for (int64_t j = 0; j < nvis; ++j)
        p[j] = exp(p[j] - m) / l;
    return nvis;
}

/*
 * Softmax of x[0..n) computed segment by segment with the two-segment merge
 * identity ("flash-attention-evolution", section FlashAttention "核心机制"):
 * for x = (x1, x2),
 *   m(x) = max(m(x1), m(x2)),
 *   l(x) = e^{m(x1)-m(x)} l(x1) + e^{m(x2)-m(x)} l(x2),
 *   f(x) = [e^{m(x1)-m(x)} f(x1), e^{m(x2)-m(x)} f(x2)],
 *   softmax(x) = f(x) / l(x),
 * where for one segment m is its max, f = exp(x - m) and l = sum f.
 * The segment boundaries are cuts[0..ncuts) (strictly increasing, inside
 * (0, n)).  Segments are merged left to right into a running (m, l, f).
 * Writes softmax(x) to out and returns 0; *m_out and *l_out get the merged
 * statistics.
 */
int oracle_softmax_merge(const double *x, int64_t n, const int64_t *cuts, int64_t ncuts,
                         double *out, double *m_out, double *l_out)
{
    if (!x || !out || n <= 0 || ncuts < 0 || (ncuts > 0 && !cuts))
        return ORACLE_EINVAL;
    for (int64_t c = 0; c < ncuts; ++c)
        if (cuts[c] <= 0 || cuts[c] >= n || (c > 0 && cuts[c] <= cuts[c - 1]))
            return ORACLE_EINVAL;
    double m_run = -INFINITY, l_run = 0.0;
    int64_t lo = 0;
    for (int64_t seg = 0; seg <= ncuts; ++seg) {
        const int64_t hi = seg < ncuts ? cuts[seg] : n;
        /* statistics of the new segment x2 = x[lo, hi) */
        double m2 = -INFINITY;
        for (int64_t j = lo; j < hi; ++j)
            if (x[j] > m2)
                m2 = x[j];
        double l2 = 0.0;
        for (int64_t j = lo; j < hi; ++j) {
            out[j] = exp(x[j] - m2); /* f(x2) */
            l2 += out[j];
        }
        /* merge (m_run, l_run, f_run = out[0, lo)) with (m2, l2, f2 = out[lo, hi)) */
        const double m = m_run > m2 ? m_run : m2;
        const double a1 = lo > 0 ? exp(m_run - m) : 0.0;
        const double a2 = exp(m2 - m);
        for (int64_t j = 0; j < lo; ++j)
            out[j] *= a1;
        for (int64_t j = lo; j < hi; ++j)
            out[j] *= a2;
        l_run = a1 * l_run + a2 * l2;
        m_run = m;
        lo = hi;
    }
    for (int64_t j = 0; j < n; ++j)
        out[j] /= l_run;
    if (m_out)
        *m_out = m_run;
    if (l_out)
        *l_out = l_run;
    return ORACLE_OK;
}

/*
 * O and LSE of the requested rows by the block-wise online loop
 * ("FlashAttention", compassingai, section 3, online softmax listing): keys
 * are visited in blocks of bc; per block
 *   S = scores of the block, m_new = max(m, rowmax S), P = exp(S - m_new),
 *   l = exp(m - m_new) l + rowsum P, O = exp(m - m_new) O + P V, m = m_new,
 * and at the end O / l (the merge equations' final normalisation) and
 * LSE = m + log l.  Single-threaded; used only to pin the definition.
 */
int oracle_attn_online(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const int64_t *cu_seqlens, int64_t nseq, int H, int d,
                       double scale, int causal, const int64_t *rows, int64_t nrows,
                       int64_t bc, double *o, double *lse)
{
    int st = check_common(q, k, v, cu_seqlens, nseq, H, d, scale);
    if (st != ORACLE_OK || bc <= 0 || nrows < 0 || (nrows > 0 && (!rows || !o || !lse)))
        return ORACLE_EINVAL;
    double *sblk = (double *)malloc(sizeof(double) * (size_t)bc);
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    if (!sblk || !acc) {
        free(sblk);
        free(acc);
        return ORACLE_ENOMEM;
    }
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t s = rows[3 * r], hh = rows[3 * r + 1], i = rows[3 * r + 2];
        if (s < 0 || s >= nseq || hh < 0 || hh >= H) {
            st = ORACLE_EINVAL;
            break;
        }
        const int64_t base = cu_seqlens[s], L = cu_seqlens[s + 1] - base;
        if (i < 0 || i >= L) {
            st = ORACLE_EINVAL;
            break;
        }
        const int64_t nvis = causal ? i + 1 : L;
        const uint16_t *qi = q + ((base + i) * H + hh) * (int64_t)d;
        double m = -INFINITY, l = 0.0;
        for (int c = 0; c < d; ++c)
            acc[c] = 0.0;
        for (int64_t j0 = 0; j0 < nvis; j0 += bc) {
            const int64_t nb = nvis - j0 < bc ? nvis - j0 : bc;
            double bmax = -INFINITY;
            for (int64_t jj = 0; jj < nb; ++jj) {
                const uint16_t *kj = k + ((base + j0 + jj) * H + hh) * (int64_t)d;
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += widen_bf16(qi[c]) * widen_bf16(kj[c]);
                sblk[jj] = scale * dot;
                if (sblk[jj] > bmax)
                    bmax = sblk[jj];
            }
            const double m_new = m > bmax ? m : bmax;
            const double alpha = exp(m - m_new); /* 0 on the first block (m = -inf) */
            double rowsum = 0.0;
            for (int c = 0; c < d; ++c)
                acc[c] *= alpha;
            for (int64_t jj = 0; jj < nb; ++jj) {
                const double p = exp(sblk[jj] - m_new);
                rowsum += p;
                const uint16_t *vj = v + ((base + j0 + jj) * H + hh) * (int64_t)d;
                for (int c = 0; c < d; ++c)
                    acc[c] += p * widen_bf16(vj[c]);
            }
            l = alpha * l + rowsum;
            m = m_new;
        }
        for (int c = 0; c < d; ++c)
            o[r * d + c] = acc[c] / l;
        lse[r] = m + log(l);
    }
    free(sblk);
    free(acc);
    return st;
}

/* ------------------------------------------------------------- backward -- */

typedef struct {
    const uint16_t *q, *k, *v, *dout;
    int64_t base, L;
    int H, h, d;
    double scale;
    int causal;
    int64_t wl, wr; /* window: i - wl <= j <= i + wr; negative = unbounded */
    int64_t begin, end; /* query rows of this worker */
    double *dq;         /* [L][d], rows begin..end-1 written */
    double *dk, *dv;    /* [L][d] private accumulators of this worker */
    int status;
} bwd_job;

static void *bwd_worker(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    const int H = jb->H, h = jb->h, d = jb->d;
    const int64_t L = jb->L, base = jb->base;
    double *p = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double *qf = (double *)malloc(sizeof(double) * (size_t)d);
    double *dorow = (double *)malloc(sizeof(double) * (size_t)d);
    if (!p || !dp || !qf || !dorow) {
        free(p);
        free(dp);
        free(qf);
        free(dorow);
        jb->status = ORACLE_ENOMEM;
        return NULL;
    }
    for (int64_t i = jb->begin; i < jb->end; ++i) {
        /* visible keys [klo, khi), as in the forward */
        int64_t klo = 0, khi = jb->causal ? i + 1 : L;
        if (jb->wl >= 0 && i - jb->wl > klo)
            klo = i - jb->wl;
        if (jb->wr >= 0 && i + jb->wr + 1 < khi)
            khi = i + jb->wr + 1;
        const int64_t nvis = khi > klo ? khi - klo : 0;
        const uint16_t *qsrc = jb->q + ((base + i) * H + h) * (int64_t)d;
        const uint16_t *doi = jb->dout + ((base + i) * H + h) * (int64_t)d;
        for (int c = 0; c < d; ++c) {
            qf[c] = widen_bf16(qsrc[c]);
            dorow[c] = widen_bf16(doi[c]);
        }
        /* the forward's row: S_ij, m_i, l_i, P_ij */
        double m = -INFINITY;
        for (int64_t j = 0; j < nvis; ++j) {
            const uint16_t *kr = jb->k + ((base + klo + j) * H + h) * (int64_t)d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += qf[c] * widen_bf16(kr[c]);
            p[j] = jb->scale * acc;
            if (p[j] > m)
                m = p[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nvis; ++j)
            l += exp(p[j] - m);
        for (int64_t j = 0; j < nvis; ++j)
            p[j] = exp(p[j] - m) / l;
        /* dP_ij = <dO_i, v_j>;  D_i = sum_j P_ij dP_ij */
        double D = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            const uint16_t *vr = jb->v + ((base + klo + j) * H + h) * (int64_t)d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += dorow[c] * widen_bf16(vr[c]);
            dp[j] = acc;
            D += p[j] * dp[j];
        }
        /* dS_ij = P_ij (dP_ij - D_i); dQ_i, and this row's share of dK_j, dV_j */
        double *dqi = jb->dq + i * (int64_t)d;
        for (int c = 0; c < d; ++c)
            dqi[c] = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            const double ds = p[j] * (dp[j] - D);
            const uint16_t *kr = jb->k + ((base + klo + j) * H + h) * (int64_t)d;
            double *dkr = jb->dk + (klo + j) * (int64_t)d;
            double *dvr = jb->dv + (klo + j) * (int64_t)d;
            for (int c = 0; c < d; ++c) {
                dqi[c] += jb->scale * ds * widen_bf16(kr[c]);
                dkr[c] += jb->scale * ds * qf[c];
                dvr[c] += p[j] * dorow[c];
            }
        }
    }
    free(p);
    free(dp);
    free(qf);
    free(dorow);
    return NULL;
}

/*
 * dQ, dK, dV of the listed (sequence, head) pairs, by the chain rule written
 * out above.  pairs is [npairs][2] = (seq, head); the outputs hold, pair after
 * pair, the L_s rows of that pair ([sum_p L_{s_p}][d] each, fp64).  dout is
 * the upstream gradient dO in the layout of q.  nthreads <= 0 uses every CPU
 * of the affinity mask (the query rows of a pair are split among the threads;
 * each keeps its own dK, dV sums, added up at the end).  Returns 0 or a
 * negative code.
 */
int oracle_attn_bwd_window(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const uint16_t *dout, const int64_t *cu_seqlens, int64_t nseq, int H,
                           int d, double scale, int causal, int64_t wl, int64_t wr,
                           const int64_t *pairs, int64_t npairs, double *dq, double *dk,
                           double *dv, int nthreads, int *threads_used)
{
    int st = check_common(q, k, v, cu_seqlens, nseq, H, d, scale);
    if (st != ORACLE_OK || !dout || npairs < 0 || (npairs > 0 && (!pairs || !dq || !dk || !dv)))
        return ORACLE_EINVAL;
    for (int64_t pp = 0; pp < npairs; ++pp)
        if (pairs[2 * pp] < 0 || pairs[2 * pp] >= nseq || pairs[2 * pp + 1] < 0 ||
            pairs[2 * pp + 1] >= H)
            return ORACLE_EINVAL;
    const int ncpu = nthreads > 0 ? nthreads : oracle_cpu_count();
    int used_max = 1;
    int64_t out_row = 0;
    for (int64_t pp = 0; pp < npairs && st == ORACLE_OK; ++pp) {
        const int64_t s = pairs[2 * pp];
        const int h = (int)pairs[2 * pp + 1];
        const int64_t base = cu_seqlens[s], L = cu_seqlens[s + 1] - base;
        int nt = ncpu;
        if (nt > L)
            nt = L > 0 ? (int)L : 1;
        bwd_job *jobs = (bwd_job *)calloc((size_t)nt, sizeof(bwd_job));
        pthread_t *tid = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
        double *acc = (double *)calloc((size_t)nt * 2 * (size_t)(L > 0 ? L : 1) * (size_t)d,
                                       sizeof(double));
        if (!jobs || !tid || !acc) {
            free(jobs);
            free(tid);
            free(acc);
            return ORACLE_ENOMEM;
        }
        /* equal work per thread: causal row i costs i + 1 keys, so the split
           points of the rows go as L * sqrt(t / nt) */
        for (int t = 0; t < nt; ++t) {
            bwd_job *jb = &jobs[t];
            jb->q = q; jb->k = k; jb->v = v; jb->dout = dout;
            jb->base = base; jb->L = L;
            jb->H = H; jb->h = h; jb->d = d; jb->scale = scale; jb->causal = causal;
            jb->wl = wl; jb->wr = wr;
            if (causal) {
                jb->begin = t == 0 ? 0 : (int64_t)((double)L * sqrt((double)t / nt));
                jb->end = t == nt - 1 ? L : (int64_t)((double)L * sqrt((double)(t + 1) / nt));
            } else {
                jb->begin = L * t / nt;
                jb->end = L * (t + 1) / nt;
            }
            jb->dq = dq + out_row * (int64_t)d;
            jb->dk = acc + (size_t)t * 2 * (size_t)L * (size_t)d;
            jb->dv = jb->dk + (size_t)L * (size_t)d;
            jb->status = ORACLE_OK;
        }
        int started = 0;
        if (nt == 1) {
            bwd_worker(&jobs[0]);
            started = 1;
        } else {
            for (int t = 0; t < nt; ++t) {
                if (pthread_create(&tid[t], NULL, bwd_worker, &jobs[t]) != 0)
                    break;
                ++started;
            }
            for (int t = started; t < nt; ++t)
                bwd_worker(&jobs[t]);
            for (int t = 0; t < started; ++t)
                pthread_join(tid[t], NULL);
        }
        /* dK_j, dV_j = the sums over every worker's rows */
        for (int64_t x = 0; x < L * (int64_t)d; ++x) {
            double sk = 0.0, sv = 0.0;
            for (int t = 0; t < nt; ++t) {
                sk += jobs[t].dk[x];
                sv += jobs[t].dv[x];
            }
            dk[out_row * (int64_t)d + x] = sk;
            dv[out_row * (int64_t)d + x] = sv;
        }
        for (int t = 0; t < nt; ++t)
            if (jobs[t].status != ORACLE_OK)
                st = jobs[t].status;
        if (nt > 1 && started > used_max)
            used_max = started;
        out_row += L;
        free(jobs);
        free(tid);
        free(acc);
    }
    if (threads_used)
        *threads_used = used_max;
    return st;
}

/* ----------------------------------------------------------------- FP8 -- */

/*
 * e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinity,
 * the all-ones magnitude is NaN): the code of x rounded to nearest, ties to
 * even, with finite overflow saturating to +-448.  x is fp32; NaN maps to the
 * NaN code 0x7f.
 */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7f;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7e; /* largest finite: 1.75 * 2^8 */
    /* the value grid: subnormals m * 2^-9 (m < 8), normals (8 + m) * 2^(e - 10)
       for e in 1..15; find the spacing of the binade of a */
    int e;
    double spacing;
    if (a < 0.015625) { /* 2^-6: subnormal range */
        e = 0;
        spacing = 0.001953125; /* 2^-9 */
    } else {
        e = (int)floor(log2(a)) + 7; /* biased exponent of a's binade */
        if (ldexp(1.0, e - 7) > a)
            --e; /* guard the log2 rounding */
        else if (ldexp(1.0, e - 6) <= a)
            ++e;
        spacing = ldexp(1.0, e - 10);
    }
    const double q = a / spacing; /* exact: spacing is a power of two */
    double n = floor(q);
    const double frac = q - n;
    if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) == 1.0))
        n += 1.0;
    /* n counts spacings from 0: subnormal n in 0..8, normal n in 8..16 */
    if (e == 0) {
        if (n >= 8.0)
            return sign | 0x08; /* rounded up to the smallest normal 2^-6 */
        return sign | (uint8_t)n;
    }
    if (n >= 16.0) { /* rounded up into the next binade */
        ++e;
        n = 8.0;
        if (e > 15 || (e == 15 && n - 8.0 > 6.0))
            return sign | 0x7e;
    }
    if (e == 15 && n - 8.0 > 6.0)
        return sign | 0x7e;
    return sign | (uint8_t)((e << 3) | ((int)n - 8));
}

/* The value of an e4m3 code (NaN for 0x7f / 0xff). */
double oracle_e4m3_decode(uint8_t c)
{
    const int sign = c & 0x80, e = (c >> 3) & 0xf, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return sign ? -v : v;
}

/*
 * The unnormalised Hadamard transform of x[0..d) (d a power of two) times the
 * signs, in fp32: y = (x * signs) H_d, computed by butterflies over strides
 * 1, 2, 4, ..., d/2 (pairs (i, i + h) with bit h of i clear become
 * (a + b, a - b)).  signs may be NULL (all +1).
 */
void oracle_fwht_f32(float *x, int d, const int8_t *signs)
{
    if (signs)
        for (int c = 0; c < d; ++c)
            x[c] = signs[c] < 0 ? -x[c] : x[c];
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; ++i)
            if (!(i & h)) {
                const float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
}

/*
 * Block quantisation of a [tokens, H, d] bf16 tensor of B dense sequences of
 * length N: blocks of block_rows rows per sequence and head (the last block
 * pulled back to end at the sequence end, the rows it shares with the block
 * before it taking that block's codes; block_rows = 0: one block per
 * sequence and head), each row optionally rotated by oracle_fwht_f32 with
 * the given signs first (rotate != 0).  codes: [tokens, H, d] e4m3;
 * scales: [B][H][nblocks] fp32 = amax / 448 (1 when the block is all zero).
 */
int oracle_fp8_quantize(const uint16_t *x, int64_t B, int64_t N, int H, int d, int block_rows,
                        int rotate, const int8_t *signs, uint8_t *codes, float *scales)
{
    if (!x || !codes || !scales || B < 0 || N <= 0 || H <= 0 || d <= 0 || block_rows < 0 ||
        (d & (d - 1)))
        return ORACLE_EINVAL;
    const int64_t rows_per = block_rows > 0 ? block_rows : N;
    const int64_t nblk = (N + rows_per - 1) / rows_per;
    float *blk = (float *)malloc(sizeof(float) * (size_t)rows_per * (size_t)d);
    if (!blk)
        return ORACLE_ENOMEM;
    for (int64_t b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int64_t t = 0; t < nblk; ++t) {
                /* rows [r0, r0 + rows_per) of the block, pulled back at the end */
                int64_t r0 = t * rows_per;
                if (r0 + rows_per > N)
                    r0 = N - rows_per;
                const int64_t nominal = t * rows_per;
                float amax = 0.0f;
                for (int64_t r = 0; r < rows_per; ++r) {
                    float *y = blk + r * d;
                    const int64_t row = r0 + r;
                    for (int c = 0; c < d; ++c)
                        y[c] = row >= 0 ? (float)widen_bf16(x[((b * N + row) * H + h) * (int64_t)d + c])
                                        : 0.0f;
                    if (rotate)
                        oracle_fwht_f32(y, d, signs);
                    for (int c = 0; c < d; ++c)
                        if (fabsf(y[c]) > amax)
                            amax = fabsf(y[c]);
                }
                const float inv = amax > 0.0f ? 448.0f / amax : 1.0f;
                scales[(b * H + h) * nblk + t] = amax > 0.0f ? amax / 448.0f : 1.0f;
                for (int64_t r = 0; r < rows_per; ++r) {
                    const int64_t row = r0 + r;
                    if (row < nominal || row < 0)
                        continue; /* the previous block's row */
                    for (int c = 0; c < d; ++c)
                        codes[((b * N + row) * H + h) * (int64_t)d + c] =
                            oracle_e4m3_encode(blk[r * d + c] * inv);
                }
            }
    free(blk);
    return ORACLE_OK;
}

/*
 * Per-tensor e4m3 quantisation, the baseline the pages measure the FP8 path
 * against ("flash-attention-evolution" (letsgetai), FlashAttention-3
 * section, results: block quantisation with incoherent processing gives 2.6x
 * lower error than per-tensor FP8 attention).  Reading: one scale per tensor
 * and head (the largest |x| of head h over every token of x maps to 448), no
 * rotation, and the block quantiser's fp32 steps (448 / amax, x * (448 /
 * amax), e4m3 rounding).  x: [tokens, H, d] bf16; codes: [tokens, H, d];
 * scales: [H] = amax / 448 (1 when the head is all zero).
 */
int oracle_fp8_quantize_tensor(const uint16_t *x, int64_t tokens, int H, int d, uint8_t *codes,
                               float *scales)
{
    if (!x || !codes || !scales || tokens <= 0 || H <= 0 || d <= 0)
        return ORACLE_EINVAL;
    for (int h = 0; h < H; ++h) {
        float amax = 0.0f;
        for (int64_t t = 0; t < tokens; ++t)
            for (int c = 0; c < d; ++c) {
                const float y = (float)widen_bf16(x[(t * H + h) * (int64_t)d + c]);
                if (fabsf(y) > amax)
                    amax = fabsf(y);
            }
        const float inv_t = amax > 0.0f ? 448.0f / amax : 1.0f;
        scales[h] = amax > 0.0f ? amax / 448.0f : 1.0f;
        for (int64_t t = 0; t < tokens; ++t)
            for (int c = 0; c < d; ++c) {
                const int64_t at = (t * H + h) * (int64_t)d + c;
                codes[at] = oracle_e4m3_encode((float)widen_bf16(x[at]) * inv_t);
            }
    }
    return ORACLE_OK;
}

/*
 * O and LSE of the requested rows, by the plain definition, for fp64 inputs
 * in the packed layout [tokens, H, d] (e.g. dequantised FP8 values).
 * Single-threaded.
 */
int oracle_attn_rows_f64(const double *q, const double *k, const double *v,
                         const int64_t *cu_seqlens, int64_t nseq, int H, int d, double scale,
                         int causal, const int64_t *rows, int64_t nrows, double *o, double *lse)
{
    if (!q || !k || !v || !cu_seqlens || nseq < 0 || H <= 0 || d <= 0 || !isfinite(scale) ||
        nrows < 0 || (nrows > 0 && (!rows || !o || !lse)))
        return ORACLE_EINVAL;
    int64_t maxL = 0;
    for (int64_t s = 0; s < nseq; ++s)
        if (cu_seqlens[s + 1] - cu_seqlens[s] > maxL)
            maxL = cu_seqlens[s + 1] - cu_seqlens[s];
    double *sc = (double *)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1));
    if (!sc)
        return ORACLE_ENOMEM;
    int st = ORACLE_OK;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t s = rows[3 * r], hh = rows[3 * r + 1], i = rows[3 * r + 2];
        if (s < 0 || s >= nseq || hh < 0 || hh >= H) {
            st = ORACLE_EINVAL;
            break;
        }
        const int64_t base = cu_seqlens[s], L = cu_seqlens[s + 1] - base;
        if (i < 0 || i >= L) {
            st = ORACLE_EINVAL;
            break;
        }
        const int64_t nv = causal ? i + 1 : L;
        const double *qi = q + ((base + i) * H + hh) * (int64_t)d;
        double mx = -INFINITY;
        for (int64_t j = 0; j < nv; ++j) {
            const double *kk = k + ((base + j) * H + hh) * (int64_t)d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += qi[c] * kk[c];
            sc[j] = scale * acc;
            if (sc[j] > mx)
                mx = sc[j];
        }
        double z = 0.0;
        for (int64_t j = 0; j < nv; ++j)
            z += exp(sc[j] - mx);
        double *orow = o + r * (int64_t)d;
        for (int c = 0; c < d; ++c)
            orow[c] = 0.0;
        for (int64_t j = 0; j < nv; ++j) {
            const double w = exp(sc[j] - mx) / z;
            const double *vv = v + ((base + j) * H + hh) * (int64_t)d;
            for (int c = 0; c < d; ++c)
                orow[c] += w * vv[c];
        }
        lse[r] = mx + log(z);
    }
    free(sc);
    return st;
}

/* The gradients without a window (every visible key). */
int oracle_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    const uint16_t *dout, const int64_t *cu_seqlens, int64_t nseq, int H,
                    int d, double scale, int causal, const int64_t *pairs, int64_t npairs,
                    double *dq, double *dk, double *dv, int nthreads, int *threads_used)
{
    return oracle_attn_bwd_window(q, k, v, dout, cu_seqlens, nseq, H, d, scale, causal, -1, -1,
                                  pairs, npairs, dq, dk, dv, nthreads, threads_used);
}
