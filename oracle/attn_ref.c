/*
 * attn_ref.c -- the fp64 CPU oracle for the fused attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against.  Only the tests, the smoke
 * check and the CPU-baseline leg of the benchmark may load it; the product
 * library never links, includes or calls it, and it shares no code with it.
 *
 * What it computes (for every batch b, head h and query row i):
 *
 *   J(i)   = {0 .. N-1}              (full attention)
 *          = {0 .. i}                (causal: query i sees keys 0..i)
 *   s_ij   = scale * sum_k q_ik k_jk                      for j in J(i)
 *   m_i    = max_{j in J(i)} s_ij
 *   LSE_i  = m_i + ln sum_{j in J(i)} exp(s_ij - m_i)      (natural log)
 *   O_i    = sum_{j in J(i)} exp(s_ij - LSE_i) v_j
 *
 * Sources (the pages this follows):
 *   - LeetCUDA "flash_attn_mma_tiling_qk.cu", kernel body: the scores are the
 *     Q.K^T products multiplied by the softmax scale before the exponential
 *     ("P = Exp(S - m_new)" with S already scaled), the softmax is taken along
 *     the key axis and the final output is divided by the row sum
 *     ("O_output = (1/l_final) * O_final").
 *   - flash-attention "hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp", causal
 *     masking loop of CollectiveMainloopBwd::mma: a key column is masked when
 *     it lies past the query row (bottom-right alignment; with one sequence
 *     length for queries and keys this is "key j allowed iff j <= i"); and
 *     scale_apply_exp2 against the stored LSE, which shows the LSE is the
 *     log-normaliser of the *scaled* scores.
 *   - flash-attention "hopper/flash_fwd_kernel.h", consumer path: a row with
 *     no admissible key gets O = 0 and LSE = -inf (store_zero).
 *
 * The LSE is reported in natural-log units (the Hopper pages keep a base-2
 * copy for their backward pass; ln 2 times that is the same quantity).
 *
 * Two generalisations, both from the same backward page: grouped K/V heads
 * (query head h reads K/V head h / (H / H_kv): the page's
 * qhead_per_khead) and a local window (query i sees keys j with
 * i - window_left <= j <= i + window_right; a negative bound is unbounded:
 * the page's window_size_left / window_size_right and its Is_local mask).
 * With H_kv = H and both bounds negative they reduce to the definition above.
 *
 * FP8 inputs (attn_ref_fwd_fp8): E4M3 bytes times one descale factor per
 * tensor, decoded exactly here; then the same definition.
 *
 * Backward (attn_ref_bwd_u16, and attn_ref_bwd_qk_u16 for separate query and
 * key lengths, bottom-right aligned): the gradients dQ, dK, dV of the
 * definition above against dO, as the same backward page computes them (P,
 * dP, the row sums D_i = sum_j P_ij dP_ij, dS = P (dP - D)), in double.
 *
 * Variable-length batches (attn_ref_varlen_u16): sequences of different
 * lengths packed along the rows of [total][H][d] tensors, sequence b being
 * rows cu[b] .. cu[b+1]-1 -- the cu_seqlens mode of the Hopper pages.  Each
 * sequence is the definition above on its own rows, positions counted from
 * its first row.  attn_ref_varlen_qk_u16 generalises it to separate query
 * and key offsets and used lengths (cross-attention, a KV cache), with the
 * pages' bottom-right alignment of the masks.
 *
 * Inputs are the caller's 16-bit words (IEEE binary16 or bfloat16), widened
 * exactly to double here; every product, sum and exponential is in double.
 * The computation is the textbook two-pass softmax per row -- no tiling, no
 * online recurrence, no reordering beyond the definition above.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC attn_ref.c -o libattn_ref.so -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* 16-bit float decoding, written from the IEEE 754 binary16 and the   */
/* bfloat16 (upper half of binary32) bit layouts.                      */
/* ------------------------------------------------------------------ */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);            /* zero or subnormal */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(1024 + frac), expo - 25);
    }
    return sign ? -mag : mag;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 value. */
static double bf16_to_double(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

double attn_ref_widen(uint16_t bits, int is_bf16) {
    return is_bf16 ? bf16_to_double(bits) : half_to_double(bits);
}

int attn_ref_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* One query row against one (b,h) slice, all in double.                */
/*   q_row [d], kmat [N][d], vmat [N][d], scores: scratch of N doubles. */
/*   Admissible keys: j0 <= j < j1.                                     */
/* ------------------------------------------------------------------ */
static void attend_range(const double *q_row, const double *kmat,
                         const double *vmat, long d, long j0, long j1,
                         double scale, double *scores, double *o_row,
                         double *lse_out) {
    if (j1 <= j0) {                   /* no admissible key: O = 0, LSE = -inf */
        for (long c = 0; c < d; ++c) o_row[c] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    /* pass 1: scaled scores and their maximum */
    double m = -INFINITY;
    for (long j = j0; j < j1; ++j) {
        const double *k_row = kmat + j * d;
        double dot = 0.0;
        for (long c = 0; c < d; ++c) dot += q_row[c] * k_row[c];
        double s = scale * dot;
        scores[j] = s;
        if (s > m) m = s;
    }
    /* pass 2: log-normaliser */
    double sum = 0.0;
    for (long j = j0; j < j1; ++j) sum += exp(scores[j] - m);
    double lse = m + log(sum);
    /* pass 3: probability-weighted sum of value rows */
    for (long c = 0; c < d; ++c) o_row[c] = 0.0;
    for (long j = j0; j < j1; ++j) {
        double p = exp(scores[j] - lse);
        const double *v_row = vmat + j * d;
        for (long c = 0; c < d; ++c) o_row[c] += p * v_row[c];
    }
    *lse_out = lse;
}

/* Admissible keys of query i: [j0, j1). */
static void key_range(long N, long i, int causal, long wl, long wr,
                      long *j0, long *j1) {
    long lo = 0, hi = N;                          /* full attention */
    if (causal && i + 1 < hi) hi = i + 1;         /* keys 0..i */
    if (wl >= 0 && i - wl > lo) lo = i - wl;      /* keys >= i - wl */
    if (wr >= 0 && i + wr + 1 < hi) hi = i + wr + 1;  /* keys <= i + wr */
    *j0 = lo;
    *j1 = hi;
}

static void attend_row(const double *q_row, const double *kmat,
                       const double *vmat, long N, long d, long i,
                       double scale, int causal, double *scores,
                       double *o_row, double *lse_out) {
    long j0, j1;
    key_range(N, i, causal, -1, -1, &j0, &j1);
    attend_range(q_row, kmat, vmat, d, j0, j1, scale, scores, o_row, lse_out);
}

static void widen_slice(const uint16_t *src, double *dst, long count,
                        int is_bf16) {
    for (long t = 0; t < count; ++t) dst[t] = attn_ref_widen(src[t], is_bf16);
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/*
 * Full problem on 16-bit inputs.
 *   q, k, v : [B][H][N][d] 16-bit words; is_bf16 selects the format
 *   o       : [B][H][N][d] double (written)
 *   lse     : [B][H][N]    double (written)
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int attn_ref_fwd_u16(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int is_bf16, long B, long H, long N, long d, double scale,
                     int causal, double *o, double *lse, int nthreads) {
    if (!q || !k || !v || !o || !lse || B < 0 || H < 0 || N < 0 || d <= 0)
        return -1;
    set_threads(nthreads);
    long slice = N * d;
    double *qd = (double *)malloc(sizeof(double) * (size_t)(slice > 0 ? slice : 1));
    double *kd = (double *)malloc(sizeof(double) * (size_t)(slice > 0 ? slice : 1));
    double *vd = (double *)malloc(sizeof(double) * (size_t)(slice > 0 ? slice : 1));
    if (!qd || !kd || !vd) { free(qd); free(kd); free(vd); return -1; }
    int rc = 0;
    for (long bh = 0; bh < B * H && rc == 0; ++bh) {
        widen_slice(q + bh * slice, qd, slice, is_bf16);
        widen_slice(k + bh * slice, kd, slice, is_bf16);
        widen_slice(v + bh * slice, vd, slice, is_bf16);
#pragma omp parallel
        {
            double *scores = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
            if (!scores) {
#pragma omp atomic write
                rc = -1;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (long i = 0; i < N; ++i)
                    attend_row(qd + i * d, kd, vd, N, d, i, scale, causal,
                               scores, o + (bh * N + i) * d, lse + bh * N + i);
                free(scores);
            }
        }
    }
    free(qd); free(kd); free(vd);
    return rc;
}

/*
 * Selected rows only, for problems too large to evaluate in full.
 *   rows    : n_rows triples (b, h, i), row-major [n_rows][3]
 *   o_rows  : [n_rows][d] double (written);  lse_rows: [n_rows] (written)
 * The K/V slice of each (b,h) is widened once per call and shared by every
 * requested row of that head.  Returns 0, or -1 on bad arguments.
 */
int attn_ref_rows_u16(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      int is_bf16, long B, long H, long N, long d,
                      double scale, int causal, const long *rows, long n_rows,
                      double *o_rows, double *lse_rows, int nthreads) {
    if (!q || !k || !v || !rows || !o_rows || !lse_rows || N <= 0 || d <= 0)
        return -1;
    for (long r = 0; r < n_rows; ++r) {
        long b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= N) return -1;
    }
    set_threads(nthreads);
    long slice = N * d;
    double *kd = (double *)malloc(sizeof(double) * (size_t)slice);
    double *vd = (double *)malloc(sizeof(double) * (size_t)slice);
    char *done = (char *)calloc((size_t)(n_rows > 0 ? n_rows : 1), 1);
    if (!kd || !vd || !done) { free(kd); free(vd); free(done); return -1; }
    int rc = 0;
    for (long r0 = 0; r0 < n_rows && rc == 0; ++r0) {
        if (done[r0]) continue;
        long bh = rows[3 * r0] * H + rows[3 * r0 + 1];
        widen_slice(k + bh * slice, kd, slice, is_bf16);
        widen_slice(v + bh * slice, vd, slice, is_bf16);
#pragma omp parallel
        {
            double *scores = (double *)malloc(sizeof(double) * (size_t)N);
            double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
            if (!scores || !qrow) {
#pragma omp atomic write
                rc = -1;
            } else {
#pragma omp for schedule(dynamic, 1)
                for (long r = r0; r < n_rows; ++r) {
                    if (done[r] || rows[3 * r] * H + rows[3 * r + 1] != bh)
                        continue;
                    long i = rows[3 * r + 2];
                    widen_slice(q + (bh * N + i) * d, qrow, d, is_bf16);
                    attend_row(qrow, kd, vd, N, d, i, scale, causal, scores,
                               o_rows + r * d, lse_rows + r);
                }
            }
            free(scores); free(qrow);
        }
        for (long r = r0; r < n_rows; ++r)
            if (rows[3 * r] * H + rows[3 * r + 1] == bh) done[r] = 1;
    }
    free(kd); free(vd); free(done);
    return rc;
}

/*
 * Same definition on double inputs (q, k, v as [B][H][N][d] doubles), for
 * checks whose inputs are not 16-bit representable.
 */
int attn_ref_fwd_f64(const double *q, const double *k, const double *v,
                     long B, long H, long N, long d, double scale, int causal,
                     double *o, double *lse, int nthreads) {
    if (!q || !k || !v || !o || !lse || B < 0 || H < 0 || N < 0 || d <= 0)
        return -1;
    set_threads(nthreads);
    long slice = N * d;
    int rc = 0;
    for (long bh = 0; bh < B * H && rc == 0; ++bh) {
#pragma omp parallel
        {
            double *scores = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
            if (!scores) {
#pragma omp atomic write
                rc = -1;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (long i = 0; i < N; ++i)
                    attend_row(q + bh * slice + i * d, k + bh * slice,
                               v + bh * slice, N, d, i, scale, causal, scores,
                               o + (bh * N + i) * d, lse + bh * N + i);
                free(scores);
            }
        }
    }
    return rc;
}

/*
 * Grouped heads and a local window.
 *   q, o : [B][H][N][d];  k, v : [B][H_kv][N][d];  lse : [B][H][N]
 *   H must be a multiple of H_kv; window bounds < 0 mean unbounded.
 * Full evaluation (_fwd) or listed (b, h, i) rows (_rows), as above.
 */
int attn_ref_fwd_u16_ex(const uint16_t *q, const uint16_t *k,
                        const uint16_t *v, int is_bf16, long B, long H,
                        long H_kv, long N, long d, double scale, int causal,
                        long wl, long wr, double *o, double *lse,
                        int nthreads) {
    if (!q || !k || !v || !o || !lse || B < 0 || H <= 0 || H_kv <= 0 ||
        H % H_kv != 0 || N < 0 || d <= 0)
        return -1;
    set_threads(nthreads);
    long slice = N * d, group = H / H_kv;
    double *qd = (double *)malloc(sizeof(double) * (size_t)(slice > 0 ? slice : 1));
    double *kd = (double *)malloc(sizeof(double) * (size_t)(slice > 0 ? slice : 1));
    double *vd = (double *)malloc(sizeof(double) * (size_t)(slice > 0 ? slice : 1));
    if (!qd || !kd || !vd) { free(qd); free(kd); free(vd); return -1; }
    int rc = 0;
    for (long b = 0; b < B && rc == 0; ++b) {
        for (long h = 0; h < H && rc == 0; ++h) {
            long bh = b * H + h, bkv = b * H_kv + h / group;
            widen_slice(q + bh * slice, qd, slice, is_bf16);
            widen_slice(k + bkv * slice, kd, slice, is_bf16);
            widen_slice(v + bkv * slice, vd, slice, is_bf16);
#pragma omp parallel
            {
                double *scores = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
                if (!scores) {
#pragma omp atomic write
                    rc = -1;
                } else {
#pragma omp for schedule(dynamic, 4)
                    for (long i = 0; i < N; ++i) {
                        long j0, j1;
                        key_range(N, i, causal, wl, wr, &j0, &j1);
                        attend_range(qd + i * d, kd, vd, d, j0, j1, scale, scores,
                                     o + (bh * N + i) * d, lse + bh * N + i);
                    }
                    free(scores);
                }
            }
        }
    }
    free(qd); free(kd); free(vd);
    return rc;
}

int attn_ref_rows_u16_ex(const uint16_t *q, const uint16_t *k,
                         const uint16_t *v, int is_bf16, long B, long H,
                         long H_kv, long N, long d, double scale, int causal,
                         long wl, long wr, const long *rows, long n_rows,
                         double *o_rows, double *lse_rows, int nthreads) {
    if (!q || !k || !v || !rows || !o_rows || !lse_rows || N <= 0 || d <= 0 ||
        H <= 0 || H_kv <= 0 || H % H_kv != 0)
        return -1;
    for (long r = 0; r < n_rows; ++r) {
        long b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= N) return -1;
    }
    set_threads(nthreads);
    long slice = N * d, group = H / H_kv;
    double *kd = (double *)malloc(sizeof(double) * (size_t)slice);
    double *vd = (double *)malloc(sizeof(double) * (size_t)slice);
    char *done = (char *)calloc((size_t)(n_rows > 0 ? n_rows : 1), 1);
    if (!kd || !vd || !done) { free(kd); free(vd); free(done); return -1; }
    int rc = 0;
    for (long r0 = 0; r0 < n_rows && rc == 0; ++r0) {
        if (done[r0]) continue;
        long bkv = rows[3 * r0] * H_kv + rows[3 * r0 + 1] / group;
        widen_slice(k + bkv * slice, kd, slice, is_bf16);
        widen_slice(v + bkv * slice, vd, slice, is_bf16);
#pragma omp parallel
        {
            double *scores = (double *)malloc(sizeof(double) * (size_t)N);
            double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
            if (!scores || !qrow) {
#pragma omp atomic write
                rc = -1;
            } else {
#pragma omp for schedule(dynamic, 1)
                for (long r = r0; r < n_rows; ++r) {
                    long b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
                    if (done[r] || b * H_kv + h / group != bkv) continue;
                    long j0, j1;
                    key_range(N, i, causal, wl, wr, &j0, &j1);
                    widen_slice(q + ((b * H + h) * N + i) * d, qrow, d, is_bf16);
                    attend_range(qrow, kd, vd, d, j0, j1, scale, scores,
                                 o_rows + r * d, lse_rows + r);
                }
            }
            free(scores); free(qrow);
        }
        for (long r = r0; r < n_rows; ++r)
            if (rows[3 * r] * H_kv + rows[3 * r + 1] / group == bkv) done[r] = 1;
    }
    free(kd); free(vd); free(done);
    return rc;
}

/*
 * Variable-length batch with separate query and key sequences -- the
 * cu_seqlens_q / cu_seqlens_k / seqused_q / seqused_k arguments of
 * flash-attention "hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp"
 * (CollectiveMainloopBwd::Arguments, get_seqlen_q / get_seqlen_k) and the
 * variable-length mode of "hopper/flash_fwd_kernel.h":
 *   q, o : [total_q][H][d];  k, v : [total_k][H_kv][d];  lse : [H][total_q]
 *   sequence b has n_q = used_q[b] queries (cu_q[b+1] - cu_q[b] when used_q
 *   is NULL) in rows cu_q[b] .. cu_q[b] + n_q - 1, and n_k = used_k[b] keys
 *   (cu_k[b+1] - cu_k[b] when used_k is NULL) in rows cu_k[b] ..
 *   cu_k[b] + n_k - 1.
 * Masks are bottom-right aligned, as on the backward page (its causal and
 * local masking loops shift the query row by seqlen_k - seqlen_q): query i
 * of the sequence sits at key position i + n_k - n_q, so causal keeps keys
 * j <= i + n_k - n_q and the window keeps i + n_k - n_q - wl <= j <=
 * i + n_k - n_q + wr.  A query with no admissible key gets O = 0 and
 * LSE = -inf (the forward page's store_zero).  Rows of o / lse outside every
 * sequence's used query rows are not written.  Returns 0, or -1 on bad
 * arguments (offsets not non-decreasing within [0, total], a used length
 * beyond its sequence's rows) or allocation failure.
 */
static void gather_rows(const uint16_t *src, long stride, long rows, long d,
                        double *dst, int is_bf16) {
    for (long r = 0; r < rows; ++r)
        widen_slice(src + r * stride, dst + r * d, d, is_bf16);
}

/* Rows and used length of sequence b under offsets cu and lengths used. */
static int seq_rows(const long *cu, const long *used, long b, long total,
                    long *first, long *n) {
    if (cu[b] < 0 || cu[b + 1] < cu[b] || cu[b + 1] > total) return -1;
    *first = cu[b];
    *n = used ? used[b] : cu[b + 1] - cu[b];
    if (*n < 0 || *n > cu[b + 1] - cu[b]) return -1;
    return 0;
}

int attn_ref_varlen_qk_u16(const uint16_t *q, const uint16_t *k,
                           const uint16_t *v, int is_bf16, const long *cu_q,
                           const long *cu_k, const long *used_q,
                           const long *used_k, long batch, long total_q,
                           long total_k, long H, long H_kv, long d,
                           double scale, int causal, long wl, long wr,
                           double *o, double *lse, int nthreads) {
    if (!q || !k || !v || !cu_q || !cu_k || !o || !lse || batch < 0 ||
        total_q < 0 || total_k < 0 || H <= 0 || H_kv <= 0 || H % H_kv != 0 ||
        d <= 0)
        return -1;
    long longest = 1;
    for (long b = 0; b < batch; ++b) {
        long q0, nq, k0, nk;
        if (seq_rows(cu_q, used_q, b, total_q, &q0, &nq) != 0 ||
            seq_rows(cu_k, used_k, b, total_k, &k0, &nk) != 0)
            return -1;
        if (nq > longest) longest = nq;
        if (nk > longest) longest = nk;
    }
    set_threads(nthreads);
    long group = H / H_kv;
    double *qd = (double *)malloc(sizeof(double) * (size_t)(longest * d));
    double *kd = (double *)malloc(sizeof(double) * (size_t)(longest * d));
    double *vd = (double *)malloc(sizeof(double) * (size_t)(longest * d));
    if (!qd || !kd || !vd) { free(qd); free(kd); free(vd); return -1; }
    int rc = 0;
    for (long b = 0; b < batch && rc == 0; ++b) {
        long q0, nq, k0, nk;
        seq_rows(cu_q, used_q, b, total_q, &q0, &nq);
        seq_rows(cu_k, used_k, b, total_k, &k0, &nk);
        if (nq == 0) continue;
        for (long h = 0; h < H && rc == 0; ++h) {
            long hk = h / group;
            gather_rows(q + (q0 * H + h) * d, H * d, nq, d, qd, is_bf16);
            gather_rows(k + (k0 * H_kv + hk) * d, H_kv * d, nk, d, kd, is_bf16);
            gather_rows(v + (k0 * H_kv + hk) * d, H_kv * d, nk, d, vd, is_bf16);
#pragma omp parallel
            {
                double *scores = (double *)malloc(sizeof(double) * (size_t)longest);
                if (!scores) {
#pragma omp atomic write
                    rc = -1;
                } else {
#pragma omp for schedule(dynamic, 4)
                    for (long i = 0; i < nq; ++i) {
                        long j0, j1;
                        /* bottom-right: query i at key position i + nk - nq */
                        key_range(nk, i + nk - nq, causal, wl, wr, &j0, &j1);
                        attend_range(qd + i * d, kd, vd, d, j0, j1, scale, scores,
                                     o + ((q0 + i) * H + h) * d,
                                     lse + h * total_q + q0 + i);
                    }
                    free(scores);
                }
            }
        }
    }
    free(qd); free(kd); free(vd);
    return rc;
}

/*
 * Variable-length batch of self-attention sequences: one set of offsets for
 * queries and keys (sequence b is rows cu[b] .. cu[b+1]-1 of q, k, v, o;
 * lse [H][total]), i.e. attn_ref_varlen_qk_u16 with cu_k = cu_q and no used
 * lengths, where the bottom-right alignment is the plain diagonal.
 */
int attn_ref_varlen_u16(const uint16_t *q, const uint16_t *k,
                        const uint16_t *v, int is_bf16, const long *cu,
                        long batch, long total, long H, long H_kv, long d,
                        double scale, int causal, long wl, long wr, double *o,
                        double *lse, int nthreads) {
    return attn_ref_varlen_qk_u16(q, k, v, is_bf16, cu, cu, NULL, NULL, batch,
                                  total, total, H, H_kv, d, scale, causal, wl,
                                  wr, o, lse, nthreads);
}

/*
 * Backward pass: the gradients of O = attention(Q, K, V) against dO, as
 * flash-attention "hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp"
 * (CollectiveMainloopBwd::mma) computes them, written from the definition:
 *
 *   P_ij  = exp(s_ij - LSE_i)  for j in J(i), 0 otherwise
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_j P_ij dP_ij                 (the page's dPsum)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_i dS_ij q_i
 *
 * with s_ij and LSE_i those of the forward definition above (recomputed here
 * in double from the 16-bit inputs).  With grouped heads, dK and dV of a K/V
 * head sum over the query heads that read it.
 *
 * attn_ref_bwd_qk_u16 takes Nq query rows and Nk key rows per (b, h), with
 * the masks aligned bottom-right as the backward page's masking loops shift
 * them by seqlen_k - seqlen_q (query i at key position i + Nk - Nq, as the
 * forward's attn_ref_varlen_qk_u16); a query row that sees no key has P = 0
 * in every column, so its dQ row is 0 and it adds nothing to dK, dV.
 *   q, dout, dq : [B][H][Nq][d];  k, v, dk, dv : [B][H_kv][Nk][d]
 * Pass 1 (rows i in parallel): LSE_i, D_i and dQ_i.  Pass 2 (keys j in
 * parallel): dK_j and dV_j from the stored LSE_i and D_i.
 */
int attn_ref_bwd_qk_u16(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const uint16_t *dout, int is_bf16, long B, long H, long H_kv,
                        long Nq, long Nk, long d, double scale, int causal, long wl,
                        long wr, double *dq, double *dk, double *dv, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv || B < 0 || H <= 0 ||
        H_kv <= 0 || H % H_kv != 0 || Nq < 0 || Nk < 0 || d <= 0)
        return -1;
    set_threads(nthreads);
    long qslice = Nq * d, kslice = Nk * d, group = H / H_kv;
    long qcap = qslice > 0 ? qslice : 1, kcap = kslice > 0 ? kslice : 1;
    double *kd = (double *)malloc(sizeof(double) * (size_t)kcap);
    double *vd = (double *)malloc(sizeof(double) * (size_t)kcap);
    double *qd = (double *)malloc(sizeof(double) * (size_t)(qcap * group));
    double *dod = (double *)malloc(sizeof(double) * (size_t)(qcap * group));
    double *lse = (double *)malloc(sizeof(double) * (size_t)((Nq > 0 ? Nq : 1) * group));
    double *dsum = (double *)malloc(sizeof(double) * (size_t)((Nq > 0 ? Nq : 1) * group));
    if (!kd || !vd || !qd || !dod || !lse || !dsum) {
        free(kd); free(vd); free(qd); free(dod); free(lse); free(dsum);
        return -1;
    }
    const long shift = Nk - Nq;  /* key position of query row i: i + shift */
    int rc = 0;
    for (long b = 0; b < B && rc == 0; ++b) {
        for (long hk = 0; hk < H_kv && rc == 0; ++hk) {
            long bkv = b * H_kv + hk;
            widen_slice(k + bkv * kslice, kd, kslice, is_bf16);
            widen_slice(v + bkv * kslice, vd, kslice, is_bf16);
            for (long g = 0; g < group; ++g) {
                long bh = b * H + hk * group + g;
                widen_slice(q + bh * qslice, qd + g * qslice, qslice, is_bf16);
                widen_slice(dout + bh * qslice, dod + g * qslice, qslice, is_bf16);
            }
            /* pass 1: per query row i of every head of the group */
#pragma omp parallel
            {
                double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
                if (!s) {
#pragma omp atomic write
                    rc = -1;
                } else {
#pragma omp for schedule(dynamic, 4)
                    for (long gi = 0; gi < group * Nq; ++gi) {
                        long g = gi / Nq, i = gi % Nq;
                        const double *qi = qd + g * qslice + i * d;
                        const double *doi = dod + g * qslice + i * d;
                        double *dqi = dq + ((b * H + hk * group + g) * Nq + i) * d;
                        long j0, j1;
                        key_range(Nk, i + shift, causal, wl, wr, &j0, &j1);
                        for (long c = 0; c < d; ++c) dqi[c] = 0.0;
                        if (j1 <= j0) {
                            lse[gi] = -INFINITY;
                            dsum[gi] = 0.0;
                            continue;
                        }
                        double m = -INFINITY;
                        for (long j = j0; j < j1; ++j) {
                            double dot = 0.0;
                            for (long c = 0; c < d; ++c) dot += qi[c] * kd[j * d + c];
                            s[j] = scale * dot;
                            if (s[j] > m) m = s[j];
                        }
                        double sum = 0.0;
                        for (long j = j0; j < j1; ++j) sum += exp(s[j] - m);
                        double l = m + log(sum);
                        double dsi = 0.0;   /* D_i = sum_j P_ij dP_ij */
                        for (long j = j0; j < j1; ++j) {
                            double dp = 0.0;
                            for (long c = 0; c < d; ++c) dp += doi[c] * vd[j * d + c];
                            dsi += exp(s[j] - l) * dp;
                        }
                        for (long j = j0; j < j1; ++j) {
                            double dp = 0.0;
                            for (long c = 0; c < d; ++c) dp += doi[c] * vd[j * d + c];
                            double ds = exp(s[j] - l) * (dp - dsi);
                            for (long c = 0; c < d; ++c) dqi[c] += scale * ds * kd[j * d + c];
                        }
                        lse[gi] = l;
                        dsum[gi] = dsi;
                    }
                    free(s);
                }
            }
            if (rc != 0) break;
            /* pass 2: per key row j, summed over the group's query rows */
#pragma omp parallel for schedule(dynamic, 4)
            for (long j = 0; j < Nk; ++j) {
                double *dkj = dk + (bkv * Nk + j) * d;
                double *dvj = dv + (bkv * Nk + j) * d;
                for (long c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
                for (long gi = 0; gi < group * Nq; ++gi) {
                    long g = gi / Nq, i = gi % Nq;
                    long j0, j1;
                    key_range(Nk, i + shift, causal, wl, wr, &j0, &j1);
                    if (j < j0 || j >= j1) continue;
                    const double *qi = qd + g * qslice + i * d;
                    const double *doi = dod + g * qslice + i * d;
                    double dot = 0.0, dp = 0.0;
                    for (long c = 0; c < d; ++c) {
                        dot += qi[c] * kd[j * d + c];
                        dp += doi[c] * vd[j * d + c];
                    }
                    double p = exp(scale * dot - lse[gi]);
                    double ds = p * (dp - dsum[gi]);
                    for (long c = 0; c < d; ++c) {
                        dvj[c] += p * doi[c];
                        dkj[c] += scale * ds * qi[c];
                    }
                }
            }
        }
    }
    free(kd); free(vd); free(qd); free(dod); free(lse); free(dsum);
    return rc;
}

/* Equal query and key lengths (the bottom-right alignment is the plain
 * diagonal):  q, dout, dq : [B][H][N][d];  k, v, dk, dv : [B][H_kv][N][d]. */
int attn_ref_bwd_u16(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const uint16_t *dout, int is_bf16, long B, long H, long H_kv,
                     long N, long d, double scale, int causal, long wl, long wr,
                     double *dq, double *dk, double *dv, int nthreads) {
    return attn_ref_bwd_qk_u16(q, k, v, dout, is_bf16, B, H, H_kv, N, N, d, scale, causal,
                               wl, wr, dq, dk, dv, nthreads);
}

/*
 * FP8 forward: Q, K, V given as OCP FP8 E4M3 bytes (1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent 0 is subnormal, m/8 * 2^-6; the
 * all-ones code S.1111.111 is NaN and there is no infinity) with one
 * descale factor per tensor, as flash-attention "hopper/flash_fwd_kernel.h"
 * takes them (descale_q/k/v: the stored values times the descale are the
 * real inputs).  The result is the definition above on q = dq * Q8,
 * k = dk * K8, v = dv * V8:
 *   q, k, v : [B][H or H_kv][N][d] bytes;  o : [B][H][N][d];  lse : [B][H][N]
 */
static double e4m3_to_double(uint8_t b) {
    int sign = (b >> 7) & 1, expo = (b >> 3) & 0xF, mant = b & 7;
    double mag;
    if (expo == 0xF && mant == 7) return NAN;
    if (expo == 0) mag = ldexp((double)mant, -9);          /* (m/8) 2^-6 */
    else mag = ldexp(8.0 + mant, expo - 10);               /* (1+m/8) 2^(e-7) */
    return sign ? -mag : mag;
}

double attn_ref_e4m3(uint8_t code) { return e4m3_to_double(code); }

int attn_ref_fwd_fp8(const uint8_t *q, const uint8_t *k, const uint8_t *v,
                     long B, long H, long H_kv, long N, long d, double scale,
                     double dq, double dk, double dv, int causal, long wl, long wr,
                     double *o, double *lse, int nthreads) {
    if (!q || !k || !v || !o || !lse || B < 0 || H <= 0 || H_kv <= 0 ||
        H % H_kv != 0 || N < 0 || d <= 0)
        return -1;
    set_threads(nthreads);
    long slice = N * d, group = H / H_kv, cap = slice > 0 ? slice : 1;
    double *qd = (double *)malloc(sizeof(double) * (size_t)cap);
    double *kd = (double *)malloc(sizeof(double) * (size_t)cap);
    double *vd = (double *)malloc(sizeof(double) * (size_t)cap);
    if (!qd || !kd || !vd) { free(qd); free(kd); free(vd); return -1; }
    int rc = 0;
    for (long b = 0; b < B && rc == 0; ++b) {
        for (long h = 0; h < H && rc == 0; ++h) {
            long bh = b * H + h, bkv = b * H_kv + h / group;
            for (long t = 0; t < slice; ++t) {
                qd[t] = dq * e4m3_to_double(q[bh * slice + t]);
                kd[t] = dk * e4m3_to_double(k[bkv * slice + t]);
                vd[t] = dv * e4m3_to_double(v[bkv * slice + t]);
            }
#pragma omp parallel
            {
                double *scores = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
                if (!scores) {
#pragma omp atomic write
                    rc = -1;
                } else {
#pragma omp for schedule(dynamic, 4)
                    for (long i = 0; i < N; ++i) {
                        long j0, j1;
                        key_range(N, i, causal, wl, wr, &j0, &j1);
                        attend_range(qd + i * d, kd, vd, d, j0, j1, scale, scores,
                                     o + (bh * N + i) * d, lse + bh * N + i);
                    }
                    free(scores);
                }
            }
        }
    }
    free(qd); free(kd); free(vd);
    return rc;
}
