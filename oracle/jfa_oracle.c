/*
 * jfa_oracle.c -- plain fp64 CPU oracle for Jagged Flash Attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or table with the CUDA library.
 *
 * What it computes (the plain definition; FlashAttention reaches the same
 * result up to rounding order):
 *
 *   The pages say the kernel "applies the FlashAttention algorithm directly"
 *   to packed Q/K/V whose sequence boundaries live in an offsets tensor
 *   (Meta's TLX Jagged Flash Attention Beats FA4 on Blackwell With 3x Less
 *   Code, section "Why attention in GEM needed a rewrite"; Meta's 3.2K-line
 *   Triton kernel outruns FlashAttention-4 on jagged Blackwell attention,
 *   third paragraph).  So for every sequence b (keys j in
 *   [offsets[b], offsets[b+1])) and head h, independently:
 *
 *     s_ij  = scale * <q_i, k_j>            (-inf where causal and j > i)
 *     LSE_i = ln sum_j exp(s_ij)           (natural log of scaled logits)
 *     P_ij  = exp(s_ij - LSE_i)
 *     O_i   = sum_j P_ij v_j
 *
 *   Backward, given dO:
 *     dP_ij = <dO_i, v_j>
 *     Delta_i = sum_j P_ij dP_ij
 *     dS_ij = P_ij (dP_ij - Delta_i)
 *     dV_j  = sum_i P_ij dO_i
 *     dK_j  = scale * sum_i dS_ij q_i
 *     dQ_i  = scale * sum_j dS_ij k_j
 *
 *   Broadcast-Q mode: one dense Q [Lq,H,D] is shared by every sequence and
 *   dQ is summed over the whole batch (Meta's 3.2K-line Triton kernel ...,
 *   second paragraph; Meta's TLX Jagged Flash Attention ..., section
 *   "Optimizations layered on top").  Jagged (self-attention) mode: Q is
 *   packed like K/V and sequence b's queries are rows offsets[b]..; causal
 *   is top-left aligned inside a sequence (query i sees keys j <= i).
 *
 * Readings the pages leave open (stated once here, applied below):
 *   - LSE is the natural log of the scaled logits; an empty row (no visible
 *     key) has LSE = -inf and O = 0 and contributes no gradient.
 *   - Layouts: Q [Lq,H,D] (broadcast) or [N,H,D]; K,V [N,H,D];
 *     O [B,Lq,H,D] or [N,H,D]; LSE [B,H,Lq] or [H,N]; dQ like Q.
 *
 * Block-sparse variant (the *_block_sparse entry points): the pages say only
 * that it only adds iteration over selected blocks, the rest of the kernel
 * staying as it is (TLX porta l'attenzione jagged su Blackwell oltre FA4 con
 * un terzo del codice, section "The turning point").  Reading taken:
 * keys come in blocks of 128 counted from each sequence's start, and a
 * selection applies to one (sequence, head) pair as a whole: key j of
 * sequence b is visible to every query of head h iff
 *     kv_block_mask[(block_start[b] + j / 128) * H + h] != 0,
 * where block_start[b] = sum over b' < b of ceil(len_b' / 128).  Keys of
 * unselected blocks behave exactly like keys outside the sequence: score
 * -inf, no weight in O, zero dK and dV; a row with no visible key is an
 * empty row (O = 0, LSE = -inf, no gradient).
 *
 * Inputs are either fp64 or bf16 bit patterns (uint16) that are widened
 * exactly to fp64 before any arithmetic.  All arithmetic is fp64.  Outputs
 * are fp64; an output pointer may be NULL, in which case that output is
 * computed but not stored.
 *
 * Parallelism: OpenMP over (sequence, head) pairs.  In broadcast mode each
 * thread accumulates dQ into a private buffer; the buffers are summed after
 * the parallel loop.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top 16 bits of an IEEE-754 binary32; widening is exact. */
static double widen_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Copy row `row` of head `h` of a [rows, H, D] tensor into dst[0..D). */
static void load_row(double *dst, const void *src, int64_t row, int h, int H, int D, int is_bf16) {
    int64_t base = (row * H + h) * (int64_t)D;
    if (is_bf16) {
        const uint16_t *s = (const uint16_t *)src + base;
        for (int d = 0; d < D; ++d) dst[d] = widen_bf16(s[d]);
    } else {
        const double *s = (const double *)src + base;
        for (int d = 0; d < D; ++d) dst[d] = s[d];
    }
}

static double dot(const double *a, const double *b, int D) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += a[d] * b[d];
    return acc;
}

int jfa_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Query row index inside Q for query i of sequence b. */
static int64_t q_row(const int32_t *off, int b, int i, int broadcast_q) {
    return broadcast_q ? (int64_t)i : (int64_t)off[b] + i;
}

/* Output-row index for (b, i) in O / dO ([B,Lq,H,D] or [N,H,D]). */
static int64_t o_row(const int32_t *off, int b, int i, int Lq, int broadcast_q) {
    return broadcast_q ? (int64_t)b * Lq + i : (int64_t)off[b] + i;
}

/* LSE index for (b, h, i): [B,H,Lq] or [H,N]. */
static int64_t lse_index(const int32_t *off, int b, int h, int i, int Lq, int H, int N, int broadcast_q) {
    return broadcast_q ? ((int64_t)b * H + h) * Lq + i : (int64_t)h * N + off[b] + i;
}

/*
 * Scores of query i against all Lk keys of one (b, h), written to s[0..Lk).
 * Returns the number of visible keys (j <= i under causal).
 */
static int scores(double *s, const double *qi, const double *kmat, int Lk, int D, int i,
                  int causal, double scale, const uint8_t *sel, int sel_stride) {
    int visible = 0;
    for (int j = 0; j < Lk; ++j) {
        if (causal && j > i) {
            s[j] = -INFINITY;
        } else if (sel && !sel[(int64_t)(j / 128) * sel_stride]) {
            s[j] = -INFINITY; /* key block not selected */
        } else {
            s[j] = scale * dot(qi, kmat + (int64_t)j * D, D);
            ++visible;
        }
    }
    return visible;
}

/*
 * First global block index of every sequence (block_start above), or NULL
 * when there is no mask.  The caller frees it.
 */
static int64_t *block_starts(const int32_t *offsets, int B, const uint8_t *mask) {
    if (!mask) return NULL;
    int64_t *bs = (int64_t *)malloc(sizeof(int64_t) * ((size_t)B + 1));
    bs[0] = 0;
    for (int b = 0; b < B; ++b) bs[b + 1] = bs[b] + (offsets[b + 1] - offsets[b] + 127) / 128;
    return bs;
}

/* LSE_i = max + ln sum exp(s - max) over visible keys; -inf when none. */
static double log_sum_exp(const double *s, int Lk) {
    double m = -INFINITY;
    for (int j = 0; j < Lk; ++j)
        if (s[j] > m) m = s[j];
    if (m == -INFINITY) return -INFINITY;
    double acc = 0.0;
    for (int j = 0; j < Lk; ++j) acc += exp(s[j] - m);
    return m + log(acc);
}

void jfa_oracle_fwd_block_sparse(const void *q, const void *k, const void *v, int in_bf16,
                                 const int32_t *offsets, int B, int Lq, int H, int D,
                                 int broadcast_q, int causal, double scale, const uint8_t *kv_block_mask,
                                 double *o, double *lse) {
    int64_t *bstart = block_starts(offsets, B, kv_block_mask);
    const int N = B > 0 ? offsets[B] : 0;
    const int64_t pairs = (int64_t)B * H;
#pragma omp parallel
    {
        double *qi = NULL, *kmat = NULL, *vmat = NULL, *s = NULL;
        int cap = 0;
        qi = (double *)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < pairs; ++bh) {
            const int b = (int)(bh / H), h = (int)(bh % H);
            const int Lk = offsets[b + 1] - offsets[b];
            const int Lqb = broadcast_q ? Lq : Lk;
            if (Lk > cap) {
                cap = Lk;
                kmat = (double *)realloc(kmat, sizeof(double) * (size_t)cap * D);
                vmat = (double *)realloc(vmat, sizeof(double) * (size_t)cap * D);
                s = (double *)realloc(s, sizeof(double) * (size_t)cap);
            }
            for (int j = 0; j < Lk; ++j) {
                load_row(kmat + (int64_t)j * D, k, (int64_t)offsets[b] + j, h, H, D, in_bf16);
                load_row(vmat + (int64_t)j * D, v, (int64_t)offsets[b] + j, h, H, D, in_bf16);
            }
            const uint8_t *sel = kv_block_mask ? kv_block_mask + bstart[b] * H + h : NULL;
            for (int i = 0; i < Lqb; ++i) {
                load_row(qi, q, q_row(offsets, b, i, broadcast_q), h, H, D, in_bf16);
                scores(s, qi, kmat, Lk, D, i, causal, scale, sel, H);
                const double L = log_sum_exp(s, Lk);
                if (lse) lse[lse_index(offsets, b, h, i, Lq, H, N, broadcast_q)] = L;
                if (o) {
                    double *oi = o + (o_row(offsets, b, i, Lq, broadcast_q) * H + h) * (int64_t)D;
                    for (int d = 0; d < D; ++d) oi[d] = 0.0;
                    if (L == -INFINITY) continue;
                    for (int j = 0; j < Lk; ++j) {
                        const double p = exp(s[j] - L);
                        for (int d = 0; d < D; ++d) oi[d] += p * vmat[(int64_t)j * D + d];
                    }
                }
            }
        }
        free(qi);
        free(kmat);
        free(vmat);
        free(s);
    }
    free(bstart);
}

void jfa_oracle_fwd(const void *q, const void *k, const void *v, int in_bf16,
                    const int32_t *offsets, int B, int Lq, int H, int D,
                    int broadcast_q, int causal, double scale,
                    double *o, double *lse) {
    jfa_oracle_fwd_block_sparse(q, k, v, in_bf16, offsets, B, Lq, H, D, broadcast_q, causal, scale, NULL, o, lse);
}

void jfa_oracle_bwd_block_sparse(const void *q, const void *k, const void *v, const void *dout, int in_bf16,
                                 const int32_t *offsets, int B, int Lq, int H, int D,
                                 int broadcast_q, int causal, double scale, const uint8_t *kv_block_mask,
                                 double *dq, double *dk, double *dv) {
    int64_t *bstart = block_starts(offsets, B, kv_block_mask);
    const int N = B > 0 ? offsets[B] : 0;
    const int64_t pairs = (int64_t)B * H;
    const int64_t q_elems = (int64_t)(broadcast_q ? Lq : N) * H * D;
    const int nthreads = jfa_oracle_max_threads();
    /* Broadcast mode: every thread sums its sequences' dQ into its own buffer. */
    double *dq_private = NULL;
    if (dq && broadcast_q)
        dq_private = (double *)calloc((size_t)nthreads * (size_t)q_elems, sizeof(double));
    if (dq && !broadcast_q) memset(dq, 0, sizeof(double) * (size_t)q_elems);

#pragma omp parallel num_threads(nthreads)
    {
#ifdef _OPENMP
        const int tid = omp_get_thread_num();
#else
        const int tid = 0;
#endif
        double *my_dq = dq ? (broadcast_q ? dq_private + (int64_t)tid * q_elems : dq) : NULL;
        double *qi = (double *)malloc(sizeof(double) * D);
        double *doi = (double *)malloc(sizeof(double) * D);
        double *kmat = NULL, *vmat = NULL, *s = NULL, *dp = NULL, *dkacc = NULL, *dvacc = NULL;
        int cap = 0;
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < pairs; ++bh) {
            const int b = (int)(bh / H), h = (int)(bh % H);
            const int Lk = offsets[b + 1] - offsets[b];
            const int Lqb = broadcast_q ? Lq : Lk;
            if (Lk > cap) {
                cap = Lk;
                kmat = (double *)realloc(kmat, sizeof(double) * (size_t)cap * D);
                vmat = (double *)realloc(vmat, sizeof(double) * (size_t)cap * D);
                dkacc = (double *)realloc(dkacc, sizeof(double) * (size_t)cap * D);
                dvacc = (double *)realloc(dvacc, sizeof(double) * (size_t)cap * D);
                s = (double *)realloc(s, sizeof(double) * (size_t)cap);
                dp = (double *)realloc(dp, sizeof(double) * (size_t)cap);
            }
            for (int j = 0; j < Lk; ++j) {
                load_row(kmat + (int64_t)j * D, k, (int64_t)offsets[b] + j, h, H, D, in_bf16);
                load_row(vmat + (int64_t)j * D, v, (int64_t)offsets[b] + j, h, H, D, in_bf16);
            }
            if (Lk > 0) {
                memset(dkacc, 0, sizeof(double) * (size_t)Lk * D);
                memset(dvacc, 0, sizeof(double) * (size_t)Lk * D);
            }
            const uint8_t *sel = kv_block_mask ? kv_block_mask + bstart[b] * H + h : NULL;
            for (int i = 0; i < Lqb; ++i) {
                load_row(qi, q, q_row(offsets, b, i, broadcast_q), h, H, D, in_bf16);
                load_row(doi, dout, o_row(offsets, b, i, Lq, broadcast_q), h, H, D, in_bf16);
                scores(s, qi, kmat, Lk, D, i, causal, scale, sel, H);
                const double L = log_sum_exp(s, Lk);
                if (L == -INFINITY) continue; /* no visible key: no gradient */
                /* P_ij overwrites s_ij; dP_ij and Delta_i from the definition. */
                double delta = 0.0;
                for (int j = 0; j < Lk; ++j) {
                    s[j] = exp(s[j] - L);
                    dp[j] = dot(doi, vmat + (int64_t)j * D, D);
                    delta += s[j] * dp[j];
                }
                double *dqi = my_dq ? my_dq + (q_row(offsets, b, i, broadcast_q) * H + h) * (int64_t)D : NULL;
                for (int j = 0; j < Lk; ++j) {
                    const double p = s[j];
                    const double ds = p * (dp[j] - delta);
                    for (int d = 0; d < D; ++d) {
                        dvacc[(int64_t)j * D + d] += p * doi[d];
                        dkacc[(int64_t)j * D + d] += scale * ds * qi[d];
                    }
                    if (dqi)
                        for (int d = 0; d < D; ++d) dqi[d] += scale * ds * kmat[(int64_t)j * D + d];
                }
            }
            for (int j = 0; j < Lk; ++j) {
                const int64_t row = ((int64_t)offsets[b] + j) * H + h;
                if (dk) memcpy(dk + row * D, dkacc + (int64_t)j * D, sizeof(double) * D);
                if (dv) memcpy(dv + row * D, dvacc + (int64_t)j * D, sizeof(double) * D);
            }
        }
        free(qi);
        free(doi);
        free(kmat);
        free(vmat);
        free(s);
        free(dp);
        free(dkacc);
        free(dvacc);
    }
    if (dq_private) {
        memset(dq, 0, sizeof(double) * (size_t)q_elems);
        for (int t = 0; t < nthreads; ++t)
            for (int64_t e = 0; e < q_elems; ++e) dq[e] += dq_private[(int64_t)t * q_elems + e];
        free(dq_private);
    }
    free(bstart);
}

void jfa_oracle_bwd(const void *q, const void *k, const void *v, const void *dout, int in_bf16,
                    const int32_t *offsets, int B, int Lq, int H, int D,
                    int broadcast_q, int causal, double scale,
                    double *dq, double *dk, double *dv) {
    jfa_oracle_bwd_block_sparse(q, k, v, dout, in_bf16, offsets, B, Lq, H, D, broadcast_q, causal, scale, NULL,
                                dq, dk, dv);
}
