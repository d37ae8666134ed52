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
 * MXFP8 variant (the *_mxfp8 functions and the E4M3 / E8M0 helpers): see
 * the section at the end of this file, which states its readings.
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

/*
 * ===========================================================================
 * MXFP8 variant (the *_mxfp8 entry points below).
 *
 * The pages say only that an MXFP8 version of the kernel runs its matmuls in
 * microscaling precision, quantizes P to FP8 on the fly and keeps the scale
 * factors in tensor memory (TLX porta l'attenzione jagged su Blackwell oltre
 * FA4 con un terzo del codice, section "The turning point").  Readings taken:
 *
 *   - MXFP8 is the OCP microscaling format: E4M3 elements (1 sign bit, 4
 *     exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
 *     subnormals m * 2^-9; S.1111.111 is NaN; no infinities; largest finite
 *     magnitude 448), one E8M0 scale 2^(code - 127) per block of 32
 *     consecutive elements along the contraction dimension.  The block scale
 *     is 2^X with X = floor(log2(amax)) - 8, 8 being the exponent of E4M3's
 *     top binade, so the block's largest magnitude lands in [256, 512);
 *     elements round to nearest (ties to even mantissa) and magnitudes above
 *     448 saturate to 448.  An all-zero block, or one holding no element,
 *     gets code 0.
 *   - The product in MXFP8 is P V; Q K^T stays bf16.
 *   - V comes quantized.  Blocks of 32 keys are counted from each sequence's
 *     start, per head and per column d; the scales are stored per 128-key
 *     block as v_scale[((block_start[b] + n) * H + h) * D + d][c] for chunk c
 *     (keys 128 n + 32 c .. + 31 of sequence b), with block_start as in the
 *     block-sparse variant.
 *   - P is quantized in the log2 domain: with x_ij = scale * s_ij * log2(e),
 *     the 32-key chunk c of row i (chunks counted from the sequence start)
 *     has X = floor(max_{j in c} x_ij) - 8, and
 *         pq_ij = 2^X * E4M3(2^(x_ij - X)).
 *     This is the MX rule applied to the weights 2^x_ij; because X is an
 *     integer it does not depend on where the running maximum of an online
 *     softmax stood, so a kernel that keeps that maximum at an integer
 *     reaches the same pq.
 *   - O_i = sum_j pq_ij v_j / sum_j 2^x_ij: the normaliser is the row sum of
 *     the unquantized weights, and LSE is the one of the bf16 forward.
 *
 * Slack (optional output of jfa_oracle_fwd_mxfp8): a kernel computes x_ij in
 * fp32, so where the oracle's fp64 x_ij sits within 1e-4 of a decision
 * boundary (a chunk maximum near an integer, or 2^(x - X) near the midpoint
 * of two E4M3 values) the kernel may legitimately take the other side.  For
 * every output element the slack is sum_j |pq'_ij - pq_ij| |v_jd| / sum_j
 * 2^x_ij over the keys whose decision is that close, pq' the other side's
 * value.  It is zero almost everywhere.
 * ===========================================================================
 */

double jfa_oracle_e4m3_value(uint8_t c) {
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return s ? -mag : mag;
}

/* Nearest E4M3 code to a finite x (ties to the even mantissa, magnitudes of
 * 448 and above give 448); the sign of x is kept, also when it rounds to 0. */
uint8_t jfa_oracle_e4m3_encode(double x) {
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    int ex;
    frexp(a, &ex); /* a in [2^(ex-1), 2^ex) */
    /* spacing of E4M3 values around a: 2^-9 below 2^-6, else 2^(ex-1-3) */
    const int q = a < ldexp(1.0, -6) ? -9 : ex - 4;
    const double r = ldexp(nearbyint(ldexp(a, -q)), q); /* default rounding: to nearest, ties to even */
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -6)) return sign | (uint8_t)ldexp(r, 9); /* subnormal: m * 2^-9 */
    int e2;
    const double f = frexp(r, &e2); /* r = 2f * 2^(e2-1), 2f in [1, 2) */
    return sign | (uint8_t)((e2 - 1 + 7) << 3) | (uint8_t)((2.0 * f - 1.0) * 8.0);
}

void jfa_oracle_e4m3_encode_array(const double *x, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = jfa_oracle_e4m3_encode(x[i]);
}

void jfa_oracle_e4m3_value_array(const uint8_t *c, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = jfa_oracle_e4m3_value(c[i]);
}

/* Shared exponent X of an MX block with largest magnitude amax (see above),
 * within the E8M0 code range; -127 (code 0) for an all-zero block. */
int jfa_oracle_mx_exponent(double amax) {
    if (!(amax > 0.0)) return -127;
    int ex;
    frexp(amax, &ex); /* floor(log2(amax)) = ex - 1 */
    int X = ex - 1 - 8;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    return X;
}

/* block_start[b] for b = 0..B (always computed; the caller frees it). */
static int64_t *all_block_starts(const int32_t *offsets, int B) {
    int64_t *bs = (int64_t *)malloc(sizeof(int64_t) * ((size_t)B + 1));
    bs[0] = 0;
    for (int b = 0; b < B; ++b) bs[b + 1] = bs[b] + (offsets[b + 1] - offsets[b] + 127) / 128;
    return bs;
}

void jfa_oracle_quantize_v_mxfp8(const uint16_t *v, const int32_t *offsets, int B, int H, int D, uint8_t *v8,
                                 uint8_t *v_scale) {
    int64_t *bstart = all_block_starts(offsets, B);
    for (int b = 0; b < B; ++b) {
        const int Lk = offsets[b + 1] - offsets[b];
        for (int n = 0; 128 * n < Lk; ++n)
            for (int h = 0; h < H; ++h)
                for (int d = 0; d < D; ++d)
                    for (int c = 0; c < 4; ++c) {
                        const int j0 = 128 * n + 32 * c, j1 = j0 + 32 < Lk ? j0 + 32 : Lk;
                        double amax = 0.0;
                        for (int j = j0; j < j1; ++j) {
                            const double a = fabs(widen_bf16(v[(((int64_t)offsets[b] + j) * H + h) * D + d]));
                            if (a > amax) amax = a;
                        }
                        const int X = j0 < j1 ? jfa_oracle_mx_exponent(amax) : -127;
                        for (int j = j0; j < j1; ++j) {
                            const int64_t e = (((int64_t)offsets[b] + j) * H + h) * D + d;
                            v8[e] = jfa_oracle_e4m3_encode(ldexp(widen_bf16(v[e]), -X));
                        }
                        v_scale[(((bstart[b] + n) * H + h) * (int64_t)D + d) * 4 + c] = (uint8_t)(X + 127);
                    }
    }
    free(bstart);
}

/* Distance from a decision boundary within which the slack counts the other
 * side (in log2 units for a chunk maximum, relative for a rounding input). */
static const double kMxEpsFloor = 1e-4, kMxEpsRound = 1e-4;
static const double kLog2e = 1.4426950408889634074;

/* Quantized weights of one row.  x[0..n) are log2-domain logits (-inf for
 * hidden keys); chunks of 32 start at index 0.  pq[j] = 2^X E4M3(2^(x_j - X))
 * with X = floor(max of x over the chunk) - 8, 0 for hidden keys.  With
 * slack != NULL, slack[j] = |pq'_j - pq_j| for keys whose rounding or chunk
 * exponent lies within the boundary distance above (the largest such change),
 * else 0. */
void jfa_oracle_mx_quantize_p(const double *x, int n, double *pq, double *slack) {
    for (int c0 = 0; c0 < n; c0 += 32) {
        const int c1 = c0 + 32 < n ? c0 + 32 : n;
        double mx = -INFINITY;
        for (int j = c0; j < c1; ++j)
            if (x[j] > mx) mx = x[j];
        if (mx == -INFINITY) {
            for (int j = c0; j < c1; ++j) {
                pq[j] = 0.0;
                if (slack) slack[j] = 0.0;
            }
            continue;
        }
        const double f = floor(mx);
        const int X = (int)f - 8;
        int X_alt = X;
        if (mx - f < kMxEpsFloor) X_alt = X - 1;
        else if (f + 1.0 - mx < kMxEpsFloor) X_alt = X + 1;
        for (int j = c0; j < c1; ++j) {
            if (x[j] == -INFINITY) {
                pq[j] = 0.0;
                if (slack) slack[j] = 0.0;
                continue;
            }
            const double y = exp2(x[j] - X);
            const double val = ldexp(jfa_oracle_e4m3_value(jfa_oracle_e4m3_encode(y)), X);
            pq[j] = val;
            if (!slack) continue;
            double sl = 0.0;
            for (int k = -1; k <= 1; k += 2)
                sl = fmax(sl, fabs(ldexp(jfa_oracle_e4m3_value(jfa_oracle_e4m3_encode(y * (1.0 + k * kMxEpsRound))), X) - val));
            if (X_alt != X) {
                const double ya = exp2(x[j] - X_alt);
                for (int k = -1; k <= 1; ++k)
                    sl = fmax(sl, fabs(ldexp(jfa_oracle_e4m3_value(jfa_oracle_e4m3_encode(ya * (1.0 + k * kMxEpsRound))),
                                             X_alt) - val));
            }
            slack[j] = sl;
        }
    }
}

void jfa_oracle_fwd_mxfp8(const void *q, const void *k, const uint8_t *v8, const uint8_t *v_scale, int in_bf16,
                          const int32_t *offsets, int B, int Lq, int H, int D, int broadcast_q, int causal,
                          double scale, double *o, double *lse, double *o_slack) {
    int64_t *bstart = all_block_starts(offsets, B);
    const int N = B > 0 ? offsets[B] : 0;
    const int64_t pairs = (int64_t)B * H;
#pragma omp parallel
    {
        double *qi = (double *)malloc(sizeof(double) * D);
        double *kmat = NULL, *vmat = NULL, *s = NULL, *x = NULL, *pq = NULL, *sl = NULL;
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
                s = (double *)realloc(s, sizeof(double) * (size_t)cap);
                x = (double *)realloc(x, sizeof(double) * (size_t)cap);
                pq = (double *)realloc(pq, sizeof(double) * (size_t)cap);
                sl = (double *)realloc(sl, sizeof(double) * (size_t)cap);
            }
            for (int j = 0; j < Lk; ++j) {
                const int64_t row = (int64_t)offsets[b] + j;
                load_row(kmat + (int64_t)j * D, k, row, h, H, D, in_bf16);
                for (int d = 0; d < D; ++d) {
                    const uint8_t code =
                        v_scale[(((bstart[b] + j / 128) * H + h) * (int64_t)D + d) * 4 + (j % 128) / 32];
                    vmat[(int64_t)j * D + d] = ldexp(jfa_oracle_e4m3_value(v8[(row * H + h) * D + d]), code - 127);
                }
            }
            for (int i = 0; i < Lqb; ++i) {
                load_row(qi, q, q_row(offsets, b, i, broadcast_q), h, H, D, in_bf16);
                scores(s, qi, kmat, Lk, D, i, causal, scale, NULL, 0);
                const double L = log_sum_exp(s, Lk);
                if (lse) lse[lse_index(offsets, b, h, i, Lq, H, N, broadcast_q)] = L;
                const int64_t orow = (o_row(offsets, b, i, Lq, broadcast_q) * H + h) * (int64_t)D;
                if (o) memset(o + orow, 0, sizeof(double) * D);
                if (o_slack) memset(o_slack + orow, 0, sizeof(double) * D);
                if (L == -INFINITY || (!o && !o_slack)) continue;
                /* log2-domain logits, shifted by an integer so that 2^x stays in range */
                double R = -INFINITY;
                for (int j = 0; j < Lk; ++j) {
                    x[j] = s[j] * kLog2e;
                    if (x[j] > R) R = x[j];
                }
                R = floor(R);
                double den = 0.0;
                for (int j = 0; j < Lk; ++j) {
                    x[j] -= R;
                    den += exp2(x[j]);
                }
                jfa_oracle_mx_quantize_p(x, Lk, pq, o_slack ? sl : NULL);
                for (int j = 0; j < Lk; ++j)
                    for (int d = 0; d < D; ++d) {
                        const double vv = vmat[(int64_t)j * D + d];
                        if (o) o[orow + d] += pq[j] * vv / den;
                        if (o_slack) o_slack[orow + d] += sl[j] * fabs(vv) / den;
                    }
            }
        }
        free(qi);
        free(kmat);
        free(vmat);
        free(s);
        free(x);
        free(pq);
        free(sl);
    }
    free(bstart);
}
