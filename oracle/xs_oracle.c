/*
 * xs_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow fp64 CPU oracle for the fused attention + post-attention
 * All-to-All path. Only the tests, the smoke check and the bench's CPU-baseline
 * leg may load it. It shares no code, header or constant with the CUDA path.
 *
 * What it computes, and where the pages define it
 * -----------------------------------------------
 * Source: "X-Stage: An Overlooked Pipeline Stage for Communication-Computation
 * Overlap in DiT Inference" (arXiv 2607.23264v1).
 *
 *  - Attention (section 4.3): the DiT setting uses full, non-causal attention.
 *    For one head with queries q_i, keys k_j, values v_j (j = 0..S-1):
 *        s_j = scale * <q_i, k_j>,  m = max_j s_j,  p_j = exp(s_j - m),
 *        l = sum_j p_j,             o_i = (sum_j p_j v_j) / l.
 *    This is the textbook definition written out in two passes (max, then
 *    exponentials and sums). The online rescaling recurrence that FlashAttention
 *    uses reaches the same value up to rounding; the oracle does not use it.
 *
 *  - Causal attention (section 4.3 sets the DiT setting against the causal
 *    attention of autoregressive language models and does not write the mask
 *    out). Reading taken: query token i of a head sees key tokens j <= i of the
 *    same sequence, so every sum above runs over j = 0..i instead of 0..S-1.
 *
 *  - FP8 inputs (an extension; the pages evaluate bf16 only): q and k, and
 *    optionally v, may be given as E4M3 bytes, the format of the OCP 8-bit floating point
 *    specification (OFP8): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 *    bits; exponent field 0 holds subnormals m/8 * 2^-6; S.1111.111 is NaN and
 *    there is no infinity (largest finite 1.75 * 2^8 = 448). They are widened
 *    exactly to double and the attention above is unchanged.
 *
 *  - Ulysses post-attention All-to-All (section 4.3, Figure 5 d-e): attention
 *    runs head-partitioned (rank r holds heads r*Hl .. r*Hl+Hl-1 for all S
 *    tokens); the All-to-All restores the sequence partition (rank r' holds
 *    tokens r'*Sl .. r'*Sl+Sl-1 for all H heads), Hl = H/P, Sl = S/P.
 *
 * Layouts (the pages fix none; this is the plainest contiguous reading):
 *    head-partitioned  [P][B][S][Hl][D]   element ((r*B+b)*S+s)*Hl*D + hl*D + d
 *    sequence-part.    [P][B][Sl][H][D]   element ((r'*B+b)*Sl+sl)*H*D + h*D + d
 *    with h = r*Hl + hl, r' = s / Sl, sl = s - r'*Sl.
 *
 * Inputs are bf16 bit patterns (uint16); they are widened exactly to double.
 * exp() is libm's double exp. Parallelism is over independent query rows only;
 * every row is computed by one thread in the order written above.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define XSO_EINVAL (-1)
#define XSO_ENOMEM (-2)

static double bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OFP8 E4M3 code -> value (NaN for the two NaN codes). */
static double e4m3_to_double(uint8_t x) {
    const int sign = x >> 7, e = (x >> 3) & 15, m = x & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

int xs_oracle_e4m3_decode(const uint8_t *in, double *out, int64_t n) {
    if (n < 0 || (n && (!in || !out))) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_double(in[i]);
    return 0;
}

static int check_shape(int64_t B, int64_t S, int64_t H, int64_t D, int64_t P) {
    if (B < 0 || S < 0 || H <= 0 || D <= 0 || P <= 0) return XSO_EINVAL;
    if (H % P != 0 || S % P != 0) return XSO_EINVAL;
    return 0;
}

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads > 512 ? 512 : nthreads;
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    if (c < 1) c = 1;
    return c > 512 ? 512 : (int)c;
}

/* ---------------------------------------------------------------- layout maps */

/* Element offset of (r, b, s, hl, d) in the head-partitioned layout. */
int64_t xs_oracle_head_offset(int64_t r, int64_t b, int64_t s, int64_t hl, int64_t d,
                              int64_t B, int64_t S, int64_t H, int64_t D, int64_t P) {
    int64_t Hl = H / P;
    return (((r * B + b) * S + s) * Hl + hl) * D + d;
}

/* Element offset of token s of global head h, batch b, in the sequence-partitioned layout. */
int64_t xs_oracle_seq_offset(int64_t b, int64_t s, int64_t h, int64_t d,
                             int64_t B, int64_t S, int64_t H, int64_t D, int64_t P) {
    int64_t Sl = S / P;
    int64_t rd = s / Sl;       /* destination rank: owner of token s */
    int64_t sl = s - rd * Sl;  /* token index inside that rank's slice */
    return (((rd * B + b) * Sl + sl) * H + h) * D + d;
}

/* Post-attention All-to-All, written as explicit loops over the source layout:
 * every element of `in` (head-partitioned) is copied to its slot in `out`
 * (sequence-partitioned). Elements are opaque `esize`-byte payloads. */
int xs_oracle_a2a(const void *in, void *out, int64_t B, int64_t S, int64_t H, int64_t D, int64_t P,
                  int64_t esize) {
    if (check_shape(B, S, H, D, P) || esize <= 0) return XSO_EINVAL;
    if (!in || !out) return XSO_EINVAL;
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    int64_t Hl = H / P;
    for (int64_t r = 0; r < P; ++r)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t s = 0; s < S; ++s)
                for (int64_t hl = 0; hl < Hl; ++hl) {
                    int64_t h = r * Hl + hl;
                    for (int64_t d = 0; d < D; ++d) {
                        int64_t i = xs_oracle_head_offset(r, b, s, hl, d, B, S, H, D, P);
                        int64_t o = xs_oracle_seq_offset(b, s, h, d, B, S, H, D, P);
                        memcpy(dst + o * esize, src + i * esize, (size_t)esize);
                    }
                }
    return 0;
}

/* Inverse of xs_oracle_a2a (sequence-partitioned -> head-partitioned), the
 * pre-attention direction of the same exchange. */
int xs_oracle_a2a_inverse(const void *in, void *out, int64_t B, int64_t S, int64_t H, int64_t D,
                          int64_t P, int64_t esize) {
    if (check_shape(B, S, H, D, P) || esize <= 0) return XSO_EINVAL;
    if (!in || !out) return XSO_EINVAL;
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    int64_t Hl = H / P;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t s = 0; s < S; ++s)
            for (int64_t h = 0; h < H; ++h) {
                int64_t r = h / Hl, hl = h - (h / Hl) * Hl;
                for (int64_t d = 0; d < D; ++d) {
                    int64_t i = xs_oracle_seq_offset(b, s, h, d, B, S, H, D, P);
                    int64_t o = xs_oracle_head_offset(r, b, s, hl, d, B, S, H, D, P);
                    memcpy(dst + o * esize, src + i * esize, (size_t)esize);
                }
            }
    return 0;
}

/* ------------------------------------------------------------------ attention */

typedef struct {
    const uint16_t *q, *k, *v;
    const uint8_t *q8, *k8;  /* E4M3 q and k instead of q and k when not NULL */
    const uint8_t *v8;       /* E4M3 v instead of v when not NULL */
    int64_t B, S, H, D, P;
    double scale;
    int causal;        /* 1: query token i sees keys 0..i only */
    /* row list: head-partitioned row ids ((r*B+b)*S+s)*Hl+hl; NULL = all rows */
    const int64_t *rows;
    int64_t nrows;
    double *out;       /* [nrows][D] when rows != NULL, else head-partitioned [..][D] */
    int64_t begin, end;
    int err;
} attn_job_t;

/* One query row of one head: the two-pass definition above. */
static void attend_row(const attn_job_t *j, int64_t row, double *p, double *qi, double *o) {
    const int64_t S = j->S, D = j->D, Hl = j->H / j->P;
    const int64_t hl = row % Hl;
    const int64_t s_i = (row / Hl) % S;
    const int64_t rb = row / (Hl * S);
    /* row j of K/V for this (r, b, hl) head starts at ((rb*S + j)*Hl + hl)*D */
    const int64_t head_base = (rb * S * Hl + hl) * D;
    const int64_t row_stride = Hl * D;

    for (int64_t d = 0; d < D; ++d)
        qi[d] = j->q8 ? e4m3_to_double(j->q8[head_base + s_i * row_stride + d])
                      : bf16_to_double(j->q[head_base + s_i * row_stride + d]);

    /* the keys this query sees: all S, or 0..s_i when causal */
    const int64_t t0 = 0, t1 = j->causal ? s_i + 1 : S;

    /* scores s_j = scale * <q_i, k_j> */
    for (int64_t t = t0; t < t1; ++t) {
        double acc = 0.0;
        if (j->k8) {
            const uint8_t *kt = j->k8 + head_base + t * row_stride;
            for (int64_t d = 0; d < D; ++d) acc += qi[d] * e4m3_to_double(kt[d]);
        } else {
            const uint16_t *kt = j->k + head_base + t * row_stride;
            for (int64_t d = 0; d < D; ++d) acc += qi[d] * bf16_to_double(kt[d]);
        }
        p[t] = j->scale * acc;
    }
    /* m = max_j s_j */
    double m = p[t0];
    for (int64_t t = t0 + 1; t < t1; ++t)
        if (p[t] > m) m = p[t];
    /* p_j = exp(s_j - m), l = sum_j p_j */
    double l = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        p[t] = exp(p[t] - m);
        l += p[t];
    }
    /* o = sum_j p_j v_j / l ; for every d the sum runs over j in ascending order */
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        if (j->v8) {
            const uint8_t *vt = j->v8 + head_base + t * row_stride;
            for (int64_t d = 0; d < D; ++d) o[d] += p[t] * e4m3_to_double(vt[d]);
        } else {
            const uint16_t *vt = j->v + head_base + t * row_stride;
            for (int64_t d = 0; d < D; ++d) o[d] += p[t] * bf16_to_double(vt[d]);
        }
    }
    for (int64_t d = 0; d < D; ++d) o[d] /= l;
}

static void *attn_worker(void *arg) {
    attn_job_t *j = (attn_job_t *)arg;
    double *p = (double *)malloc(sizeof(double) * (size_t)(j->S > 0 ? j->S : 1));
    double *qi = (double *)malloc(sizeof(double) * (size_t)j->D);
    if (!p || !qi) {
        free(p);
        free(qi);
        j->err = XSO_ENOMEM;
        return 0;
    }
    for (int64_t i = j->begin; i < j->end; ++i) {
        int64_t row = j->rows ? j->rows[i] : i;
        attend_row(j, row, p, qi, j->out + i * j->D);
    }
    free(p);
    free(qi);
    return 0;
}

static int run_attention(attn_job_t base, int64_t total, int nthreads) {
    nthreads = resolve_threads(nthreads);
    if ((int64_t)nthreads > total) nthreads = total > 0 ? (int)total : 1;
    attn_job_t *jobs = (attn_job_t *)calloc((size_t)nthreads, sizeof(attn_job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return XSO_ENOMEM;
    }
    /* interleaved row blocks so that threads share the same heads' K/V in cache */
    int64_t per = (total + nthreads - 1) / nthreads;
    int used = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].begin = (int64_t)t * per;
        jobs[t].end = jobs[t].begin + per > total ? total : jobs[t].begin + per;
        if (jobs[t].begin >= jobs[t].end) break;
        used++;
    }
    for (int t = 1; t < used; ++t) pthread_create(&tid[t], 0, attn_worker, &jobs[t]);
    if (used > 0) attn_worker(&jobs[0]);
    for (int t = 1; t < used; ++t) pthread_join(tid[t], 0);
    int err = 0;
    for (int t = 0; t < used; ++t)
        if (jobs[t].err) err = jobs[t].err;
    free(jobs);
    free(tid);
    return err ? err : used;
}

/* Attention for every (r, b, hl) head; o is head-partitioned [P][B][S][Hl][D].
 * causal = 1 restricts query i to keys 0..i. Returns the number of threads
 * used (> 0), or a negative error. */
int xs_oracle_attention_ex(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *o, int64_t B,
                           int64_t S, int64_t H, int64_t D, int64_t P, double scale, int causal, int nthreads) {
    if (check_shape(B, S, H, D, P)) return XSO_EINVAL;
    int64_t total = P * B * S * (H / P);
    if (total == 0) return 1;
    if (!q || !k || !v || !o) return XSO_EINVAL;
    attn_job_t base = {q, k, v, 0, 0, 0, B, S, H, D, P, scale, causal != 0, 0, 0, o, 0, 0, 0};
    return run_attention(base, total, nthreads);
}

/* As xs_oracle_attention_ex with q and k given as E4M3 bytes (same layout);
 * v is bf16, or E4M3 bytes when v_e4m3 != 0. */
int xs_oracle_attention_q8(const uint8_t *q8, const uint8_t *k8, const void *v, int v_e4m3, double *o, int64_t B,
                           int64_t S, int64_t H, int64_t D, int64_t P, double scale, int causal, int nthreads) {
    if (check_shape(B, S, H, D, P)) return XSO_EINVAL;
    int64_t total = P * B * S * (H / P);
    if (total == 0) return 1;
    if (!q8 || !k8 || !v || !o) return XSO_EINVAL;
    attn_job_t base = {0, 0, v_e4m3 ? 0 : (const uint16_t *)v, q8, k8, v_e4m3 ? (const uint8_t *)v : 0,
                       B, S, H, D, P, scale, causal != 0, 0, 0, o, 0, 0, 0};
    return run_attention(base, total, nthreads);
}

int xs_oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *o, int64_t B,
                        int64_t S, int64_t H, int64_t D, int64_t P, double scale, int nthreads) {
    return xs_oracle_attention_ex(q, k, v, o, B, S, H, D, P, scale, 0, nthreads);
}

/* Attention for a list of head-partitioned row ids; o_rows is [nrows][D]. */
int xs_oracle_attention_rows_ex(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                                int64_t S, int64_t H, int64_t D, int64_t P, double scale, int causal,
                                const int64_t *rows, int64_t nrows, double *o_rows, int nthreads) {
    if (check_shape(B, S, H, D, P) || nrows < 0) return XSO_EINVAL;
    if (nrows == 0) return 1;
    if (!q || !k || !v || !rows || !o_rows) return XSO_EINVAL;
    int64_t total_rows = P * B * S * (H / P);
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= total_rows) return XSO_EINVAL;
    attn_job_t base = {q, k, v, 0, 0, 0, B, S, H, D, P, scale, causal != 0, rows, nrows, o_rows, 0, 0, 0};
    return run_attention(base, nrows, nthreads);
}

int xs_oracle_attention_rows_q8(const uint8_t *q8, const uint8_t *k8, const void *v, int v_e4m3, int64_t B,
                                int64_t S, int64_t H, int64_t D, int64_t P, double scale, int causal,
                                const int64_t *rows, int64_t nrows, double *o_rows, int nthreads) {
    if (check_shape(B, S, H, D, P) || nrows < 0) return XSO_EINVAL;
    if (nrows == 0) return 1;
    if (!q8 || !k8 || !v || !rows || !o_rows) return XSO_EINVAL;
    int64_t total_rows = P * B * S * (H / P);
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= total_rows) return XSO_EINVAL;
    attn_job_t base = {0, 0, v_e4m3 ? 0 : (const uint16_t *)v, q8, k8, v_e4m3 ? (const uint8_t *)v : 0,
                       B, S, H, D, P, scale, causal != 0, rows, nrows, o_rows, 0, 0, 0};
    return run_attention(base, nrows, nthreads);
}

int xs_oracle_attention_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                             int64_t S, int64_t H, int64_t D, int64_t P, double scale,
                             const int64_t *rows, int64_t nrows, double *o_rows, int nthreads) {
    return xs_oracle_attention_rows_ex(q, k, v, B, S, H, D, P, scale, 0, rows, nrows, o_rows, nthreads);
}

/* Fused reference: attention followed by the All-to-All of its fp64 result.
 * out is sequence-partitioned [P][B][Sl][H][D] (doubles). */
int xs_oracle_attention_a2a_ex(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *out,
                               int64_t B, int64_t S, int64_t H, int64_t D, int64_t P, double scale, int causal,
                               int nthreads) {
    if (check_shape(B, S, H, D, P)) return XSO_EINVAL;
    int64_t n = P * B * S * (H / P) * D;
    if (n == 0) return 1;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)n);
    if (!tmp) return XSO_ENOMEM;
    int used = xs_oracle_attention_ex(q, k, v, tmp, B, S, H, D, P, scale, causal, nthreads);
    if (used > 0) {
        int e = xs_oracle_a2a(tmp, out, B, S, H, D, P, (int64_t)sizeof(double));
        if (e) used = e;
    }
    free(tmp);
    return used;
}

int xs_oracle_attention_a2a(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *out,
                            int64_t B, int64_t S, int64_t H, int64_t D, int64_t P, double scale,
                            int nthreads) {
    return xs_oracle_attention_a2a_ex(q, k, v, out, B, S, H, D, P, scale, 0, nthreads);
}

int xs_oracle_default_threads(void) { return resolve_threads(0); }
