/*
 * Seeded synthetic inputs shared by the tests, the bench and the oracle checks.
 *
 * This file holds no attention or All-to-All arithmetic: it only turns a
 * (seed, stream) pair into a reproducible sequence of bf16 values.
 *
 *   generator : PCG32, XSH-RR output on a 64-bit LCG (M. E. O'Neill, "PCG: A
 *               Family of Simple Fast Space-Efficient Statistically Good
 *               Algorithms for Random Number Generation", 2014), seeded the way
 *               the paper's pcg32_srandom does it.
 *   jump-ahead: F. B. Brown, "Random Number Generation with Arbitrary Strides",
 *               1994 (used only so that threads can start mid-sequence; the
 *               values are the same as a single sequential pass).
 *   uniform   : u = ((x >> 8) + 1) * 2^-24, in (0, 1].
 *   normal    : Box-Muller on consecutive pairs (u1, u2); both outputs are used,
 *               cos first: z0 = sqrt(-2 ln u1) cos(2 pi u2),
 *               z1 = sqrt(-2 ln u1) sin(2 pi u2).
 *   bf16      : sigma * z is rounded to fp32 (round to nearest even) and then
 *               to bf16 (round to nearest even on the upper 16 bits).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#include <unistd.h>

#define PCG_MULT 6364136223846793005ULL

typedef struct {
    uint64_t state;
    uint64_t inc;
} pcg32_t;

static uint32_t pcg32_next(pcg32_t *g) {
    uint64_t old = g->state;
    g->state = old * PCG_MULT + g->inc;
    uint32_t xorshifted = (uint32_t)(((old >> 18u) ^ old) >> 27u);
    uint32_t rot = (uint32_t)(old >> 59u);
    return (xorshifted >> rot) | (xorshifted << ((32u - rot) & 31u));
}

static void pcg32_seed(pcg32_t *g, uint64_t seed, uint64_t stream) {
    g->state = 0u;
    g->inc = (stream << 1u) | 1u;
    (void)pcg32_next(g);
    g->state += seed;
    (void)pcg32_next(g);
}

/* Advance the LCG by `delta` steps in O(log delta) (Brown 1994). */
static void pcg32_advance(pcg32_t *g, uint64_t delta) {
    uint64_t acc_mult = 1u, acc_plus = 0u;
    uint64_t cur_mult = PCG_MULT, cur_plus = g->inc;
    while (delta > 0) {
        if (delta & 1u) {
            acc_mult *= cur_mult;
            acc_plus = acc_plus * cur_mult + cur_plus;
        }
        cur_plus = (cur_mult + 1u) * cur_plus;
        cur_mult *= cur_mult;
        delta >>= 1u;
    }
    g->state = acc_mult * g->state + acc_plus;
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static double unit_open0(uint32_t x) { return ((double)(x >> 8) + 1.0) * (1.0 / 16777216.0); }

/* Raw PCG32 outputs: used by the generator's own pins. */
void xsgen_pcg32_raw(uint64_t seed, uint64_t stream, uint64_t skip, uint32_t *out, int64_t n) {
    pcg32_t g;
    pcg32_seed(&g, seed, stream);
    pcg32_advance(&g, skip);
    for (int64_t i = 0; i < n; ++i) out[i] = pcg32_next(&g);
}

typedef struct {
    uint64_t seed, stream;
    double sigma;
    uint16_t *out;
    int64_t n, pair_begin, pair_end;
} normal_job_t;

static void *normal_worker(void *arg) {
    normal_job_t *j = (normal_job_t *)arg;
    pcg32_t g;
    pcg32_seed(&g, j->seed, j->stream);
    pcg32_advance(&g, 2u * (uint64_t)j->pair_begin);
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t p = j->pair_begin; p < j->pair_end; ++p) {
        double u1 = unit_open0(pcg32_next(&g));
        double u2 = unit_open0(pcg32_next(&g));
        double r = sqrt(-2.0 * log(u1));
        double z0 = r * cos(two_pi * u2);
        double z1 = r * sin(two_pi * u2);
        int64_t e = 2 * p;
        j->out[e] = f32_to_bf16_rne((float)(j->sigma * z0));
        if (e + 1 < j->n) j->out[e + 1] = f32_to_bf16_rne((float)(j->sigma * z1));
    }
    return 0;
}

/* Fill out[0..n) with bf16 bits of sigma * N(0,1). Returns the thread count used. */
int xsgen_normal_bf16(uint64_t seed, uint64_t stream, double sigma, uint16_t *out, int64_t n, int nthreads) {
    if (n <= 0) return 0;
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > 256) nthreads = 256;
    int64_t npairs = (n + 1) / 2;
    if (npairs < (int64_t)nthreads * 4096) nthreads = 1;
    normal_job_t jobs[256];
    pthread_t tid[256];
    int64_t per = (npairs + nthreads - 1) / nthreads;
    int used = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t b = (int64_t)t * per, e = b + per;
        if (b >= npairs) break;
        if (e > npairs) e = npairs;
        jobs[t] = (normal_job_t){seed, stream, sigma, out, n, b, e};
        used++;
    }
    if (used == 1) {
        normal_worker(&jobs[0]);
        return 1;
    }
    for (int t = 0; t < used; ++t) pthread_create(&tid[t], 0, normal_worker, &jobs[t]);
    for (int t = 0; t < used; ++t) pthread_join(tid[t], 0);
    return used;
}
