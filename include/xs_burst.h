/*
 * xs_burst.h -- C ABI of the Burst-Gap store microbenchmark in libxs.so.
 *
 * Source: "X-Stage: An Overlooked Pipeline Stage for Communication-Computation
 * Overlap in DiT Inference" (arXiv 2607.23264v1), section 3.1. K concurrent
 * producers each write B bytes per burst (aggregate volume V = K*B) and then
 * spend a producer-side gap G without stores. Two modes:
 *   periodic  : bursts follow each other after the gap; the start-to-start
 *               period and the sender-visible issue time of each burst are
 *               recorded (zero gap exposes the drain rate, section 3.3; a gap
 *               sweep exposes recovery, section 3.4);
 *   isolated  : before each burst the producers idle for the gap (a recovery
 *               interval) and then start together at a grid-wide barrier; the
 *               issue time of each burst is recorded (capacity knee, section 3.5).
 * The stores go to this GPU's own memory: on one GPU this is the pages'
 * local-memory control path.
 *
 * A producer is one CTA of `warps` warps, one per SM; four warps reproduce the
 * epilogue warpgroup of the fused attention kernel, and more warps let the
 * producers inject faster than the store path drains. Its burst is written with
 * 16-byte stores, 32 consecutive chunks per warp instruction, as rows of
 * `row_bytes` bytes placed `row_stride` bytes apart (row_bytes = 128 and
 * row_stride = H*D*2 reproduce the fused kernel's scatter). Producer k's burst
 * n fills the burst-sized slot ((n*K + k) mod n_slots) of `buf`, n_slots =
 * floor(buf_bytes / (row_stride * B / row_bytes)), so a buffer larger than L2
 * makes the stores drain to HBM and a small one keeps them in L2.
 *
 * Issue time of a burst = clock64 from the producer's synchronised start to
 * the point where all its warps have issued their last store (issue, not
 * completion: a full store path stalls issue, which is the backpressure the
 * model describes).
 */
#ifndef XS_BURST_H
#define XS_BURST_H

#include <stddef.h>

#include "xs.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    double t_iss_mean_ns;   /* mean over measured bursts of the mean producer issue time */
    double t_iss_max_ns;    /* mean over measured bursts of the slowest producer's issue time */
    double t_period_ns;     /* periodic mode: mean start-to-start period (0 in isolated mode) */
    double sm_clock_mhz;    /* SM clock measured over the launch (clock64 against %globaltimer) */
    int bursts_measured;    /* bursts per producer in the means (periodic mode skips the first quarter) */
} xs_burst_stats;

/* Bytes of the device record buffer that xs_burst_gap needs for K producers
 * and n_bursts bursts each. */
size_t xs_burst_rec_bytes(int K, int n_bursts);

/*
 * Runs one microbenchmark launch on `stream` and waits for it (the call
 * synchronises the stream and reads the records back).
 *   buf, buf_bytes : device buffer the bursts write (contents overwritten);
 *                    16-byte aligned, at least row_stride * B / row_bytes bytes.
 *   rec, rec_bytes : device record buffer of at least xs_burst_rec_bytes(K,
 *                    n_bursts) bytes, 16-byte aligned; need not be initialised.
 *   K              : producers, 1 .. number of SMs.
 *   warps          : warps per producer, 1 .. 32.
 *   B              : bytes per producer per burst, a multiple of 512*warps and
 *                    of row_bytes, at most 64 MiB.
 *   gap_ns         : producer-side gap (periodic) or recovery interval before
 *                    each burst (isolated), 0 .. 1e6 ns.
 *   n_bursts       : bursts per producer, 2 .. 4096.
 *   isolated       : 0 periodic, 1 isolated.
 *   row_bytes      : 16 .. 4096, a power of two.
 *   row_stride     : >= row_bytes, a multiple of 16.
 *   stats          : results (host memory).
 * Returns XS_OK; XS_ERR_NULL / XS_ERR_SHAPE / XS_ERR_ALIGN for bad arguments,
 * XS_ERR_CUDA if the launch fails (for example when K producers cannot be
 * co-resident), XS_ERR_TIMEOUT if a bounded grid barrier ran out.
 */
xs_status xs_burst_gap(void *buf, size_t buf_bytes, void *rec, size_t rec_bytes, int K, int warps, int B,
                       double gap_ns, int n_bursts, int isolated, int row_bytes, int row_stride, xs_burst_stats *stats,
                       void *stream);

#ifdef __cplusplus
}
#endif

#endif /* XS_BURST_H */
