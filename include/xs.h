/*
 * xs.h -- C ABI of the fused attention + post-attention All-to-All library (libxs.so).
 *
 * What the calls compute. Source: "X-Stage: An Overlooked Pipeline Stage for
 * Communication-Computation Overlap in DiT Inference" (arXiv 2607.23264v1).
 *   - Section 4.3: DiT self-attention is full, non-causal softmax attention,
 *       O = softmax(scale * Q K^T) V   per (batch, head),
 *     computed FlashAttention-style: a CTA owns a block of 128 query rows and
 *     walks all K/V tiles (Figure 6); finishing the walk yields one output tile.
 *   - Section 4.3, Figure 5 (d-e): Ulysses sequence parallelism runs attention
 *     head-partitioned and then an All-to-All restores the sequence partition.
 *     The fused design (Figure 7) issues each finished output tile's stores to
 *     its destination at the tile boundary and then starts the next tile.
 *   - Section 5.3: "FA-only" (xs_attn), "A2A-only" (xs_a2a_permute), "Serial"
 *     (xs_attn then xs_a2a_permute) and "Fused" (xs_attn_a2a) are the four
 *     compared implementations.
 *   - Section 4.3, Figure 5 (a-c): before attention a first All-to-All turns
 *     the sequence partition into the head partition (xs_a2a_permute_inverse);
 *     xs_ulysses_attn folds it into the attention kernel's loads.
 *
 * Ranks. P ranks are simulated as P contiguous slices of one allocation on the
 * calling GPU, so the All-to-All is a scatter of rows into slices; nothing
 * crosses a device boundary. Hl = H / P heads per rank, Sl = S / P tokens per rank.
 *
 * Layouts (row-major, elements are bf16 stored as uint16_t, D contiguous):
 *   head-partitioned      [P][B][S][Hl][D]  rank r holds global heads r*Hl .. r*Hl+Hl-1
 *                                            for all S tokens
 *   sequence-partitioned  [P][B][Sl][H][D]  rank r' holds tokens r'*Sl .. r'*Sl+Sl-1
 *                                            for all H heads, heads in ascending order
 *   element (r,b,s,hl,d) of the first is element (r',b,s-r'*Sl,h,d) of the second,
 *   with h = r*Hl + hl and r' = s / Sl. With P = 1 both are plain [B][S][H][D].
 *
 * Common rules for every compute call:
 *   - Pointers are DEVICE pointers on the current CUDA device, 16-byte aligned,
 *     owned and allocated by the caller. The library allocates no device memory;
 *     it keeps only host-side state (per-device attributes).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls are asynchronous: they return after the kernel is enqueued.
 *   - Arguments are checked before anything is enqueued. A violation returns a
 *     non-zero xs_status, enqueues nothing and leaves `out` untouched;
 *     xs_last_error() then describes it.
 *   - Shapes: B >= 0, S >= 0 (B == 0 or S == 0 is a valid empty call that
 *     enqueues nothing), H >= 1, P >= 1, H % P == 0, S % P == 0, D in {64, 96, 128, 256},
 *     scale positive and finite. Every tensor must stay below 2^40 bytes. S need
 *     not be a multiple of 128: the last query tile is then partial (rows past
 *     S are neither computed into nor stored) and the keys past S in the last
 *     K/V tile are masked out of the softmax.
 *   - `out` must not overlap q, k or v (XS_ERR_ALIAS).
 *   - The GPU must be compute capability 10.3 (sm_103); otherwise
 *     XS_ERR_UNSUPPORTED.
 *   - Inside the kernels every wait is bounded in time. A wait that runs out sets
 *     a device-side error word and the kernel returns; xs_device_status() reports
 *     it as XS_ERR_TIMEOUT. No valid input causes this.
 */
#ifndef XS_H
#define XS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    XS_OK = 0,
    XS_ERR_NULL = 1,        /* a required pointer is NULL */
    XS_ERR_SHAPE = 2,       /* a shape rule above is violated */
    XS_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
    XS_ERR_UNSUPPORTED = 4, /* D not in {64,96,128,256}, wrong GPU, or a pointer that is not device memory */
    XS_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed (message in xs_last_error) */
    XS_ERR_TIMEOUT = 6,     /* a bounded in-kernel wait ran out (reported by xs_device_status) */
    XS_ERR_ALIAS = 7,       /* out overlaps an input */
    XS_ERR_WORKSPACE = 8    /* workspace too small, misaligned or overlapping */
} xs_status;

/*
 * Fused attention + All-to-All scatter (the paper's "X-Stage-Fused" variant,
 * section 4.3, Figure 7).
 *   q, k, v : head-partitioned [P][B][S][Hl][D] bf16, read only.
 *   out     : sequence-partitioned [P][B][Sl][H][D] bf16, fully overwritten.
 *   scale   : multiplies Q K^T before the softmax (usually 1/sqrt(D)); > 0.
 * Each finished 128-row output tile of head (r, b, hl) is written straight into
 * the slices of the ranks that own its tokens. Bit-identical to
 * xs_a2a_permute(xs_attn(q, k, v)) for the same arguments.
 */
xs_status xs_attn_a2a(const void *q, const void *k, const void *v, void *out, int B, int S, int H,
                      int D, int P, float scale, void *stream);

/*
 * Attention only (the paper's "FA-only" variant, section 5.3).
 *   q, k, v : head-partitioned [P][B][S][Hl][D] bf16.
 *   out     : head-partitioned [P][B][S][Hl][D] bf16 (same layout as q), fully
 *             overwritten. P only defines the layout; P = 1 is plain [B][S][H][D].
 */
xs_status xs_attn(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D,
                  int P, float scale, void *stream);

/*
 * Standalone post-attention All-to-All (the paper's "A2A-only" variant, and the
 * second half of "Serial", section 5.3).
 *   in  : head-partitioned [P][B][S][Hl][D], 16-bit elements (any payload).
 *   out : sequence-partitioned [P][B][Sl][H][D], fully overwritten.
 * A pure copy: out is bit-for-bit a permutation of in. Same shape rules as the
 * attention calls except that scale does not apply. in and out must not overlap.
 */
xs_status xs_a2a_permute(const void *in, void *out, int B, int S, int H, int D, int P, void *stream);

/*
 * Standalone pre-attention All-to-All (Ulysses, section 4.3, Figure 5 (a-c)):
 * the inverse of xs_a2a_permute.
 *   in  : sequence-partitioned [P][B][Sl][H][D], 16-bit elements (any payload).
 *   out : head-partitioned [P][B][S][Hl][D], fully overwritten.
 * A pure copy; xs_a2a_permute(xs_a2a_permute_inverse(x)) == x bit for bit.
 * Shape and pointer rules as for xs_a2a_permute.
 */
xs_status xs_a2a_permute_inverse(const void *in, void *out, int B, int S, int H, int D, int P, void *stream);

/*
 * Both Ulysses All-to-Alls fused into one attention call (section 4.3,
 * Figure 5 (a-e), with the output side of Figure 7): attention over the whole
 * sequence for every head, from and to the sequence partition.
 *   q, k, v : sequence-partitioned [P][B][Sl][H][D] bf16, read only. Each
 *             128-row tile of head h is loaded where the sequence partition
 *             keeps it, from the slices of the ranks that own its tokens (one
 *             TMA tensor map per rank and operand), so no head-partitioned
 *             copy is ever made.
 *   out     : sequence-partitioned [P][B][Sl][H][D] bf16, fully overwritten.
 *   workspace, workspace_bytes : as for xs_attn_a2a_ws (NULL, 0: whole-item
 *             schedule); the size is xs_attn_workspace_size's.
 * Bit-identical to xs_attn_a2a_ws(xs_a2a_permute_inverse(q), ...(k), ...(v))
 * with the same workspace choice. Extra rules: P <= 8 and S/P % 8 == 0
 * (XS_ERR_UNSUPPORTED otherwise).
 */
xs_status xs_ulysses_attn(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D,
                          int P, float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Causal attention, the autoregressive-LLM case the paper contrasts with DiT's
 * full attention (section 4.3): query token i of a head attends to key tokens
 * 0..i of the same sequence only. Same arguments, layouts and rules as
 * xs_attn_a2a (fused scatter, sequence-partitioned out) and xs_attn
 * (head-partitioned out); xs_attn_causal_a2a is bit-identical to
 * xs_a2a_permute(xs_attn_causal(...)). K/V tiles entirely above the diagonal
 * are skipped; work items (pairs of 128-row query tiles) are dealt longest
 * first to balance the CTAs.
 */
xs_status xs_attn_causal_a2a(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D,
                             int P, float scale, void *stream);
xs_status xs_attn_causal(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D,
                         int P, float scale, void *stream);

/*
 * Balanced-schedule variants. Identical results contract and layouts as
 * xs_attn_a2a / xs_attn, plus a caller-owned device workspace that lets the
 * last one to two waves of work be split evenly over all SMs instead of
 * leaving some SMs idle: an output tile pair whose K/V range is split across
 * CTAs is computed in pieces whose partial rows (unnormalised O in fp32, row
 * max, row sum) meet in the workspace and are merged in a fixed order.
 * Small calls run on fewer CTAs so that pieces hold at least 16 K/V tiles,
 * but never on fewer CTAs than work items (or SMs).
 *   workspace       : device memory, 256-byte aligned, at least the size that
 *                     xs_attn_workspace_size reports for these shapes on the
 *                     current device; its contents need no initialisation and
 *                     may be left arbitrary between calls. NULL (with
 *                     workspace_bytes = 0) falls back to the whole-item schedule.
 *   workspace_bytes : its size in bytes.
 * Calls that may run concurrently must not share a workspace. xs_attn_a2a_ws
 * and xs_a2a_permute(xs_attn_ws(...)) are bit-identical for the same
 * arguments on the same device; against the whole-item schedule the split
 * tiles differ only by rounding.
 */
xs_status xs_attn_a2a_ws(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D,
                         int P, float scale, void *workspace, size_t workspace_bytes, void *stream);
xs_status xs_attn_ws(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D, int P,
                     float scale, void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes that the *_ws calls need for these shapes on the current
 * device (written to *bytes). Shape rules as for the attention calls. */
xs_status xs_attn_workspace_size(int B, int S, int H, int D, int P, size_t *bytes);

/*
 * The balanced fused call for callers that cannot allocate device memory. The
 * paper has no counterpart to this call; it exists for deployment.
 * Some callers can pass q, k, v and out but cannot allocate a workspace: a
 * plug-in inside a framework that owns all device memory through its own pool,
 * a latency-critical path that cannot afford cudaMalloc's implicit device-wide
 * synchronisation, or a process whose device memory is reserved up front.
 * This call computes what xs_attn_a2a_ws computes (same arguments minus the
 * workspace), using instead a scratch area built into the library: 48 MiB per
 * device that loads the library, held until the process exits. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   - Shapes whose balanced schedule needs more than the 48 MiB are rejected
 *     with XS_ERR_WORKSPACE before anything is enqueued
 *     (xs_attn_workspace_size reports the need).
 *   - Every call on a device shares the one scratch area, which keeps the
 *     previous call's contents. Nothing in it needs clearing: partial rows are
 *     written before they are read, and the arrival counters carry a per-launch
 *     generation stamp. Only the kernel of a call that passed every argument
 *     check writes it. Calls that may overlap on the GPU race on the scratch
 *     area and must not be issued.
 *   - The first call on a device looks up the scratch area's device address
 *     with that device current; make that first call before any stream capture.
 */
xs_status xs_attn_a2a_noalloc(const void *q, const void *k, const void *v, void *out, int B, int S, int H,
                              int D, int P, float scale, void *stream);

/*
 * Fused attention + All-to-All scatter with 8-bit queries and keys: an
 * extension, the X-Stage paper evaluates bf16 only. Same operation as
 * xs_attn_a2a_ws / xs_attn_ws, with Q K^T taken from E4M3 inputs.
 *   q8, k8 : head-partitioned [P][B][S][Hl][D] bytes, each one OCP OFP8 E4M3
 *            value (sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 *            infinities; 0x7F and 0xFF are NaN). Read only.
 *   v      : head-partitioned [P][B][S][Hl][D] bf16, read only.
 *   out    : bf16, sequence-partitioned [P][B][Sl][H][D] (xs_attn_a2a_q8) or
 *            head-partitioned like v (xs_attn_q8), fully overwritten.
 *   scale  : multiplies the exact product of the decoded q8 and k8 before the
 *            softmax; per-tensor dequantisation factors of q8 and k8 fold in
 *            here (softmax scale x q factor x k factor). > 0.
 *   workspace, workspace_bytes : as for xs_attn_a2a_ws (the same size;
 *            NULL, 0: whole-item schedule).
 * D = 128 only (XS_ERR_UNSUPPORTED otherwise). Q K^T runs on the 8-bit tensor
 * path with fp32 accumulation; the softmax, P and P V stay as in the bf16
 * calls. xs_attn_a2a_q8 is bit-identical to xs_a2a_permute(xs_attn_q8(...)).
 * XS_ERR_ALIAS when out overlaps the B*S*H*D bytes of q8 or k8 or the bf16 v.
 */
xs_status xs_attn_a2a_q8(const void *q8, const void *k8, const void *v, void *out, int B, int S, int H, int D,
                         int P, float scale, void *workspace, size_t workspace_bytes, void *stream);
xs_status xs_attn_q8(const void *q8, const void *k8, const void *v, void *out, int B, int S, int H, int D, int P,
                     float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The same with E4M3 values as well (an extension; the X-Stage paper evaluates
 * bf16 only): q8, k8 and v8 are head-partitioned [P][B][S][Hl][D] E4M3 bytes,
 * out bf16 as for xs_attn_a2a_q8 / xs_attn_q8. Each V tile is widened exactly
 * to f16 on chip, P is rounded to f16 (10 mantissa bits, against bf16's 7 in
 * the other calls) and P V runs as f16 x f16 with fp32 accumulation. A
 * dequantisation factor of v8 multiplies the output; apply it to out (or fold
 * it into the next operation). D = 128 only. xs_attn_a2a_qkv8 is bit-identical
 * to xs_a2a_permute(xs_attn_qkv8(...)). XS_ERR_ALIAS when out overlaps the
 * B*S*H*D bytes of q8, k8 or v8.
 */
xs_status xs_attn_a2a_qkv8(const void *q8, const void *k8, const void *v8, void *out, int B, int S, int H, int D,
                           int P, float scale, void *workspace, size_t workspace_bytes, void *stream);
xs_status xs_attn_qkv8(const void *q8, const void *k8, const void *v8, void *out, int B, int S, int H, int D, int P,
                       float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The fused call (xs_attn_a2a_host) and attention only (xs_attn_host) on inputs
 * and output in HOST memory, for callers whose tensors live on the host. The X-Stage
 * paper has no counterpart; these calls exist for deployment. The copies are pipelined
 * with the compute: the inputs' units, one head of one (rank, batch) slice each, are
 * split in order into up to 16 chunks of at least 8 MiB of inputs each (one chunk
 * for small calls), the first and the last the smallest. Chunk c's rows of q, k, v
 * (whole slices, and the chunk's heads of every row of a partial slice at either
 * end) are copied in on an internal stream, the caller's stream
 * runs the attention kernel over that chunk's work items, and an internal stream
 * copies the chunk's output out while later chunks are copied in and computed. For
 * xs_attn_a2a_host that output is the columns of the chunk's heads in the rows of its
 * batches of the sequence-partitioned output; for xs_attn_host, its part of the
 * head-partitioned one.
 *   q_host, k_host, v_host : head-partitioned [P][B][S][Hl][D] bf16 in host
 *       memory, read only. out_host : host memory for the output (layouts as for
 *       xs_attn_a2a / xs_attn), fully overwritten. Page-locked (pinned) host
 *       memory lets the copies run asynchronously and overlap; pageable memory
 *       works but the copies then serialise. Device or managed memory passed
 *       as a host buffer is rejected with XS_ERR_UNSUPPORTED.
 *   q, k, v, out : device staging buffers of the full sizes, 16-byte aligned,
 *       overwritten by the call (q, k, v hold the inputs afterwards, out the
 *       output). No two buffers, host or device, may overlap (XS_ERR_ALIAS).
 *   workspace, workspace_bytes : as for xs_attn_a2a_ws (NULL, 0: whole-item
 *       schedule); each chunk's launch uses it in turn. A chunk holds only a
 *       share of the work items, so without a workspace most SMs idle.
 * Asynchronous like every call. When the caller's stream reaches the point after
 * the call, out_host holds the result, and later work on that stream is ordered
 * after the copies. The first call on a device creates two streams and 34 events
 * there, kept until the process exits. A per-device lock keeps concurrent calls'
 * enqueue sequences apart. The result equals that of xs_attn_a2a_ws / xs_attn_ws
 * with the same workspace up to the rounding of split tiles (the chunks split
 * differently). Without a workspace it is bit-identical to xs_attn_a2a / xs_attn.
 */
xs_status xs_attn_a2a_host(const void *q_host, const void *k_host, const void *v_host, void *out_host, void *q,
                           void *k, void *v, void *out, int B, int S, int H, int D, int P, float scale,
                           void *workspace, size_t workspace_bytes, void *stream);
xs_status xs_attn_host(const void *q_host, const void *k_host, const void *v_host, void *out_host, void *q, void *k,
                       void *v, void *out, int B, int S, int H, int D, int P, float scale, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * The fused call (xs_attn_a2a, whole-item schedule) with its epilogue traced:
 * the per-tile record the paper's section 5.2.3 uses to measure each output
 * tile's sender-visible store span, and the section 4.3 audit its Q-loop gap.
 * Results are bit-identical to xs_attn_a2a; the records cost a few clock reads
 * and one 40-byte store per tile and epilogue warp. D = 128 only
 * (XS_ERR_UNSUPPORTED otherwise).
 *   trace, trace_bytes : device buffer of at least the size xs_attn_trace_layout
 *       reports, 16-byte aligned; zeroed and then filled by the call. Layout:
 *       [ctas][items_per_cta][tile 0..1][epilogue warp 0..3] records of five
 *       uint64: clock64 when the tile's O and row sums were ready, clock64 just
 *       before its first global store, clock64 after its last store was issued,
 *       %globaltimer (ns) when ready, and item << 8 | tile << 4 | warp (bit 3
 *       set when the tile is absent: ceil(S/128) odd). Records of a CTA that ran out
 *       of items stay zero. clock64 values compare only within one CTA. After
 *       the records come 20 uint64 per CTA; the first four are the CTA's
 *       %globaltimer at kernel entry, after set-up (barriers, tensor memory),
 *       when its first Q load was issued, and when it finished. Last come
 *       [2 items][2 tiles][64 K/V steps][4] uint64 for CTA 0's first two items:
 *       clock64 when the softmax's first warp saw the step's scores ready,
 *       when it handed P over, when the MMA issuer saw P complete, and after
 *       it issued that P V.
 */
xs_status xs_attn_a2a_trace(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D,
                            int P, float scale, void *trace, size_t trace_bytes, void *stream);

/* Grid size, items per CTA and trace bytes of xs_attn_a2a_trace for these
 * shapes on the current device. */
xs_status xs_attn_trace_layout(int B, int S, int H, int D, int P, int *ctas, int *items_per_cta, size_t *bytes);

/* Human-readable description of the last non-OK status returned on this host
 * thread (empty string if none). The pointer stays valid until the next call
 * on this thread. */
const char *xs_last_error(void);

/*
 * Synchronises `stream` and reads the device-side error word that the kernels
 * set when a bounded wait runs out. Returns XS_OK, XS_ERR_TIMEOUT (the word is
 * then cleared if `clear` != 0) or XS_ERR_CUDA if the synchronisation failed.
 */
xs_status xs_device_status(void *stream, int clear);

/*
 * Self-test of the bounded-wait path: launches one small kernel that waits on a
 * barrier nothing will ever complete, with a limit of `timeout_us` microseconds
 * (1 .. 2,000,000), then returns. The call synchronises `stream` and returns
 * XS_ERR_TIMEOUT when the wait ran out as designed (XS_OK would mean it did not),
 * leaving the device error word cleared afterwards.
 */
xs_status xs_selftest_wait_timeout(unsigned int timeout_us, void *stream);

/* Library version, major*10000 + minor*100 + patch. */
int xs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* XS_H */
