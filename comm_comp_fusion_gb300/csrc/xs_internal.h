// xs_internal.h -- declarations shared by the host API (xs_api.cpp) and the
// kernel translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace xs {

// Work decomposition of one attention call. A work item is a pair of
// consecutive 128-row query tiles of one (rank, batch, local head); the second
// tile of the last pair is absent when ceil(S/128) is odd, and the last tile
// is partial when S is not a multiple of 128. A unit is one item and
// one 128-row K/V tile.
//
// Schedule: CTA c first takes whole items c, c + G, ..., c + (n_dp - 1) G
// (G = gridDim.x). The remaining items, the "balanced region" starting at
// sk_item0, hold sk_units units that are dealt out as G contiguous ranges of
// equal length, [c*U/G, (c+1)*U/G); an item whose units fall into several
// ranges is computed in pieces whose partial results meet in the workspace.
struct AttnParams {
    int B, S, H, P, Hl, Sl;
    int ld_rows;  // sequence-partitioned inputs: token rows per TMA box (gcd(Sl, 128))
    int n_qt;     // 128-row query tiles per head  (ceil(S / 128))
    int n_pairs;  // work items per head           (ceil(n_qt / 2))
    int n_kv;     // 128-row K/V tiles per head    (ceil(S / 128))
    int kv_tail;  // keys in the last K/V tile (128 unless S is ragged); later columns are masked
    int n_items;  // P * B * Hl * n_pairs (P * B * Hl * n_qt for single-tile items), or a rank range's share
    int item0 = 0;  // global index of work item 0 (a call over the ranks from rank0 on: rank0 * B * Hl * items per head)
    float scale_log2;  // scale * log2(e): softmax runs in base 2
    uint16_t *out;
    int head_out;          // 1: output head-partitioned like q (attention only); 0: the All-to-All scatter
    int n_dp;              // round-robin waves of whole items
    int sk_item0;          // first item of the balanced region
    uint32_t sk_units;     // units U in the balanced region (0: none), below 2^31
    uint32_t sk_q, sk_r;   // U = sk_q * G + sk_r, so range starts are c*q + (c*r)/G
    float *ws_rec;         // 2 * G partial records (see partial_record_bytes)
    unsigned long long *ws_cnt;  // arrival counters, 4 per tile of each item of the balanced region
    unsigned long long gen;      // this launch's 48-bit generation, stamped into the counters
    unsigned long long *trace;  // traced instances: epilogue records, kTraceWords per (CTA, item, tile, warp)
};

// Epilogue trace record of one output tile and epilogue warp (32 rows):
// clock64 when the tile's O and row sums were ready, before its first store,
// after its last store was issued; %globaltimer when ready; then
// item << 8 | tile << 4 | warp, with bit 3 set for an absent tile.
constexpr int kTraceWords = 5;

// Head dimension 256 runs the single-query-tile kernel (xs_attn1_kernel.cuh):
// its work item is one 128-row query tile instead of a pair.
inline bool single_tile_items(int D) { return D > 128; }
inline int tiles_per_item(int D) { return single_tile_items(D) ? 1 : 2; }

// Bytes of one partial record: unnormalised O of the item's tiles (fp32) plus
// their row max and row sum.
inline size_t partial_record_bytes(int D) {
    return (size_t)tiles_per_item(D) * (128 * (size_t)D * 4 + 2 * 128 * 4);
}

// Chooses the grid and fills the schedule fields of p. With a workspace the
// tail waves are balanced; without one every CTA takes whole items only.
int attn_schedule(AttnParams &p, int num_sms, bool balanced);
// Chunks of the host-buffer pipeline over (slice, head) units; fills bounds[0..n], returns n.
int host_chunk_plan(int units, long long unit_bytes, long long min_bytes, int max_chunks, int *bounds);
// Workspace bytes a balanced call needs (records, then counters), 256-aligned parts.
size_t attn_workspace_bytes(int n_items, int n_kv, int D, int num_sms);

// Most simulated ranks a call with sequence-partitioned inputs accepts: the
// kernel takes two TMA tensor maps per source rank and operand as a parameter.
constexpr int kMaxRanks = 8;
constexpr int kSeqMaps = 2 * kMaxRanks;

// TMA tensor maps of Q, K and V. NM = 1: one map per operand over the
// head-partitioned tensor. NM = kSeqMaps: maps over each source rank's
// sequence-partitioned slice; entry r (r < P) has boxes of ld_rows = gcd(Sl, 128)
// rows, which never straddle two ranks, and entry kMaxRanks + r boxes of 128 rows
// for tiles that lie inside rank r's slice (used only when Sl >= 128).
template <int NM> struct OperandMaps {
    CUtensorMap q[NM], k[NM], v[NM];
};

// The output layout is p.head_out (head-partitioned) or the All-to-All scatter;
// both run the same compiled kernel.
cudaError_t launch_attention(int D, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                             cudaStream_t stream);
// The fused call with epilogue tracing (p.trace set, whole-item schedule).
cudaError_t launch_attention_traced(int D, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                                    cudaStream_t stream);
// Causal attention (query token i sees keys 0..i), whole-item schedule.
cudaError_t launch_causal(int D, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                          cudaStream_t stream);
// Sequence-partitioned inputs (the pre-attention All-to-All done by the loads),
// sequence-partitioned output.
cudaError_t launch_ulysses(int D, const OperandMaps<kSeqMaps> &maps, const AttnParams &p, int grid,
                           cudaStream_t stream);

// Per-head-dimension instances (xs_attn_d64.cu, xs_attn_d96.cu, xs_attn_d128.cu).
#define XS_DECLARE_ATTN_ENTRY(D)                                                                                  \
    cudaError_t launch_attention_d##D(const OperandMaps<1> &maps, const AttnParams &p, int grid,          \
                                      cudaStream_t stream);                                                       \
    cudaError_t launch_ulysses_d##D(const OperandMaps<kSeqMaps> &maps, const AttnParams &p, int grid,             \
                                    cudaStream_t stream);                                                         \
    cudaError_t launch_causal_d##D(const OperandMaps<1> &maps, const AttnParams &p, int grid,             \
                                   cudaStream_t stream);                                                          \
    cudaError_t read_error_word_d##D(unsigned int *value, bool clear);
XS_DECLARE_ATTN_ENTRY(64)
XS_DECLARE_ATTN_ENTRY(96)
XS_DECLARE_ATTN_ENTRY(128)
XS_DECLARE_ATTN_ENTRY(256)
cudaError_t launch_attention_traced_d128(const OperandMaps<1> &maps, const AttnParams &p, int grid,
                                         cudaStream_t stream);
// E4M3 inputs, D = 128 only (xs_attn_f8.cu): f8 = 1 for E4M3 q and k (maps over
// bytes) with bf16 v, f8 = 2 for E4M3 q, k and v.
cudaError_t launch_attention_f8_d128(int f8, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                                     cudaStream_t stream);
cudaError_t read_error_word_f8(unsigned int *value, bool clear);

// Sets the calling thread's xs_last_error() text; returns `status`.
int report_error(int status, const char *message);

// Device-side error word (bit 31: a bounded wait ran out; low bits: which wait).
cudaError_t read_device_error(unsigned int *value, bool clear, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);

struct PermParams {
    uint32_t rows;       // B * S * H rows of D elements
    uint32_t cpr;        // 16-byte chunks per row (D / 8)
    uint32_t cpr_log2;   // log2(cpr) when cpr is a power of two
    uint32_t mC, sC;     // magic numbers for division by cpr otherwise
    uint32_t B, S, H, Hl, Sl;
    // magic numbers for division by H, Sl, B, Hl and S (round-up method)
    uint32_t mH, sH, mSl, sSl, mB, sB, mHl, sHl, mS, sS;
};
void fastdiv_magic(uint32_t d, uint32_t *m, uint32_t *s);
// inverse = false: head-partitioned -> sequence-partitioned (post-attention
// All-to-All); inverse = true: the reverse (pre-attention All-to-All).
cudaError_t launch_permute(const void *in, void *out, const PermParams &p, bool inverse, int num_sms,
                           cudaStream_t stream);

}  // namespace xs
