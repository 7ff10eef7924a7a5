// xs_internal.h -- declarations shared by the host API (xs_api.cpp) and the
// kernel translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace xs {

// Work decomposition of one attention call. A work item is a pair of
// consecutive 128-row query tiles of one (rank, batch, local head); the second
// tile of the last pair is absent when S/128 is odd.
struct AttnParams {
    int B, S, H, P, Hl, Sl;
    int n_qt;     // 128-row query tiles per head  (S / 128)
    int n_pairs;  // work items per head           (ceil(n_qt / 2))
    int n_kv;     // 128-row K/V tiles per head    (S / 128)
    int n_items;  // P * B * Hl * n_pairs
    float scale_log2;  // scale * log2(e): softmax runs in base 2
    uint16_t *out;
};

// Grid for the persistent attention kernel: one CTA per SM, never more CTAs than items.
int attn_grid(int n_items, int num_sms);

// epi = 0: head-partitioned output (same layout as q); epi = 1: All-to-All scatter.
cudaError_t launch_attention(int D, int epi, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const AttnParams &p, int grid, cudaStream_t stream);

// Device-side error word (bit 31: a bounded wait ran out; low bits: which wait).
cudaError_t read_device_error(unsigned int *value, bool clear, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);

struct PermParams {
    uint32_t rows;       // B * S * H rows of D elements
    uint32_t cpr_log2;   // log2(16-byte chunks per row)
    uint32_t B, S, H, Hl, Sl;
    // magic numbers for division by H, Sl, B and Hl (round-up method)
    uint32_t mH, sH, mSl, sSl, mB, sB, mHl, sHl;
};
void fastdiv_magic(uint32_t d, uint32_t *m, uint32_t *s);
cudaError_t launch_permute(const void *in, void *out, const PermParams &p, int num_sms, cudaStream_t stream);

}  // namespace xs
