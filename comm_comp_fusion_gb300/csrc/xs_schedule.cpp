// xs_schedule.cpp -- the work schedule of an attention call: the grid size and
// how work items are dealt to CTAs (AttnParams: n_dp, sk_item0, sk_units,
// sk_q, sk_r), and the chunks of the host-buffer pipeline. Host code only, so
// the CPU tests compile it on its own.
#include "xs_internal.h"

namespace xs {

int attn_schedule(AttnParams &p, int num_sms, bool balanced) {
    const long long units = (long long)p.n_items * p.n_kv;
    p.sk_item0 = p.n_items;
    p.sk_units = 0;
    p.sk_q = 0;
    p.sk_r = 0;
    if (!balanced) {
        const int G = p.n_items < num_sms ? p.n_items : num_sms;
        p.n_dp = (p.n_items + G - 1) / G;
        return G;
    }
    // pieces of at least 16 K/V steps, but never fewer CTAs than items (or SMs)
    const long long by_piece = units / 16, floor_g = p.n_items < num_sms ? p.n_items : num_sms;
    long long g = by_piece > floor_g ? by_piece : floor_g;
    if (g > num_sms) g = num_sms;
    if (g > units) g = units;
    const int G = (int)g;
    if (p.n_items % G == 0) {
        p.n_dp = p.n_items / G;
        return G;
    }
    // keep one full wave (plus the remainder) for the balanced region
    p.n_dp = p.n_items / G - 1;
    if (p.n_dp < 0) p.n_dp = 0;
    p.sk_item0 = p.n_dp * G;
    const long long u = (long long)(p.n_items - p.sk_item0) * p.n_kv;
    if (u >= (1ll << 31)) {  // too long to split in 32-bit arithmetic: whole items only
        p.n_dp = (p.n_items + G - 1) / G;
        p.sk_item0 = p.n_items;
        return G;
    }
    p.sk_units = (uint32_t)u;
    p.sk_q = p.sk_units / (uint32_t)G;
    p.sk_r = p.sk_units % (uint32_t)G;
    return G;
}

// Chunks of the host-buffer pipeline over the call's P * B (rank, batch)
// slices, each contiguous in the head-partitioned inputs: one per slice, at
// most max_chunks, and about 8 MiB of inputs per chunk at least (a chunk's
// launch costs several microseconds, more than copying a small chunk takes).
// Chunk c covers slices [c n / chunks, (c + 1) n / chunks) of the n = slices.
int host_chunks(int slices, long long input_bytes, int max_chunks) {
    const long long by_size = input_bytes >> 23;
    int chunks = slices < max_chunks ? slices : max_chunks;
    if (by_size < chunks) chunks = by_size > 1 ? (int)by_size : 1;
    return chunks;
}

}  // namespace xs
