// xs_schedule.cpp -- the work schedule of an attention call: the grid size and
// how work items are dealt to CTAs (AttnParams: n_dp, sk_item0, sk_units,
// sk_q, sk_r), and the chunks of the host-buffer pipeline. Host code only, so
// the CPU tests compile it on its own.
#include <algorithm>
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

// Chunks of the host-buffer pipeline over the call's units, a unit being one
// head of one (rank, batch) slice, in work-item order (a unit's items are
// contiguous, and so are its rows within a slice). Only the first chunk's copy
// in and the last chunk's copy out are exposed, so both are small: a chunk holds
// at least min_bytes of inputs (a launch costs several microseconds, more than
// copying a small chunk takes), the sizes grow by half from the first up to
// about an eighth of the call and shrink the same way towards the last. Growing
// by half keeps the copies in ahead of the compute whenever the host link moves
// more than two thirds of the inputs' bytes per unit of compute time. At most
// max_chunks (the middle size is doubled until they fit). bounds[c] is chunk
// c's first unit, bounds[n] = units; returns n.
int host_chunk_plan(int units, long long unit_bytes, long long min_bytes, int max_chunks, int *bounds) {
    if (units <= 0) {
        bounds[0] = 0;
        return 0;
    }
    const long long ub = unit_bytes > 0 ? unit_bytes : 1;
    const int m = (int)std::min<long long>(units, std::max<long long>(1, (min_bytes + ub - 1) / ub));
    for (long long mid = std::max<long long>(m, (units + 7) / 8);; mid *= 2) {
        // the ramp: m, 1.5 m, 2.25 m, ... below the middle size
        int ramp[16], nr = 0;
        const int nr_max = std::min(16, (max_chunks - 1) / 2);  // 2 nr + 1 chunks fit
        long long in_ramps = 0;
        for (double x = m; x < (double)mid && nr < nr_max; x *= 1.5) {
            const int r = (int)(x + 0.5);
            if (in_ramps + 2 * r > units) break;
            ramp[nr++] = r;
            in_ramps += 2 * r;
        }
        const long long middle = units - in_ramps;
        const long long n_mid = middle > 0 ? std::max<long long>(1, middle / mid) : 0;  // each at least mid
        const long long n = 2 * nr + n_mid;
        if (n > max_chunks && mid < units) continue;
        int c = 0, u = 0;
        bounds[0] = 0;
        for (int i = 0; i < nr; ++i) bounds[++c] = (u += ramp[i]);
        for (long long i = 0; i < n_mid; ++i) bounds[++c] = (u += (int)(middle * (i + 1) / n_mid - middle * i / n_mid));
        for (int i = nr - 1; i >= 0; --i) bounds[++c] = (u += ramp[i]);
        return c;
    }
}

}  // namespace xs
