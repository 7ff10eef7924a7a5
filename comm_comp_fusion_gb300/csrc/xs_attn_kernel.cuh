// xs_attn_kernel.cuh -- persistent, warp-specialised non-causal attention for sm_103a
// whose epilogue writes each finished output tile either head-partitioned or
// straight into the post-attention All-to-All layout.
//
// What it computes (X-Stage paper, arXiv 2607.23264v1):
//   * section 4.3, Figure 6: a CTA owns 128 query rows of one head and walks all
//     ceil(S/128) K/V tiles (the Q-loop); finishing the walk yields a 128 x D
//     output tile, and successive output tiles form the outer loop;
//   * section 4.3, Figure 7: at an output-tile boundary the role that owns O
//     issues that tile's stores to the destination rank, then the next tile's
//     Q-loop runs while those stores drain; no warp or SM is reserved for
//     communication;
//   * section 4.3, Figure 5 (d-e): the destination is the Ulysses sequence
//     partition: token s of global head h = r*Hl + hl goes to rank r' = s / Sl;
//   * section 4.3, Figure 5 (a-c): optionally (LD = 1) the pre-attention
//     All-to-All is folded into the loads too: Q, K and V rows of head h are
//     fetched from the sequence-partitioned slices of the ranks that own them,
//     through TMA tensor maps per rank;
//   * causal (CAU) and ragged (RAG, S not a multiple of 128) instances, and
//     E4M3 inputs (F8, D = 128): queries and keys, or queries, keys and values.
//
// Softmax is computed online (running row max m, running sum l, rescaling of
// O when m grows), in base 2 with scale*log2(e) folded into one FMA. The row
// max used for the exponentials is only moved when the new maximum exceeds it
// by more than 2^8 in value; otherwise the stale maximum is kept, which bounds
// p by 256 and leaves O/l unchanged mathematically. After a work item's first
// step the max is not taken up front: the exponentials use the stale m, and
// only a row sum of p above 256 (the sole sign that some p may pass 2^8) sends
// the warp back to S for the max and a second pass.
//
// Roles (512 threads, one CTA per SM, persistent over work items):
//   warp 0      TMA producer: Q tile pair, then K_j, V_j into a 4-slot ring
//   warp 1      MMA issuer (one thread): S_t = Q_t K_j^T, O_t += P_t V_j
//   warp 2      tensor-memory allocator
//   warps 2-3   (F8 = 2) widen each E4M3 V tile to f16 in its ring slot
//   warps 4-7   softmax of query tile 0 (one thread per row)
//   warps 8-11  softmax of query tile 1
//   warps 12-15 epilogue: O/l -> bf16 -> shared-memory transpose -> coalesced
//               16-byte stores into the destination rows
// Tensor memory (512 columns): S0 | S1 | O0 | O1; P_t (bf16, or f16 with F8 = 2)
// overwrites the first half of S_t after the softmax has read it.
//
// Schedule: whole items round-robin, then (when the caller passes a workspace)
// the last one to two waves of (item, K/V tile) units split evenly over all
// CTAs. An item cut by a range boundary is computed in pieces; each piece's
// epilogue warp writes its unnormalised rows, row max and row sum to the
// workspace, and the warp that arrives last for those rows merges the pieces
// in piece order and stores the final rows, so the result does not depend on
// which piece finishes last.
//
// Every mbarrier wait is bounded in time; if one runs out the CTA raises a
// shared abort flag, records the site in a device error word and winds down.
#pragma once

#include <atomic>

#include "xs_internal.h"
#include "xs_ptx.cuh"

namespace xs {

// Device-side error word of this translation unit (bit 31: a bounded wait ran
// out; low bits: which wait). Every translation unit that includes this header
// has its own copy; the host reads them all.
static __device__ unsigned int g_xs_error = 0;

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s; a whole call takes milliseconds

enum WaitSite : uint32_t {
    kSiteLoadQ = 0, kSiteLoadKV, kSiteMmaQ, kSiteMmaKV, kSiteMmaP, kSiteMmaOFree, kSiteSoftS,
    kSiteSoftL, kSiteEpiO, kSiteEpiL, kSiteDrain, kSiteSelftest, kSiteSoftO
};

__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                       uint32_t site, unsigned long long limit_ns) {
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1u;
            atomicOr(&g_xs_error, 0x80000000u | (1u << site));
            return false;
        }
    }
}

__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                      uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort_flag, site, kWaitLimitNs);
}

// Warp-uniform bounded wait: every lane waits, then the warp agrees.
__device__ __forceinline__ bool warp_bwait(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                           uint32_t site) {
    const bool ok = bwait(bar, parity, abort_flag, site);
    return __all_sync(0xffffffffu, ok);
}


// F8 = 1: Q and K are E4M3 bytes (one 128-byte swizzle block per row at
// D = 128); V, P and the output stay bf16. F8 = 2: V is E4M3 as well; it lands
// in a two-slot staging ring and is widened exactly to f16 in its K/V ring
// slot, and P is rounded to f16 for an f16 x f16 P V.
template <int D, int F8 = 0> struct Cfg {
    static_assert(D == 64 || D == 96 || D == 128, "head dimension");
    static_assert(F8 == 0 || D == 128, "E4M3 inputs are built for D = 128");
    static constexpr bool Q8 = F8 >= 1, V8 = F8 == 2;
    // 64-column (128-byte) swizzle blocks per row; with D = 96 the second block
    // is half used (TMA zero-fills its other half)
    static constexpr int kNDB = (D + 63) / 64;
    static constexpr uint32_t kBlk = 128u * 128u;       // one swizzle block of a 128-row tile
    static constexpr uint32_t kTile = kNDB * kBlk;      // a 128-row bf16 tile in shared memory
    static constexpr uint32_t kQKTile = Q8 ? 128u * D : kTile;  // a 128-row Q or K tile
    static constexpr int kSlots = 4;                    // K/V ring slots (K and V alternate)
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffKV = kOffQ + 2 * kQKTile;
    static constexpr uint32_t kOffStage = kOffKV + kSlots * kTile;
    static constexpr uint32_t kStageWarp = 32u * 128u;  // 32 rows x 64 bf16 per epilogue warp
    static constexpr uint32_t kV8Tile = 128u * D;       // an E4M3 V tile (staging)
    static constexpr uint32_t kOffV8 = kOffStage + 4 * kStageWarp;
    static constexpr uint32_t kOffBar = kOffV8 + (V8 ? 2 * kV8Tile : 0);
    static constexpr uint32_t kOffL = kOffBar + 8 * 32;       // float [tile][l, m][128]
    static constexpr uint32_t kOffMisc = kOffL + 2 * 2 * 128 * 4; // tmem base, abort flag
    static constexpr uint32_t kSmemUsed = kOffMisc + 16;
    static constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;  // slack to align the base to 1024
    __host__ __device__ static constexpr uint32_t colS(int t) { return 128u * (uint32_t)t; }
    __host__ __device__ static constexpr uint32_t colO(int t) { return 256u + (uint32_t)D * (uint32_t)t; }
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

// mbarrier slots
enum : int {
    BQ_FULL = 0, BQ_EMPTY = 2, BKV_FULL = 4, BKV_EMPTY = 8, BS_FULL = 12, BP_FULL = 14,
    BO_FINAL = 16, BO_FREE = 18, BL_FULL = 20, BL_EMPTY = 22, B_DRAIN = 24,
    BV8_FULL = 26, BV8_EMPTY = 28   // E4M3 V staging ring (F8 = 2)
};

struct Item {
    int rb, hl, pair;
};
__device__ __forceinline__ Item decode_item(const AttnParams &p, int item) {
    Item it;
    item += p.item0;  // scheduler items are local to the call's rank range
    it.pair = item % p.n_pairs;
    const int head = item / p.n_pairs;
    it.hl = head % p.Hl;
    it.rb = head / p.Hl;
    return it;
}

// One stretch of work for a CTA: K/V tiles [j0, j1) of an item.
struct Seg {
    int item, j0, j1;
    bool split;  // not the whole K/V range: a piece of an item
    bool first;  // starts where this CTA's balanced range starts
};
struct Sched {
    int k;
    uint32_t u, u_begin, u_end;
};
// First unit of CTA c's balanced range: floor(c * U / G), in 32-bit arithmetic.
__device__ __forceinline__ uint32_t sk_start(uint32_t c, const AttnParams &p) {
    return c * p.sk_q + (c * p.sk_r) / gridDim.x;
}
// The CTA whose balanced range holds unit u (binary search on the range starts).
__device__ __forceinline__ int sk_cta_of(uint32_t u, const AttnParams &p) {
    uint32_t lo = 0, hi = gridDim.x - 1;  // sk_start(lo) <= u < sk_start(hi + 1)
    while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) >> 1;
        if (sk_start(mid, p) <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return (int)lo;
}
__device__ __forceinline__ void sched_init(Sched &s, const AttnParams &p) {
    s.k = 0;
    s.u = s.u_begin = sk_start(blockIdx.x, p);
    s.u_end = sk_start(blockIdx.x + 1, p);
}
// CAU (causal): item lengths differ (pair p needs 2p + 2 K/V tiles), so whole
// items go out longest first, dealt to the CTAs in a snake order (wave w runs
// CTA 0..G-1 when w is even and G-1..0 when odd), a longest-processing-time
// assignment that keeps the CTAs' totals close.
template <bool CAU>
__device__ __forceinline__ bool sched_next(Sched &s, const AttnParams &p, Seg &g) {
    if (CAU) {
        const int G = (int)gridDim.x, n_heads = p.n_items / p.n_pairs;
        while (s.k < p.n_dp) {
            const int w = s.k++;
            const int rank = w * G + ((w & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
            if (rank >= p.n_items) continue;
            const int pair = p.n_pairs - 1 - rank / n_heads;
            g.item = (rank % n_heads) * p.n_pairs + pair;
            g.j0 = 0;
            g.j1 = min(2 * pair + 2, p.n_kv);
            g.split = false;
            g.first = false;
            return true;
        }
        return false;
    }
    while (s.k < p.n_dp) {
        const int item = (int)blockIdx.x + s.k * (int)gridDim.x;
        ++s.k;
        if (item < p.n_items) {
            g.item = item;
            g.j0 = 0;
            g.j1 = p.n_kv;
            g.split = false;
            g.first = false;
            return true;
        }
    }
    if (s.u >= s.u_end) return false;
    const uint32_t x = s.u / (uint32_t)p.n_kv;
    const int j0 = (int)(s.u - x * (uint32_t)p.n_kv);
    const uint32_t rem = s.u_end - s.u;
    const int j1 = rem < (uint32_t)(p.n_kv - j0) ? j0 + (int)rem : p.n_kv;
    g.item = p.sk_item0 + (int)x;
    g.j0 = j0;
    g.j1 = j1;
    g.split = !(j0 == 0 && j1 == p.n_kv);
    g.first = s.u == s.u_begin;
    s.u += (uint32_t)(j1 - j0);
    return true;
}

// True when the segment just returned by sched_next is this CTA's last.
template <bool CAU>
__device__ __forceinline__ bool sched_done(const Sched &s, const AttnParams &p) {
    Sched t = s;
    Seg g;
    return !sched_next<CAU>(t, p, g);
}

__device__ __forceinline__ float ld_cg(const float *ptr) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
    return v;
}
__device__ __forceinline__ float4 ld_cg4(const float4 *ptr) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(ptr));
    return v;
}

// Element offset of the first element of output row (rb, hl, token s).
// p.head_out: head-partitioned like q (attention only); otherwise the row's slot
// in the sequence partition (the All-to-All scatter). Attention only and the
// fused call thus run the same compiled kernel.
template <int D, bool RAG>
__device__ __forceinline__ int64_t out_row_offset(const AttnParams &p, int rb, int hl, int s) {
    if (RAG && s >= p.S) return -1;  // a row of a partial last tile that does not exist
    if (p.head_out) return (((int64_t)rb * p.S + s) * p.Hl + hl) * D;
    const int b = rb % p.B, r = rb / p.B;
    const int h = r * p.Hl + hl;
    const int rd = s / p.Sl, sl = s - rd * p.Sl;
    return ((((int64_t)rd * p.B + b) * p.Sl + sl) * p.H + h) * D;
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
// Hides a value from the optimiser so that it is recomputed where used instead
// of being hoisted (and held in registers) across a loop.
__device__ __forceinline__ uint32_t opaque(uint32_t x) {
    asm volatile("" : "+r"(x));
    return x;
}
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

// ----------------------------------------------------------------- output rows
// Output rows go through shared memory: each lane writes 16-byte chunk c (8
// bf16) of its own row into staging row `lane` (XOR-swizzled), then the warp
// copies its 32 rows out with coalesced 16-byte stores, 128 bytes per row.
__device__ __forceinline__ void stage_chunk(uint32_t stage, int lane, int c, uint32_t x0, uint32_t x1, uint32_t x2,
                                            uint32_t x3) {
    const uint32_t a = stage + lane * 128 + ((c ^ (lane & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x0), "r"(x1), "r"(x2), "r"(x3) : "memory");
}
// CPR = 16-byte chunks per row of the block (8, or 4 for the half block of D = 96).
template <bool GUARD, int CPR>
__device__ __forceinline__ void flush_rows(uint16_t *out, uint32_t stage, int lane, int64_t dst, int db) {
    __syncwarp();
#pragma unroll
    for (int i = 0; i < CPR; ++i) {
        const int idx = i * 32 + lane;
        const int rr = idx / CPR, c = idx % CPR;
        const uint32_t a = stage + rr * 128 + ((c ^ (rr & 7)) << 4);
        uint32_t y0, y1, y2, y3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(y0), "=r"(y1), "=r"(y2), "=r"(y3) : "r"(a) : "memory");
        const int64_t d = __shfl_sync(0xffffffffu, dst, rr);
        uint16_t *gp = out + d + db * 64 + c * 8;
        if (GUARD) {
            // rows past S (d < 0) are not stored; the predicate stays inside the asm
            asm volatile(
                "{\n .reg .pred p;\n setp.ge.s64 p, %5, 0;\n @p st.global.v4.b32 [%0], {%1, %2, %3, %4};\n}" ::"l"(gp),
                "r"(y0), "r"(y1), "r"(y2), "r"(y3), "l"(d)
                : "memory");
        } else {
            asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(gp), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
                         : "memory");
        }
    }
    __syncwarp();
}
// Stores the warp's 32 staged rows. With RAG (S not a multiple of 128) a row
// whose destination is -1 (past S in a partial last tile) is skipped.
template <bool RAG, int CPR = 8>
__device__ __forceinline__ void flush_block(uint16_t *out, uint32_t stage, int lane, int64_t dst, int db) {
    if (RAG && __any_sync(0xffffffffu, dst < 0))
        flush_rows<true, CPR>(out, stage, lane, dst, db);
    else
        flush_rows<false, CPR>(out, stage, lane, dst, db);
}

// ------------------------------------------------------------ split items
// Floats in one partial record: unnormalised O of both tiles as
// [tile][D/4][128 rows][4], then [tile][row max, row sum][128].
template <int D> struct Rec {
    static constexpr size_t kFloats = 2 * 128 * D + 2 * 2 * 128;
    static constexpr size_t kML = 2 * 128 * D;
};

// Record of the piece of the split item starting at unit ua that CTA c computed.
__device__ __forceinline__ const float *piece_record(const AttnParams &p, int c, uint32_t ua, size_t rec_floats) {
    const int slot = 2 * c + (sk_start((uint32_t)c, p) >= ua ? 0 : 1);
    return p.ws_rec + (size_t)slot * rec_floats;
}

// Merge of a split item's pieces for one warp's 32 rows of tile t, in piece
// order, and the store of the final rows. With self_tmem the piece computed by
// this CTA is read from tensor memory (it never went to the workspace);
// otherwise every piece, this CTA's included, comes from the workspace. Both
// read the same bits, so the result does not depend on which piece merges.
// CH columns (8, 16, 32 or 64) are gathered per round.
template <int D, int CH, bool RAG, typename DstFn>
__device__ __forceinline__ void merge_rows(const AttnParams &p, int t, int row, int lane, uint32_t stage, int c_first,
                                           int c_last, uint32_t ua, bool self_tmem, float m_self, float l_self,
                                           uint32_t tO, DstFn dst_fn, bool valid) {
    using R = Rec<D>;
    const int self = (int)blockIdx.x;
    float M = -INFINITY;
    for (int c = c_first; c <= c_last; ++c)
        M = fmaxf(M, (self_tmem && c == self) ? m_self
                                             : ld_cg(piece_record(p, c, ua, R::kFloats) + R::kML + t * 256 + row));
    float L = 0.f;
    for (int c = c_first; c <= c_last; ++c) {
        float mc, lc;
        if (self_tmem && c == self) {
            mc = m_self;
            lc = l_self;
        } else {
            const float *r = piece_record(p, c, ua, R::kFloats) + R::kML + t * 256;
            mc = ld_cg(r + row);
            lc = ld_cg(r + 128 + row);
        }
        L += ex2_approx(mc - M) * lc;
    }
    const float inv_L = 1.0f / L;
#pragma unroll 1
    for (int col0 = 0; col0 < D; col0 += CH) {
        float acc[CH];
#pragma unroll
        for (int i = 0; i < CH; ++i) acc[i] = 0.f;
        for (int c = c_first; c <= c_last; ++c) {
            if (CH >= 16 && self_tmem && c == self) {  // merges of 8 columns read only the workspace
                const float wk = ex2_approx(m_self - M);
                if constexpr (CH < 16) {
                } else if constexpr (CH == 16) {
                    uint32_t o[16];
                    tmem_ld16(tO + col0, o);
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = fmaf(wk, __uint_as_float(o[i]), acc[i]);
                } else {
#pragma unroll
                    for (int h = 0; h < CH; h += 32) {
                        uint32_t o[32];
                        tmem_ld32(tO + col0 + h, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) acc[h + i] = fmaf(wk, __uint_as_float(o[i]), acc[h + i]);
                    }
                }
            } else {
                const float *r = piece_record(p, c, ua, R::kFloats);
                const float wk = ex2_approx(ld_cg(r + R::kML + t * 256 + row) - M);
                const float4 *src = reinterpret_cast<const float4 *>(r) + (size_t)t * (D / 4) * 128;
                float4 v[CH / 4];
#pragma unroll
                for (int q = 0; q < CH / 4; ++q) v[q] = ld_cg4(src + (size_t)(col0 / 4 + q) * 128 + row);
#pragma unroll
                for (int q = 0; q < CH / 4; ++q) {
                    acc[4 * q] = fmaf(wk, v[q].x, acc[4 * q]);
                    acc[4 * q + 1] = fmaf(wk, v[q].y, acc[4 * q + 1]);
                    acc[4 * q + 2] = fmaf(wk, v[q].z, acc[4 * q + 2]);
                    acc[4 * q + 3] = fmaf(wk, v[q].w, acc[4 * q + 3]);
                }
            }
        }
        if (valid) {
#pragma unroll
            for (int c = 0; c < CH / 8; ++c)
                stage_chunk(stage, lane, (col0 % 64) / 8 + c, pack_bf16x2(acc[8 * c + 0] * inv_L, acc[8 * c + 1] * inv_L),
                            pack_bf16x2(acc[8 * c + 2] * inv_L, acc[8 * c + 3] * inv_L),
                            pack_bf16x2(acc[8 * c + 4] * inv_L, acc[8 * c + 5] * inv_L),
                            pack_bf16x2(acc[8 * c + 6] * inv_L, acc[8 * c + 7] * inv_L));
            if ((col0 + CH) % 64 == 0)
                flush_block<RAG>(p.out, stage, lane, dst_fn(), col0 / 64);
            else if (col0 + CH == D)  // the half block of D = 96
                flush_block<RAG, 4>(p.out, stage, lane, dst_fn(), col0 / 64);
        }
    }
}

// One warp's 32 rows of tile t of a split piece, after its last PV: either
// merge now (TRY_SELF and every other piece already arrived; this piece is read
// from TMEM) and return 0, or publish this piece's rows (unnormalised O, row
// max, row sum) to the workspace and return 1: the caller must then count the
// arrival with arrive_piece. `release` runs once the rows are out of TMEM.
template <int D, int CH, bool RAG, bool TRY_SELF, typename DstFn, typename Release>
__device__ __forceinline__ uint32_t finish_piece(const AttnParams &p, const Seg &g, int t, int wq, int row, int lane,
                                                 uint32_t stage, int c_first, int c_last, uint32_t ua, float m, float l,
                                                 uint32_t tO, DstFn dst_fn, bool valid, Release release) {
    using R = Rec<D>;
    const uint32_t x_local = (uint32_t)(g.item - p.sk_item0);
    const uint32_t npieces = (uint32_t)(c_last - c_first + 1);
    const unsigned long long *cnt = p.ws_cnt + ((size_t)x_local * 8 + t * 4 + wq);
    uint32_t others = 0;
    if (TRY_SELF && lane == 0) others = arrivals_now(cnt, p.gen) == npieces - 1u ? 1u : 0u;
    others = __shfl_sync(0xffffffffu, others, 0);
    if (TRY_SELF && others) {
        __threadfence();
        merge_rows<D, CH, RAG>(p, t, row, lane, stage, c_first, c_last, ua, true, m, l, tO, dst_fn, valid);
        release();
        return 0;
    }
    const int own_slot = 2 * (int)blockIdx.x + (g.first ? 0 : 1);
    float *rec = p.ws_rec + (size_t)own_slot * R::kFloats;
    float4 *o4 = reinterpret_cast<float4 *>(rec) + (size_t)t * (D / 4) * 128;
    // CH columns (16 or 32) per round
    constexpr int W = CH < 32 ? 16 : 32;
#pragma unroll 1
    for (int c = 0; c < D; c += W) {
        uint32_t o[W];
        if constexpr (W == 16)
            tmem_ld16(tO + c, o);
        else
            tmem_ld32(tO + c, o);
        if (c + W == D) release();
#pragma unroll
        for (int q = 0; q < W / 4; ++q)
            o4[(size_t)(c / 4 + q) * 128 + row] = make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                                              __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
    }
    rec[R::kML + t * 256 + row] = m;
    rec[R::kML + t * 256 + 128 + row] = l;
    return 1;
}

// Counts this piece's arrival for tile t (after its rows were published and
// fenced); the last arrival merges from the workspace.
template <int D, int CH, bool RAG, typename DstFn>
__device__ __forceinline__ void arrive_piece(const AttnParams &p, const Seg &g, int t, int wq, int row, int lane,
                                             uint32_t stage, int c_first, int c_last, uint32_t ua, DstFn dst_fn,
                                             bool valid) {
    const uint32_t x_local = (uint32_t)(g.item - p.sk_item0);
    uint32_t last = 0;
    if (lane == 0)
        last = arrive_last(p.ws_cnt + ((size_t)x_local * 8 + t * 4 + wq), p.gen, (uint32_t)(c_last - c_first + 1))
                   ? 1u
                   : 0u;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    merge_rows<D, CH, RAG>(p, t, row, lane, stage, c_first, c_last, ua, false, 0.f, 0.f, 0u, dst_fn, valid);
}


// Issues the TMA copies of token rows [s0, s0 + 128) of one head of one operand
// into a 128-row tile at shared address `dst` (D/64 swizzle blocks of 128 rows).
// Head-partitioned tensor: one 128-row box per block.
template <int D>
__device__ __forceinline__ void load_rows_head(uint32_t dst, const CUtensorMap *map, uint32_t bar, int rb, int hl,
                                               int s0) {
#pragma unroll
    for (int db = 0; db < Cfg<D>::kNDB; ++db) tma_load_4d(dst + db * Cfg<D>::kBlk, map, bar, db * 64, hl, s0, rb);
}

// Sequence-partitioned tensor: the rows are read where the sequence partition
// keeps them, in the slice of the rank that owns each token (the pre-attention
// All-to-All of Ulysses, section 4.3, Figure 5 (a-c)), through that rank's
// tensor maps. Token s0 is row `sl` of rank `rs`'s slice. A tile inside one
// rank's slice takes one 128-row box per swizzle block; a tile that straddles
// ranks takes boxes of p.ld_rows rows, which divides Sl, so no box straddles
// two ranks. Rows at or past S (the absent second tile of an odd tile count,
// the tail of a partial last tile) lie outside every map and are zero-filled.
template <int D>
__device__ __forceinline__ void load_rows_seq(uint32_t dst, const CUtensorMap *maps, uint32_t bar,
                                              const AttnParams &p, int b, int h, int rs, int sl) {
    if (sl + 128 <= p.Sl) {
#pragma unroll
        for (int db = 0; db < Cfg<D>::kNDB; ++db)
            tma_load_4d(dst + db * Cfg<D>::kBlk, maps + kMaxRanks + rs, bar, db * 64, h, sl, b);
        return;
    }
    for (int y = 0; y < 128; y += p.ld_rows) {
#pragma unroll
        for (int db = 0; db < Cfg<D>::kNDB; ++db)
            tma_load_4d(dst + db * Cfg<D>::kBlk + (uint32_t)y * 128u, maps + rs, bar, db * 64, h, sl, b);
        sl += p.ld_rows;
        if (sl == p.Sl && rs + 1 < p.P) {
            sl = 0;
            ++rs;
        }
    }
}

// Rank holding token s (the last rank for s >= S) and its row in that slice.
__device__ __forceinline__ void seq_position(const AttnParams &p, int s, int &rs, int &sl) {
    rs = s < p.S ? s / p.Sl : p.P - 1;
    sl = s - rs * p.Sl;
}

// Ragged S: the keys past S (zero-filled rows of the last K/V tile) take no
// weight; their scores become -inf in this thread's row of tensor memory.
// Kept out of line: inlined, it costs the softmax loop 2% at ragged DiT size.
static __device__ __noinline__ void mask_tail(uint32_t tS, int kv_tail) {
    for (int c = kv_tail; c < 128; ++c) tmem_st1(tS + (uint32_t)c, f2u(-INFINITY));
    tmem_st_wait();
}

template <int D, int LD, int TRACE, bool RAG, bool CAU, int F8 = 0>
__global__ void __launch_bounds__(512, 1)
    attn_fwd_kernel(const __grid_constant__ OperandMaps<LD ? kSeqMaps : 1> tm, const AttnParams p) {
    using C = Cfg<D, F8>;
    constexpr bool Q8 = C::Q8, V8 = C::V8;
    static_assert(F8 == 0 || (LD == 0 && !CAU), "E4M3 inputs: head-partitioned, non-causal");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - raw);
    const uint32_t sQ = base + C::kOffQ, sKV = base + C::kOffKV, sStage = base + C::kOffStage;
    const uint32_t sBar = base + C::kOffBar;
    float *row_ml = reinterpret_cast<float *>(sm + C::kOffL);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + C::kOffMisc);
    volatile uint32_t *abort_flag = misc + 1;
#define BAR(i) (sBar + 8u * (uint32_t)(i))

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // traced instances: per-CTA times after the tile records (kernel entry, set-up
    // done, first Q load issued, CTA done), %globaltimer
    unsigned long long *cta_times =
        TRACE ? p.trace + ((size_t)gridDim.x * p.n_dp * 8 + (size_t)blockIdx.x * 4) * kTraceWords : nullptr;
    // and, for CTA 0's first two items, per tile and K/V step (up to 64): clock64
    // when the softmax saw S ready, when it handed P over, when the MMA issuer
    // saw P complete, and after it issued that P V
    unsigned long long *step_times =
        TRACE && blockIdx.x == 0 ? p.trace + ((size_t)gridDim.x * p.n_dp * 8 + (size_t)gridDim.x * 4) * kTraceWords
                                 : nullptr;
#define STEP_TIME(item, t, j, k, v)                                                              \
    do {                                                                                         \
        if (TRACE && step_times && (item) < 2 && (j) < 64)                                       \
            step_times[(((size_t)(item) * 2 + (t)) * 64 + (size_t)(j)) * 4 + (k)] = (v);          \
    } while (0)
    if (TRACE && threadIdx.x == 0) cta_times[0] = globaltimer_ns();

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(BAR(BQ_FULL + t), 1);
            mbar_init(BAR(BQ_EMPTY + t), 1);
            mbar_init(BAR(BS_FULL + t), 1);
            mbar_init(BAR(BP_FULL + t), 4);
            mbar_init(BAR(BO_FINAL + t), 1);
            mbar_init(BAR(BO_FREE + t), 4);
            mbar_init(BAR(BL_FULL + t), 4);
            mbar_init(BAR(BL_EMPTY + t), 4);
        }
        for (int s = 0; s < C::kSlots; ++s) {
            // E4M3 V: the V slots (odd; K and V alternate) fill when both widening warps arrive
            mbar_init(BAR(BKV_FULL + s), V8 && (s & 1) ? 2 : 1);
            mbar_init(BAR(BKV_EMPTY + s), 1);
        }
        if (V8)
            for (int s = 0; s < 2; ++s) {
                mbar_init(BAR(BV8_FULL + s), 1);
                mbar_init(BAR(BV8_EMPTY + s), 2);
            }
        mbar_init(BAR(B_DRAIN), 1);
        misc[1] = 0u;
        fence_mbar_init();
        for (int r = 0; r < (LD ? p.P : 1); ++r) {
            prefetch_tmap(&tm.q[r]);
            prefetch_tmap(&tm.k[r]);
            prefetch_tmap(&tm.v[r]);
            if (LD && p.Sl >= 128) {
                prefetch_tmap(&tm.q[kMaxRanks + r]);
                prefetch_tmap(&tm.k[kMaxRanks + r]);
                prefetch_tmap(&tm.v[kMaxRanks + r]);
            }
        }
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(misc), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const int wg = warp >> 2;
    if (TRACE && threadIdx.x == 0) cta_times[1] = globaltimer_ns();

    if (wg == 0) {
        setmaxnreg_dec<48>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------ TMA producer
            uint32_t kv_it = 0, it = 0;
            bool ok = true;
            Sched sch;
            sched_init(sch, p);
            Seg g;
            for (; ok && sched_next<CAU>(sch, p, g); ++it) {
                const Item w = decode_item(p, g.item);
                // sequence-partitioned inputs: batch and global head of the item
                const int b = LD ? w.rb % p.B : 0, h = LD ? (w.rb / p.B) * p.Hl + w.hl : 0;
                for (int t = 0; t < 2 && ok; ++t) {
                    ok = bwait(BAR(BQ_EMPTY + t), (it & 1u) ^ 1u, abort_flag, kSiteLoadQ);
                    if (!ok) break;
                    mbar_arrive_expect_tx(BAR(BQ_FULL + t), C::kQKTile);
                    const int s0 = (2 * w.pair + t) * 128;  // past S for an absent tile: zero fill
                    if (TRACE && it == 0 && t == 0) cta_times[2] = globaltimer_ns();
                    if (LD) {
                        int rs, sl;
                        seq_position(p, s0, rs, sl);
                        load_rows_seq<D>(sQ + t * C::kTile, tm.q, BAR(BQ_FULL + t), p, b, h, rs, sl);
                    } else if (Q8) {  // one 128-byte box per row: 128 E4M3 elements
                        tma_load_4d(sQ + t * C::kQKTile, tm.q, BAR(BQ_FULL + t), 0, w.hl, s0, w.rb);
                    } else {
                        load_rows_head<D>(sQ + t * C::kTile, tm.q, BAR(BQ_FULL + t), w.rb, w.hl, s0);
                    }
                }
                int rs = 0, sl = 0;  // position of K/V token j * 128, advanced tile by tile
                if (LD) seq_position(p, g.j0 * 128, rs, sl);
                for (int j = g.j0; ok && j < g.j1; ++j) {
                    for (int kv = 0; kv < 2; ++kv, ++kv_it) {
                        const uint32_t slot = kv_it % C::kSlots, ph = (kv_it / C::kSlots) & 1u;
                        if (V8 && kv) {  // E4M3 V goes to staging slot slot / 2; the widening warps fill the ring slot
                            const uint32_t s8 = slot >> 1;
                            ok = bwait(BAR(BV8_EMPTY + s8), ph ^ 1u, abort_flag, kSiteLoadKV);
                            if (!ok) break;
                            mbar_arrive_expect_tx(BAR(BV8_FULL + s8), C::kV8Tile);
                            tma_load_4d(base + C::kOffV8 + s8 * C::kV8Tile, tm.v, BAR(BV8_FULL + s8), 0, w.hl,
                                        j * 128, w.rb);
                            continue;
                        }
                        ok = bwait(BAR(BKV_EMPTY + slot), ph ^ 1u, abort_flag, kSiteLoadKV);
                        if (!ok) break;
                        mbar_arrive_expect_tx(BAR(BKV_FULL + slot), kv ? C::kTile : C::kQKTile);
                        const CUtensorMap *m = kv ? tm.v : tm.k;
                        if (Q8 && !kv)
                            tma_load_4d(sKV + slot * C::kTile, m, BAR(BKV_FULL + slot), 0, w.hl, j * 128, w.rb);
                        else if (LD)
                            load_rows_seq<D>(sKV + slot * C::kTile, m, BAR(BKV_FULL + slot), p, b, h, rs, sl);
                        else
                            load_rows_head<D>(sKV + slot * C::kTile, m, BAR(BKV_FULL + slot), w.rb, w.hl, j * 128);
                    }
                    if (LD) {
                        sl += 128;
                        while (sl >= p.Sl && rs + 1 < p.P) {
                            sl -= p.Sl;
                            ++rs;
                        }
                    }
                }
            }
            if (!ok) {  // let copies already in flight land before the CTA exits
                const unsigned long long t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
        } else if (V8 && warp >= 2) {
            // ---------------------------------------------- E4M3 V widening (F8 = 2)
            // Warp 2 widens columns 0-63 (swizzle block 0), warp 3 columns 64-127.
            // Lane = 8 * (16-byte input chunk within the half row) + row within an
            // 8-row swizzle atom, so both the loads (E4M3 staging, 128-byte
            // swizzle) and the stores (f16 MN-major tile, 128-byte swizzle) hit
            // eight distinct 16-byte bank groups per quarter warp.
            const uint32_t e = (uint32_t)lane & 7u;                        // row within the atom
            const uint32_t u = (uint32_t)(warp - 2) * 4u + ((uint32_t)lane >> 3);  // input chunk 0..7
            const uint32_t db = u >> 2, c0 = (2u * u) & 7u;                 // output block and chunk pair
            const uint32_t ld_off = e * 128u + ((u ^ e) << 4);
            const uint32_t st_off0 = db * C::kBlk + e * 128u + ((c0 ^ e) << 4);
            const uint32_t st_off1 = db * C::kBlk + e * 128u + (((c0 + 1u) ^ e) << 4);
            uint32_t v_it = 0;
            bool ok = true;
            Sched sch;
            sched_init(sch, p);
            Seg g;
            while (ok && sched_next<CAU>(sch, p, g)) {
                for (int j = g.j0; ok && j < g.j1; ++j, ++v_it) {
                    const uint32_t kv_it = 2u * v_it + 1u;  // V tiles sit at odd ring positions
                    const uint32_t slot = kv_it % C::kSlots, ph = (kv_it / C::kSlots) & 1u, s8 = slot >> 1;
                    ok = warp_bwait(BAR(BV8_FULL + s8), ph, abort_flag, kSiteLoadKV) &&
                         warp_bwait(BAR(BKV_EMPTY + slot), ph ^ 1u, abort_flag, kSiteLoadKV);
                    if (!ok) break;
                    const uint32_t src = base + C::kOffV8 + s8 * C::kV8Tile + ld_off;
                    const uint32_t dst = sKV + slot * C::kTile;
#pragma unroll 2
                    for (uint32_t rg = 0; rg < 16; ++rg) {  // 8-row groups
                        uint32_t x0, x1, x2, x3, y0, y1, y2, y3, y4, y5, y6, y7;
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                                     : "r"(src + rg * 1024u)
                                     : "memory");
                        e4m3x4_to_f16x4(x0, y0, y1);
                        e4m3x4_to_f16x4(x1, y2, y3);
                        e4m3x4_to_f16x4(x2, y4, y5);
                        e4m3x4_to_f16x4(x3, y6, y7);
                        st_shared_v4(dst + rg * 1024u + st_off0, y0, y1, y2, y3);
                        st_shared_v4(dst + rg * 1024u + st_off1, y4, y5, y6, y7);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(BAR(BV8_EMPTY + s8));
                        mbar_arrive(BAR(BKV_FULL + slot));
                    }
                }
            }
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------------- MMA issuer
            constexpr uint32_t idS = Q8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, 0);
            constexpr uint32_t idO = V8 ? idesc_f16_f32(128, D, 1) : idesc_bf16_f32(128, D, 1);
            // Descriptors differ only in the start-address field (address >> 4 in
            // the low 14 bits), so each MMA adds a compile-time offset to a base.
            const uint64_t dK = sdesc_sw128(0, 16, 1024);       // K-major, 128-byte rows
            const uint64_t dV = sdesc_sw128(0, C::kBlk, 1024);  // MN-major V, 64-column blocks kBlk apart
            auto issue_S = [&](int t, uint32_t slot) {
                const uint64_t qa = dK + (opaque(sQ + t * C::kQKTile) >> 4);
                const uint64_t ka = dK + (opaque(sKV + slot * C::kTile) >> 4);
                const uint32_t d = opaque(tmem + C::colS(t));
                // one MMA per 32 bytes of a row: K = 16 bf16 or K = 32 E4M3 elements
#pragma unroll
                for (int kk = 0; kk < (Q8 ? D / 32 : D / 16); ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kBlk + (kk & 3) * 32) >> 4;
                    if (Q8)
                        tc_mma_ss_f8(d, qa + off, ka + off, idS, kk > 0 ? 1u : 0u);
                    else
                        tc_mma_ss(d, qa + off, ka + off, idS, kk > 0 ? 1u : 0u);
                }
            };
            // O_t (+)= P_t V for K/V rows [16*k0, 16*k1) of the tile
            auto issue_PV = [&](int t, uint32_t slot, bool acc, int k0, int k1) {
                const uint64_t va = dV + (opaque(sKV + slot * C::kTile) >> 4);
                const uint32_t d = opaque(tmem + C::colO(t)), a = opaque(tmem + C::colS(t));
#pragma unroll
                for (int kk = k0; kk < k1; ++kk)
                    tc_mma_ts(d, a + kk * 8, va + (kk * 2048 >> 4), idO, (acc || kk > 0) ? 1u : 0u);
            };
            uint32_t kv_it = 0, it = 0, pph0 = 0, pph1 = 0;
            bool ok = true;
            Sched sch;
            sched_init(sch, p);
            Seg g;
            for (; ok && sched_next<CAU>(sch, p, g); ++it) {
                const int nseg = g.j1 - g.j0;
                // causal: query tile 0 of pair p stops at its diagonal K/V tile 2p,
                // one step before tile 1 (which also needs tile 2p + 1)
                const int n0 = CAU ? min(2 * (g.item % p.n_pairs) + 1, nseg) : nseg;
                ok = bwait(BAR(BQ_FULL + 0), it & 1u, abort_flag, kSiteMmaQ) &&
                     bwait(BAR(BQ_FULL + 1), it & 1u, abort_flag, kSiteMmaQ);
                if (!ok) break;
                uint32_t kslot = kv_it % C::kSlots;
                ok = bwait(BAR(BKV_FULL + kslot), (kv_it / C::kSlots) & 1u, abort_flag, kSiteMmaKV);
                if (!ok) break;
                ++kv_it;
                tc_fence_after();
                issue_S(0, kslot);
                tc_commit(BAR(BS_FULL + 0));
                issue_S(1, kslot);
                tc_commit(BAR(BS_FULL + 1));
                tc_commit(BAR(BKV_EMPTY + kslot));
                if (n0 == 1) tc_commit(BAR(BQ_EMPTY + 0));
                if (nseg == 1) tc_commit(BAR(BQ_EMPTY + 1));
                for (int j = 0; j < nseg; ++j) {
                    const uint32_t vslot = kv_it % C::kSlots;
                    const bool more = j + 1 < nseg, more0 = j + 1 < n0;
                    // At D = 96, V_j and K_{j+1} (in long before they are needed) are waited
                    // for together, so that P_0 V_j and S_0 go out as one group: 3.6%
                    // faster there, about 1% slower at D = 64 and 128 (measured on GB300,
                    // builds alternated), where K_{j+1} is waited for between the two.
                    constexpr bool kEarlyK = D == 96;
                    ok = bwait(BAR(BKV_FULL + vslot), (kv_it / C::kSlots) & 1u, abort_flag, kSiteMmaKV);
                    if (kEarlyK && ok && more)
                        ok = bwait(BAR(BKV_FULL + (kv_it + 1) % C::kSlots), ((kv_it + 1) / C::kSlots) & 1u, abort_flag,
                                   kSiteMmaKV);
                    if (!ok) break;
                    ++kv_it;
                    // ---- tile 0: O0 += P0 V_j, then S0 for the next K/V tile
                    if (!CAU || j < n0) {
                        ok = bwait(BAR(BP_FULL + 0), pph0, abort_flag, kSiteMmaP);
                        STEP_TIME(it, 0, j, 2, clock64_now());
                        if (ok && j == 0) ok = bwait(BAR(BO_FREE + 0), (it & 1u) ^ 1u, abort_flag, kSiteMmaOFree);
                        if (!ok) break;
                        pph0 ^= 1u;
                        tc_fence_after();
                        issue_PV(0, vslot, j > 0, 0, 8);
                        STEP_TIME(it, 0, j, 3, clock64_now());
                        if (!more0) tc_commit(BAR(BO_FINAL + 0));
                    }
                    if (more) {
                        kslot = kv_it % C::kSlots;
                        if (!kEarlyK) {
                            ok = bwait(BAR(BKV_FULL + kslot), (kv_it / C::kSlots) & 1u, abort_flag, kSiteMmaKV);
                            if (!ok) break;
                        }
                        ++kv_it;
                        if (more0) {
                            issue_S(0, kslot);
                            tc_commit(BAR(BS_FULL + 0));
                            if (j + 2 == n0) tc_commit(BAR(BQ_EMPTY + 0));
                        }
                    }
                    // ---- tile 1
                    ok = bwait(BAR(BP_FULL + 1), pph1, abort_flag, kSiteMmaP);
                    STEP_TIME(it, 1, j, 2, clock64_now());
                    if (ok && j == 0) ok = bwait(BAR(BO_FREE + 1), (it & 1u) ^ 1u, abort_flag, kSiteMmaOFree);
                    if (!ok) break;
                    pph1 ^= 1u;
                    tc_fence_after();
                    issue_PV(1, vslot, j > 0, 0, 8);
                    STEP_TIME(it, 1, j, 3, clock64_now());
                    tc_commit(BAR(BKV_EMPTY + vslot));
                    if (!more) tc_commit(BAR(BO_FINAL + 1));
                    if (more) {
                        issue_S(1, kslot);
                        tc_commit(BAR(BS_FULL + 1));
                        tc_commit(BAR(BKV_EMPTY + kslot));
                        if (j + 2 == nseg) tc_commit(BAR(BQ_EMPTY + 1));
                    }
                }
            }
            if (!ok) {  // wait (bounded) for MMAs in flight before tensor memory is released
                tc_commit(BAR(B_DRAIN));
                uint32_t dummy = 0;
                const unsigned long long t0 = globaltimer_ns();
                while (!mbar_try_wait(BAR(B_DRAIN), 0) && globaltimer_ns() - t0 < 200000000ull) ++dummy;
            }
        }
        __syncwarp();
    } else if (wg == 1 || wg == 2) {
        // ------------------------------------------------------------- softmax
        setmaxnreg_inc<176>();
        const int t = wg - 1;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::colS(t);
        const uint32_t tO = tmem + lane_base + C::colO(t);
        const int row = (warp & 3) * 32 + lane;
        const float sl2 = p.scale_log2;
        uint32_t sph = 0, it = 0;
        bool ok = true;
        Sched sch;
        sched_init(sch, p);
        Seg g;
        float m = 0.f, l = 0.f;
        bool finish = false;
        for (; ok && sched_next<CAU>(sch, p, g); ++it) {
            // this CTA's last piece of a split item is finished by the softmax
            // warpgroups, after this loop (decided now, while few values are live)
            finish = g.split && sched_done<CAU>(sch, p);
            m = 0.f;
            l = 0.f;
            // causal: this tile's diagonal K/V tile (its last step) is 2p + t
            const int qt_diag = CAU ? 2 * (g.item % p.n_pairs) + t : -1;
            const int nseg = CAU ? min(qt_diag + 1, g.j1 - g.j0) : g.j1 - g.j0;
            const int jmask = RAG && !CAU ? p.n_kv - 1 - g.j0 : -1;  // the step that holds the last K/V tile
            for (int j = 0; j < nseg; ++j) {
                ok = warp_bwait(BAR(BS_FULL + t), sph, abort_flag, kSiteSoftS);
                if (!ok) break;
                if (TRACE && (warp & 3) == 0 && lane == 0) STEP_TIME(it, t, j, 0, clock64_now());
                sph ^= 1u;
                tc_fence_after();
                // this thread's row of S: columns 0-63 in sa, 64-127 in sb
                uint32_t sa[64], sb[64];
#define SV(i) u2f((i) < 64 ? sa[(i) & 63] : sb[(i) & 63])
                if (RAG && !CAU && j == jmask) mask_tail(tS, p.kv_tail);
                tmem_ld64x2(tS, sa, sb);
                if (CAU && j == qt_diag) {
                    // the diagonal tile: keys after this row's token take no weight
                    const uint32_t ninf = f2u(-INFINITY);
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        sa[i] = i > row ? ninf : sa[i];
                        sb[i] = 64 + i > row ? ninf : sb[i];
                    }
                }
                // the row max of S (raw scores)
                auto row_max = [&]() {
                    float mx0 = fmaxf(u2f(sa[0]), u2f(sa[1])), mx1 = fmaxf(u2f(sa[2]), u2f(sa[3]));
                    float mx2 = fmaxf(u2f(sa[4]), u2f(sa[5])), mx3 = fmaxf(u2f(sa[6]), u2f(sa[7]));
#pragma unroll
                    for (int i = 8; i < 64; i += 8) {
                        mx0 = fmax3(mx0, u2f(sa[i + 0]), u2f(sa[i + 1]));
                        mx1 = fmax3(mx1, u2f(sa[i + 2]), u2f(sa[i + 3]));
                        mx2 = fmax3(mx2, u2f(sa[i + 4]), u2f(sa[i + 5]));
                        mx3 = fmax3(mx3, u2f(sa[i + 6]), u2f(sa[i + 7]));
                    }
#pragma unroll
                    for (int i = 0; i < 64; i += 8) {
                        mx0 = fmax3(mx0, u2f(sb[i + 0]), u2f(sb[i + 1]));
                        mx1 = fmax3(mx1, u2f(sb[i + 2]), u2f(sb[i + 3]));
                        mx2 = fmax3(mx2, u2f(sb[i + 4]), u2f(sb[i + 5]));
                        mx3 = fmax3(mx3, u2f(sb[i + 6]), u2f(sb[i + 7]));
                    }
                    return fmax3(mx0, mx1, fmaxf(mx2, mx3));
                };
                // The running max m is taken at the first step only. Later steps use it
                // as it stands and check the row sum of p instead: at most 256 means no
                // p above 2^8, so the max has not passed m + 8 and the rule below would
                // keep m. Results are those of taking the max at every step, but for a
                // step whose only sizeable p lies within rounding of 256.
                if (j == 0) m = row_max() * sl2;
                // p = exp2(s * scale*log2e - m): paired FMAs, ex2, paired sums, bf16 (f16) pairs
                uint32_t pk[64];
                float lstep = 0.f;
                auto exps = [&]() {
                    const uint64_t sc2 = f2pack(sl2, sl2), nm2 = f2pack(-m, -m);
                    uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
                    for (int i = 0; i < 64; i += 2) {
                        const int e = 2 * i;
                        float e0, e1, e2, e3;
                        f2unpack(ffma2(f2pack(SV(e), SV(e + 1)), sc2, nm2), e0, e1);
                        f2unpack(ffma2(f2pack(SV(e + 2), SV(e + 3)), sc2, nm2), e2, e3);
                        e0 = ex2_approx(e0);
                        e1 = ex2_approx(e1);
                        e2 = ex2_approx(e2);
                        e3 = ex2_approx(e3);
                        acc0 = fadd2(acc0, f2pack(e0, e1));
                        acc1 = fadd2(acc1, f2pack(e2, e3));
                        pk[i] = V8 ? pack_f16x2(e0, e1) : pack_bf16x2(e0, e1);
                        pk[i + 1] = V8 ? pack_f16x2(e2, e3) : pack_bf16x2(e2, e3);
                    }
                    float a0, a1;
                    f2unpack(fadd2(acc0, acc1), a0, a1);
                    lstep = a0 + a1;
                };
                exps();
                if (j > 0 && __any_sync(0xffffffffu, !(lstep <= 256.0f))) {
                    // Some row sum passed 256: S is still in TMEM (P has not been
                    // stored), so reload it, take the max, move m where it grew by
                    // more than 8 (rescaling O and l) and redo the exponentials.
                    tmem_ld64x2(tS, sa, sb);
                    if (CAU && j == qt_diag) {
                        const uint32_t ninf = f2u(-INFINITY);
#pragma unroll
                        for (int i = 0; i < 64; ++i) {
                            sa[i] = i > row ? ninf : sa[i];
                            sb[i] = 64 + i > row ? ninf : sb[i];
                        }
                    }
                    const float mnew = row_max() * sl2;
                    float alpha = 1.f;
                    bool need = false;
                    if (mnew > m + 8.0f) {
                        alpha = ex2_approx(m - mnew);
                        m = mnew;
                        need = true;
                    }
                    if (__any_sync(0xffffffffu, need)) {
                        // The commit that signalled S_t for this step also covers the
                        // previous O_t += P V, so O_t is stable here.
#pragma unroll 1
                        for (int c = 0; c < D; c += 32) {
                            uint32_t o[32];
                            tmem_ld32(tO + c, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
                            tmem_st32(tO + c, o);
                        }
                        l *= alpha;
                    }
                    exps();
                }
                l += lstep;
                {
                    uint32_t h0[32], h1[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        h0[i] = pk[i];
                        h1[i] = pk[32 + i];
                    }
                    tmem_st32(tS, h0);
                    tmem_st32(tS + 32, h1);
                }
#undef SV
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (TRACE && (warp & 3) == 0 && lane == 0) STEP_TIME(it, t, j, 1, clock64_now());
                if (lane == 0) mbar_arrive(BAR(BP_FULL + t));
            }
            if (!ok || finish) break;
            ok = warp_bwait(BAR(BL_EMPTY + t), (it & 1u) ^ 1u, abort_flag, kSiteSoftL);
            if (!ok) break;
            row_ml[t * 256 + row] = l;
            row_ml[t * 256 + 128 + row] = m;
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(BL_FULL + t));
        }
        if (ok && finish) {
            // This CTA's last piece of a split item: tile t is finished here, both
            // tiles in parallel, instead of by the epilogue. It is done after the
            // item loop, where the loop's values are dead; inside the loop, next
            // to the softmax's registers, ptxas spilled. Every MMA that reads Q_t
            // is complete once O_t is final, so the query tile's shared memory is
            // free and serves as staging.
            ok = warp_bwait(BAR(BO_FINAL + t), it & 1u, abort_flag, kSiteSoftO);
            if (ok) {
                tc_fence_after();
                const Item w = decode_item(p, g.item);
                const uint32_t ua = (uint32_t)(g.item - p.sk_item0) * (uint32_t)p.n_kv;
                const int c_first = sk_cta_of(ua, p), c_last = sk_cta_of(ua + (uint32_t)p.n_kv - 1u, p);
                const int qt = 2 * w.pair + t;
                const bool valid = qt < p.n_qt;
                // the destination row is computed where it is stored
                auto dst_fn = [&]() { return out_row_offset<D, RAG>(p, w.rb, w.hl, qt * 128 + row); };
                const uint32_t stage = sQ + t * C::kQKTile + (warp & 3) * C::kStageWarp;
                // 64 columns per merge round (32 at D = 96): the merges of the balanced
                // tail end the kernel, so their load latency is on its critical path
                constexpr int CH = D % 64 ? 32 : 64;
                // The piece always goes to the workspace and the last of the item's
                // pieces to arrive merges them all from there. Merging at once from
                // tensor memory when the others are in saves about 3 us at DiT size,
                // but next to the softmax's registers ptxas then spilled.
                finish_piece<D, CH, RAG, false>(p, g, t, warp & 3, row, lane, stage, c_first, c_last, ua, m, l, tO,
                                                dst_fn, valid, [] {});
                __threadfence();
                __syncwarp();
                arrive_piece<D, CH, RAG>(p, g, t, warp & 3, row, lane, stage, c_first, c_last, ua, dst_fn, valid);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        setmaxnreg_dec<112>();
        // columns per merge round of a split item's pieces (16 at D = 96, where 32
        // made the epilogue spill at 112 registers)
        constexpr int kEpiMergeCols = D == 96 ? 16 : 32;
        const int wq = warp & 3;
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const int row = wq * 32 + lane;
        const uint32_t stage = sStage + wq * C::kStageWarp;
        uint32_t it = 0;
        bool ok = true;
        Sched sch;
        sched_init(sch, p);
        Seg g;
        for (; ok && sched_next<CAU>(sch, p, g); ++it) {
            // a CTA's last piece of a split item is finished by the softmax warpgroups
            if (g.split && sched_done<CAU>(sch, p)) continue;
            const Item w = decode_item(p, g.item);
            const uint32_t ua = (uint32_t)(g.item - p.sk_item0) * (uint32_t)p.n_kv;  // a split item's first unit
            int c_first = 0, c_last = 0;
            if (g.split) {
                c_first = sk_cta_of(ua, p);
                c_last = sk_cta_of(ua + (uint32_t)p.n_kv - 1u, p);
            }
            uint32_t pending = 0;  // tiles whose rows went to the workspace
            for (int t = 0; t < 2; ++t) {
                ok = warp_bwait(BAR(BO_FINAL + t), it & 1u, abort_flag, kSiteEpiO) &&
                     warp_bwait(BAR(BL_FULL + t), it & 1u, abort_flag, kSiteEpiL);
                if (!ok) break;
                const float l = row_ml[t * 256 + row];
                const float m = row_ml[t * 256 + 128 + row];
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(BL_EMPTY + t));
                tc_fence_after();
                const int qt = 2 * w.pair + t;
                const bool valid = qt < p.n_qt;
                const int64_t dst = out_row_offset<D, RAG>(p, w.rb, w.hl, qt * 128 + row);
                const uint32_t tO = tmem + lane_base + C::colO(t);
                auto release_o = [&]() {  // O_t fully read: the next item may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(BO_FREE + t));
                };
                if (g.split) {
                    auto dst_fn = [&]() { return out_row_offset<D, RAG>(p, w.rb, w.hl, qt * 128 + row); };
                    pending |= finish_piece<D, kEpiMergeCols, RAG, true>(p, g, t, wq, row, lane, stage, c_first, c_last,
                                                                        ua, m, l, tO, dst_fn, valid, release_o)
                               << t;
                    continue;
                }
                const float inv_l = 1.0f / l;
                unsigned long long t_ready = 0, t_store = 0, g_ready = 0;
                if (TRACE) {
                    t_ready = clock64_now();
                    g_ready = globaltimer_ns();
                }
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    // 32 columns per round into the staged rows; a full 128-byte row
                    // block (or the half block of D = 96) is then stored
                    uint32_t o[32];
                    tmem_ld32(tO + c0, o);
                    if (c0 + 32 == D) release_o();
                    if (!valid) continue;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        stage_chunk(stage, lane, (c0 % 64) / 8 + c,
                                    pack_bf16x2(u2f(o[8 * c + 0]) * inv_l, u2f(o[8 * c + 1]) * inv_l),
                                    pack_bf16x2(u2f(o[8 * c + 2]) * inv_l, u2f(o[8 * c + 3]) * inv_l),
                                    pack_bf16x2(u2f(o[8 * c + 4]) * inv_l, u2f(o[8 * c + 5]) * inv_l),
                                    pack_bf16x2(u2f(o[8 * c + 6]) * inv_l, u2f(o[8 * c + 7]) * inv_l));
                    if (TRACE && c0 == 32) t_store = clock64_now();
                    if ((c0 + 32) % 64 == 0)
                        flush_block<RAG>(p.out, stage, lane, dst, c0 / 64);
                    else if (c0 + 32 == D)  // the half block of D = 96
                        flush_block<RAG, 4>(p.out, stage, lane, dst, c0 / 64);
                }
                if (TRACE && lane == 0) {
                    const unsigned long long t_end = clock64_now();
                    unsigned long long *r =
                        p.trace + (((size_t)blockIdx.x * p.n_dp + it) * 8 + t * 4 + wq) * kTraceWords;
                    r[0] = t_ready;
                    r[1] = valid ? t_store : t_end;
                    r[2] = t_end;
                    r[3] = g_ready;
                    r[4] = ((unsigned long long)g.item << 8) | (uint32_t)(t << 4) | (valid ? 0u : 8u) | (uint32_t)wq;
                }
            }
            if (!ok || !pending) continue;
            // count this piece's arrival for the published tiles; the last arrival merges
            __threadfence();
            __syncwarp();
            for (int t = 0; t < 2; ++t) {
                if (!(pending & (1u << t))) continue;
                const int qt = 2 * w.pair + t;
                arrive_piece<D, kEpiMergeCols, RAG>(p, g, t, wq, row, lane, stage, c_first, c_last, ua,
                                         [&]() { return out_row_offset<D, RAG>(p, w.rb, w.hl, qt * 128 + row); },
                                         qt < p.n_qt);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if (TRACE && threadIdx.x == 0) cta_times[3] = globaltimer_ns();
#undef STEP_TIME
#undef BAR
}

template <int D, int LD, int TRACE, bool RAG, bool CAU = false, int F8 = 0>
static cudaError_t launch_one(const OperandMaps<LD ? kSeqMaps : 1> &maps, const AttnParams &p, int grid,
                              cudaStream_t stream) {
    auto kern = attn_fwd_kernel<D, LD, TRACE, RAG, CAU, F8>;
    using CQ = Cfg<D, F8>;
    // The shared-memory limit is raised once per device and instance: setting a
    // function attribute before every launch makes each launch start much later.
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CQ::kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    kern<<<grid, 512, CQ::kSmemAlloc, stream>>>(maps, p);
    e = cudaGetLastError();
    if (e == cudaErrorInvalidValue || e == cudaErrorLaunchOutOfResources) {
        // the attribute was lost (for instance by a device reset): set it again once
        configured.fetch_and(~bit, std::memory_order_acq_rel);
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)CQ::kSmemAlloc)) != cudaSuccess)
            return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
        kern<<<grid, 512, CQ::kSmemAlloc, stream>>>(maps, p);
        e = cudaGetLastError();
    }
    return e;
}

// The ragged instances (S not a multiple of 128) carry the key mask and the
// row guard; the others compile without them.
template <int D, int LD>
static cudaError_t launch_t(const OperandMaps<LD ? kSeqMaps : 1> &maps, const AttnParams &p, int grid,
                            cudaStream_t stream) {
    return p.kv_tail < 128 ? launch_one<D, LD, 0, true>(maps, p, grid, stream)
                           : launch_one<D, LD, 0, false>(maps, p, grid, stream);
}


// Per-head-dimension entry points; each xs_attn_d<D>.cu instantiates one set.
#define XS_DEFINE_ATTN_ENTRY(D)                                                                                   \
    cudaError_t launch_attention_d##D(const OperandMaps<1> &maps, const AttnParams &p, int grid,                   \
                                      cudaStream_t stream) {                                                      \
        return launch_t<D, 0>(maps, p, grid, stream);                                                             \
    }                                                                                                             \
    cudaError_t launch_ulysses_d##D(const OperandMaps<kSeqMaps> &maps, const AttnParams &p, int grid,             \
                                    cudaStream_t stream) {                                                        \
        return launch_t<D, 1>(maps, p, grid, stream);                                                             \
    }                                                                                                             \
    cudaError_t launch_causal_d##D(const OperandMaps<1> &maps, const AttnParams &p, int grid,                      \
                                   cudaStream_t stream) {                                                         \
        return launch_one<D, 0, 0, true, true>(maps, p, grid, stream);                                             \
    }                                                                                                             \
    cudaError_t read_error_word_d##D(unsigned int *value, bool clear) {                                           \
        cudaError_t e = cudaMemcpyFromSymbol(value, g_xs_error, sizeof(unsigned int));                            \
        if (e == cudaSuccess && clear && *value) {                                                                \
            const unsigned int zero = 0;                                                                          \
            e = cudaMemcpyToSymbol(g_xs_error, &zero, sizeof(unsigned int));                                      \
        }                                                                                                         \
        return e;                                                                                                 \
    }

}  // namespace xs
