// xs_attn1_kernel.cuh -- the single-query-tile variant of the attention kernel
// for sm_103a, used for head dimension 256: persistent, warp-specialised, with
// the same epilogue choices (head-partitioned, or straight into the
// post-attention All-to-All layout) as xs_attn_kernel.cuh.
//
// What it computes (X-Stage paper, arXiv 2607.23264v1):
//   * section 4.3, Figure 6: a CTA owns 128 query rows of one head and walks all
//     ceil(S/128) K/V tiles (the Q-loop); finishing the walk yields a 128 x D
//     output tile, and successive output tiles form the outer loop;
//   * section 4.3, Figure 7: at an output-tile boundary the role that owns O
//     issues that tile's stores, then the next tile's Q-loop runs while those
//     stores drain; no warp or SM is reserved for communication;
//   * section 4.3, Figure 5: the destination is the Ulysses sequence partition,
//     and optionally (LD = 1) Q, K and V are read from it too.
//
// Why a second variant: with D = 256 two query tiles do not fit, since each
// needs a 256-column O accumulator in tensor memory (512 columns in all).
// One tile with a double-buffered score matrix does:
//   tensor memory  S_0 | S_1 (128 columns each; P overwrites the first 64) | O (256)
// The MMA issuer runs S_{j+1} = Q K_{j+1}^T into the other score buffer before
// O += P_j V_j, so the tensor cores work on the next step while the softmax
// works on this one. With D = 256 the MMA work of a step (about 2250 cycles)
// exceeds the softmax's, so the loop is bound by the tensor cores. (For D <= 128
// the two-tile kernel is faster: there the softmax, not the MMA, bounds a step,
// and two tiles let two softmax warpgroups run at once.)
//
// Roles (512 threads, one CTA per SM): warp 0 TMA producer (Q, then K_0 and, per
// step, K_{j+1} before V_j, the order the MMA issuer consumes them); warp 1 the
// MMA issuer; warp 2 allocates tensor memory; warps 4-7 softmax (one thread per
// row); warps 8-11 give their registers away; warps 12-15 epilogue. Online
// softmax in base 2 with the stale-max rule of the two-tile kernel; the rare O
// rescale first waits for the previous step's P V (a per-step commit barrier),
// since this step's S was issued ahead of it.
//
// Schedule, split pieces, bounded waits: as in the two-tile kernel, with an
// item being one query tile. Every mbarrier wait is bounded in time.
#pragma once

#include <atomic>

#include "xs_internal.h"
#include "xs_ptx.cuh"

namespace xs {
namespace one {

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


template <int D> struct Cfg {
    static_assert(D == 64 || D == 96 || D == 128 || D == 256, "head dimension");
    // 64-column (128-byte) swizzle blocks per row; with D = 96 the second block
    // is half used (TMA zero-fills its other half)
    static constexpr int kNDB = (D + 63) / 64;
    static constexpr uint32_t kBlk = 128u * 128u;       // one swizzle block of a 128-row tile
    static constexpr uint32_t kTile = kNDB * kBlk;      // a 128-row Q, K or V tile in shared memory
    static constexpr int kSlots = D > 128 ? 2 : 4;      // K/V ring slots
    // O accumulators in tensor memory: two (items alternate, so the epilogue drains
    // one while the next item computes) unless D = 256 fills the space with one
    static constexpr int kOBufs = D > 128 ? 1 : 2;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffKV = kOffQ + kTile;
    static constexpr uint32_t kOffStage = kOffKV + kSlots * kTile;
    static constexpr uint32_t kStageWarp = 32u * 128u;  // 32 rows x 64 bf16 per epilogue warp
    static constexpr uint32_t kOffBar = kOffStage + 4 * kStageWarp;
    static constexpr int kNumBars = 24;
    static constexpr uint32_t kOffL = kOffBar + 8 * 32;        // float [O buffer][l, m][128]
    static constexpr uint32_t kOffMisc = kOffL + 2 * 2 * 128 * 4;  // tmem base, abort flag
    static constexpr uint32_t kSmemUsed = kOffMisc + 16;
    static constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;  // slack to align the base to 1024
    // Tensor memory (512 columns): S_0 | S_1 (double-buffered scores, P over the
    // first 64 columns of each) | O_0 | O_1 (D columns each; one of 256 for D = 256)
    __host__ __device__ static constexpr uint32_t colS(int b) { return 128u * (uint32_t)b; }
    __host__ __device__ static constexpr uint32_t colO(int ob) { return 256u + (uint32_t)D * (uint32_t)ob; }
    static constexpr uint32_t kTmemCols = 512;
    static_assert(256 + kOBufs * D <= 512, "tensor memory budget");
    static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

// mbarrier slots
enum : int {
    BQ_FULL = 0, BQ_EMPTY = 1, BKV_FULL = 2, BKV_EMPTY = 6, BS_FULL = 10, BP_FULL = 12, BPV_DONE = 14,
    BO_FINAL = 15, BO_FREE = 17, BL_FULL = 19, BL_EMPTY = 21, B_DRAIN = 23
};

struct Item {
    int rb, hl, qt;  // rank * B + batch, local head, 128-row query tile
};
__device__ __forceinline__ Item decode_item(const AttnParams &p, int item) {
    Item it;
    item += p.item0;  // scheduler items are local to the call's rank range
    it.qt = item % p.n_qt;
    const int head = item / p.n_qt;
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
// CAU (causal): item lengths differ (query tile qt needs qt + 1 K/V tiles), so
// whole items go out longest first, dealt to the CTAs in a snake order (wave w
// runs CTA 0..G-1 when w is even and G-1..0 when odd), a longest-processing-time
// assignment that keeps the CTAs' totals close.
template <bool CAU>
__device__ __forceinline__ bool sched_next(Sched &s, const AttnParams &p, Seg &g) {
    if (CAU) {
        const int G = (int)gridDim.x, n_heads = p.n_items / p.n_qt;
        while (s.k < p.n_dp) {
            const int w = s.k++;
            const int rank = w * G + ((w & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
            if (rank >= p.n_items) continue;
            const int qt = p.n_qt - 1 - rank / n_heads;
            g.item = (rank % n_heads) * p.n_qt + qt;
            g.j0 = 0;
            g.j1 = qt + 1;
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
// Floats in one partial record: the unnormalised O of the item's tile as
// [D/4][128 rows][4], then [row max, row sum][128].
template <int D> struct Rec {
    static constexpr size_t kFloats = 128 * D + 2 * 128;
    static constexpr size_t kML = 128 * D;
};

// Record of the piece of the split item starting at unit ua that CTA c computed.
__device__ __forceinline__ const float *piece_record(const AttnParams &p, int c, uint32_t ua, size_t rec_floats) {
    const int slot = 2 * c + (sk_start((uint32_t)c, p) >= ua ? 0 : 1);
    return p.ws_rec + (size_t)slot * rec_floats;
}

// Merge of a split item's pieces for one warp's 32 rows, in piece order, and
// the store of the final rows. With self_tmem the piece computed by
// this CTA is read from tensor memory (it never went to the workspace);
// otherwise every piece, this CTA's included, comes from the workspace. Both
// read the same bits, so the result does not depend on which piece merges.
// CH columns (32 or 64) are gathered per round.
template <int D, int CH, bool RAG>
__device__ __forceinline__ void merge_rows(const AttnParams &p, int row, int lane, uint32_t stage, int c_first,
                                           int c_last, uint32_t ua, bool self_tmem, float m_self, float l_self,
                                           uint32_t tO, int64_t dst, bool valid) {
    using R = Rec<D>;
    const int self = (int)blockIdx.x;
    float M = -INFINITY;
    for (int c = c_first; c <= c_last; ++c)
        M = fmaxf(M, (self_tmem && c == self) ? m_self
                                             : ld_cg(piece_record(p, c, ua, R::kFloats) + R::kML + row));
    float L = 0.f;
    for (int c = c_first; c <= c_last; ++c) {
        float mc, lc;
        if (self_tmem && c == self) {
            mc = m_self;
            lc = l_self;
        } else {
            const float *r = piece_record(p, c, ua, R::kFloats) + R::kML;
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
            if (self_tmem && c == self) {
                const float wk = ex2_approx(m_self - M);
#pragma unroll
                for (int h = 0; h < CH; h += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + col0 + h, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[h + i] = fmaf(wk, __uint_as_float(o[i]), acc[h + i]);
                }
            } else {
                const float *r = piece_record(p, c, ua, R::kFloats);
                const float wk = ex2_approx(ld_cg(r + R::kML + row) - M);
                const float4 *src = reinterpret_cast<const float4 *>(r);
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
                flush_block<RAG>(p.out, stage, lane, dst, col0 / 64);
            else if (col0 + CH == D)  // the half block of D = 96
                flush_block<RAG, 4>(p.out, stage, lane, dst, col0 / 64);
        }
    }
}

// One warp's 32 rows of a split piece, after its last PV: either
// merge now (every other piece already arrived; this piece is read from
// TMEM) and return 0, or publish this piece's rows (unnormalised O, row max,
// row sum) to the workspace and return 1: the caller must then count the
// arrival with arrive_piece. `release` runs once the rows are out of TMEM.
template <int D, int CH, bool RAG, typename Release>
__device__ __forceinline__ uint32_t finish_piece(const AttnParams &p, const Seg &g, int wq, int row, int lane,
                                                 uint32_t stage, int c_first, int c_last, uint32_t ua, float m, float l,
                                                 uint32_t tO, int64_t dst, bool valid, Release release) {
    using R = Rec<D>;
    const uint32_t x_local = (uint32_t)(g.item - p.sk_item0);
    const uint32_t npieces = (uint32_t)(c_last - c_first + 1);
    const unsigned long long *cnt = p.ws_cnt + ((size_t)x_local * 4 + wq);
    uint32_t others = 0;
    if (lane == 0) others = arrivals_now(cnt, p.gen) == npieces - 1u ? 1u : 0u;
    others = __shfl_sync(0xffffffffu, others, 0);
    if (others) {
        __threadfence();
        merge_rows<D, CH, RAG>(p, row, lane, stage, c_first, c_last, ua, true, m, l, tO, dst, valid);
        release();
        return 0;
    }
    const int own_slot = 2 * (int)blockIdx.x + (g.first ? 0 : 1);
    float *rec = p.ws_rec + (size_t)own_slot * R::kFloats;
    float4 *o4 = reinterpret_cast<float4 *>(rec);
#pragma unroll 1
    for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(tO + c, o);
        if (c + 32 == D) release();
#pragma unroll
        for (int q = 0; q < 8; ++q)
            o4[(size_t)(c / 4 + q) * 128 + row] = make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                                              __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
    }
    rec[R::kML + row] = m;
    rec[R::kML + 128 + row] = l;
    return 1;
}

// Counts this piece's arrival for one warp's rows (after they were published
// and fenced); the last arrival merges from the workspace.
template <int D, int CH, bool RAG>
__device__ __forceinline__ void arrive_piece(const AttnParams &p, const Seg &g, int wq, int row, int lane,
                                             uint32_t stage, int c_first, int c_last, uint32_t ua, int64_t dst,
                                             bool valid) {
    const uint32_t x_local = (uint32_t)(g.item - p.sk_item0);
    uint32_t last = 0;
    if (lane == 0)
        last = arrive_last(p.ws_cnt + ((size_t)x_local * 4 + wq), p.gen, (uint32_t)(c_last - c_first + 1))
                   ? 1u
                   : 0u;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    merge_rows<D, CH, RAG>(p, row, lane, stage, c_first, c_last, ua, false, 0.f, 0.f, 0u, dst, valid);
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

template <int D, int LD, int TRACE, bool RAG, bool CAU>
__global__ void __launch_bounds__(512, 1)
    attn_fwd_kernel(const __grid_constant__ OperandMaps<LD ? kSeqMaps : 1> tm, const AttnParams p) {
    using C = Cfg<D>;
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
        TRACE ? p.trace + ((size_t)gridDim.x * p.n_dp * 4 + (size_t)blockIdx.x * 4) * kTraceWords : nullptr;
    if (TRACE && threadIdx.x == 0) cta_times[0] = globaltimer_ns();

    if (threadIdx.x == 0) {
        mbar_init(BAR(BQ_FULL), 1);
        mbar_init(BAR(BQ_EMPTY), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(BAR(BS_FULL + b), 1);
            mbar_init(BAR(BP_FULL + b), 4);
            mbar_init(BAR(BO_FINAL + b), 1);
            mbar_init(BAR(BO_FREE + b), 4);
            mbar_init(BAR(BL_FULL + b), 4);
            mbar_init(BAR(BL_EMPTY + b), 4);
        }
        mbar_init(BAR(BPV_DONE), 1);
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(BAR(BKV_FULL + s), 1);
            mbar_init(BAR(BKV_EMPTY + s), 1);
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
            // Per item: Q, then K_0 and, for each step j, K_{j+1} before V_j (the
            // order in which the MMA issuer consumes them).
            uint32_t kv_it = 0, it = 0;
            bool ok = true;
            Sched sch;
            sched_init(sch, p);
            Seg g;
            auto load_kv = [&](const Item &w, int b, int h, bool kv, int jg) -> bool {
                const uint32_t slot = kv_it % C::kSlots, ph = (kv_it / C::kSlots) & 1u;
                ++kv_it;
                if (!bwait(BAR(BKV_EMPTY + slot), ph ^ 1u, abort_flag, kSiteLoadKV)) return false;
                mbar_arrive_expect_tx(BAR(BKV_FULL + slot), C::kTile);
                const CUtensorMap *m = kv ? tm.v : tm.k;
                if (LD) {
                    int rs, sl;
                    seq_position(p, jg * 128, rs, sl);
                    load_rows_seq<D>(sKV + slot * C::kTile, m, BAR(BKV_FULL + slot), p, b, h, rs, sl);
                } else {
                    load_rows_head<D>(sKV + slot * C::kTile, m, BAR(BKV_FULL + slot), w.rb, w.hl, jg * 128);
                }
                return true;
            };
            for (; ok && sched_next<CAU>(sch, p, g); ++it) {
                const Item w = decode_item(p, g.item);
                // sequence-partitioned inputs: batch and global head of the item
                const int b = LD ? w.rb % p.B : 0, h = LD ? (w.rb / p.B) * p.Hl + w.hl : 0;
                ok = bwait(BAR(BQ_EMPTY), (it & 1u) ^ 1u, abort_flag, kSiteLoadQ);
                if (!ok) break;
                mbar_arrive_expect_tx(BAR(BQ_FULL), C::kTile);
                if (TRACE && it == 0) cta_times[2] = globaltimer_ns();
                if (LD) {
                    int rs, sl;
                    seq_position(p, w.qt * 128, rs, sl);
                    load_rows_seq<D>(sQ, tm.q, BAR(BQ_FULL), p, b, h, rs, sl);
                } else {
                    load_rows_head<D>(sQ, tm.q, BAR(BQ_FULL), w.rb, w.hl, w.qt * 128);
                }
                const int nseg = g.j1 - g.j0;
                ok = load_kv(w, b, h, false, g.j0);
                for (int j = 0; ok && j < nseg; ++j) {
                    if (j + 1 < nseg) ok = load_kv(w, b, h, false, g.j0 + j + 1);
                    if (ok) ok = load_kv(w, b, h, true, g.j0 + j);
                }
            }
            if (!ok) {  // let copies already in flight land before the CTA exits
                const unsigned long long t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------------- MMA issuer
            // Per item: S_0, then for each step j: S_{j+1} into the other score
            // buffer, then O += P_j V_j once the softmax has handed P_j over. The
            // next step's QK^T therefore runs while the softmax of this step does.
            constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0);
            constexpr uint32_t idO = idesc_bf16_f32(128, D, 1);
            // Descriptors differ only in the start-address field (address >> 4 in
            // the low 14 bits), so each MMA adds a compile-time offset to a base.
            const uint64_t dK = sdesc_sw128(0, 16, 1024);       // K-major, 128-byte rows
            const uint64_t dV = sdesc_sw128(0, C::kBlk, 1024);  // MN-major V, 64-column blocks kBlk apart
            auto issue_S = [&](uint32_t b, uint32_t slot) {
                const uint64_t qa = dK + (opaque(sQ) >> 4);
                const uint64_t ka = dK + (opaque(sKV + slot * C::kTile) >> 4);
                const uint32_t d = opaque(tmem + C::colS(b));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kBlk + (kk & 3) * 32) >> 4;
                    tc_mma_ss(d, qa + off, ka + off, idS, kk > 0 ? 1u : 0u);
                }
            };
            // O (+)= P_b V for the 128 keys of the K/V tile
            auto issue_PV = [&](uint32_t ob, uint32_t b, uint32_t slot, bool acc) {
                const uint64_t va = dV + (opaque(sKV + slot * C::kTile) >> 4);
                const uint32_t d = opaque(tmem + C::colO(ob)), a = opaque(tmem + C::colS(b));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_ts(d, a + kk * 8, va + (kk * 2048 >> 4), idO, (acc || kk > 0) ? 1u : 0u);
            };
            uint32_t kv_it = 0, it = 0, sb = 0, pph = 0;  // pph: P handoff phase per score buffer (bits)
            bool ok = true;
            Sched sch;
            sched_init(sch, p);
            Seg g;
            auto kv_wait = [&](uint32_t &slot) -> bool {
                slot = kv_it % C::kSlots;
                const uint32_t ph = (kv_it / C::kSlots) & 1u;
                ++kv_it;
                return bwait(BAR(BKV_FULL + slot), ph, abort_flag, kSiteMmaKV);
            };
            for (; ok && sched_next<CAU>(sch, p, g); ++it) {
                const int nseg = g.j1 - g.j0;
                const uint32_t ob = C::kOBufs == 2 ? (it & 1u) : 0u;
                const uint32_t ouse = C::kOBufs == 2 ? (it >> 1) : it;  // uses of O buffer ob before this item
                ok = bwait(BAR(BQ_FULL), it & 1u, abort_flag, kSiteMmaQ);
                if (!ok) break;
                uint32_t kslot, vslot;
                ok = kv_wait(kslot);
                if (!ok) break;
                tc_fence_after();
                issue_S(sb & 1u, kslot);
                tc_commit(BAR(BS_FULL + (sb & 1u)));
                tc_commit(BAR(BKV_EMPTY + kslot));
                ++sb;
                if (nseg == 1) tc_commit(BAR(BQ_EMPTY));
                for (int j = 0; j < nseg; ++j) {
                    const uint32_t bj = (sb - 1u) & 1u;  // score buffer of step j
                    if (j + 1 < nseg) {
                        ok = kv_wait(kslot);
                        if (!ok) break;
                        tc_fence_after();
                        issue_S(sb & 1u, kslot);
                        tc_commit(BAR(BS_FULL + (sb & 1u)));
                        tc_commit(BAR(BKV_EMPTY + kslot));
                        ++sb;
                        if (j + 2 == nseg) tc_commit(BAR(BQ_EMPTY));
                    }
                    ok = kv_wait(vslot) && bwait(BAR(BP_FULL + bj), (pph >> bj) & 1u, abort_flag, kSiteMmaP);
                    if (ok && j == 0) ok = bwait(BAR(BO_FREE + ob), (ouse & 1u) ^ 1u, abort_flag, kSiteMmaOFree);
                    if (!ok) break;
                    pph ^= 1u << bj;
                    tc_fence_after();
                    issue_PV(ob, bj, vslot, j > 0);
                    tc_commit(BAR(BKV_EMPTY + vslot));
                    tc_commit(BAR(BPV_DONE));
                    if (j + 1 == nseg) tc_commit(BAR(BO_FINAL + ob));
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
    } else if (wg == 1) {
        // ------------------------------------------------------------- softmax
        setmaxnreg_inc<232>();
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int row = (warp & 3) * 32 + lane;
        const float sl2 = p.scale_log2;
        uint32_t sph = 0, sb = 0, npv = 0, it = 0;  // sph: S phase per score buffer (bits); npv: PVs so far
        bool ok = true;
        Sched sch;
        sched_init(sch, p);
        Seg g;
        for (; ok && sched_next<CAU>(sch, p, g); ++it) {
            const uint32_t ob = C::kOBufs == 2 ? (it & 1u) : 0u;
            const uint32_t ouse = C::kOBufs == 2 ? (it >> 1) : it;
            const uint32_t tO = tmem + lane_base + C::colO(ob);
            float m = 0.f, l = 0.f;
            const int nseg = g.j1 - g.j0;
            const int qt_diag = CAU ? g.item % p.n_qt : -1;  // causal: the item's diagonal K/V tile
            for (int j = 0; j < nseg; ++j, ++sb) {
                const uint32_t b = sb & 1u;
                ok = warp_bwait(BAR(BS_FULL + b), (sph >> b) & 1u, abort_flag, kSiteSoftS);
                if (!ok) break;
                sph ^= 1u << b;
                tc_fence_after();
                const uint32_t tS = tmem + lane_base + C::colS(b);
                // this thread's row of S: columns 0-63 in sa, 64-127 in sb
                uint32_t sa[64], sbv[64];
#define SV(i) u2f((i) < 64 ? sa[(i) & 63] : sbv[(i) & 63])
                if (RAG && !CAU && g.j0 + j == p.n_kv - 1) {
                    // keys past S (zero-filled rows of the last K/V tile) take no
                    // weight: their scores become -inf in tensor memory
#pragma unroll 1
                    for (int c = p.kv_tail; c < 128; ++c) tmem_st1(tS + (uint32_t)c, f2u(-INFINITY));
                    tmem_st_wait();
                }
                tmem_ld64(tS, sa);
                tmem_ld64(tS + 64, sbv);
                if (CAU && j == qt_diag) {
                    // the diagonal tile: keys after this row's token take no weight
                    const uint32_t ninf = f2u(-INFINITY);
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        sa[i] = i > row ? ninf : sa[i];
                        sbv[i] = 64 + i > row ? ninf : sbv[i];
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
                        mx0 = fmax3(mx0, u2f(sbv[i + 0]), u2f(sbv[i + 1]));
                        mx1 = fmax3(mx1, u2f(sbv[i + 2]), u2f(sbv[i + 3]));
                        mx2 = fmax3(mx2, u2f(sbv[i + 4]), u2f(sbv[i + 5]));
                        mx3 = fmax3(mx3, u2f(sbv[i + 6]), u2f(sbv[i + 7]));
                    }
                    return fmax3(mx0, mx1, fmaxf(mx2, mx3));
                };
                // The running max m is taken at the first step only. Later steps use it
                // as it stands and check the row sum of p instead: at most 256 means no
                // p above 2^8, so the max has not passed m + 8 and the rule below would
                // keep m. Results are those of taking the max at every step, but for a
                // step whose only sizeable p lies within rounding of 256.
                if (j == 0) m = row_max() * sl2;
                // p = exp2(s * scale*log2e - m): paired FMAs, ex2, paired sums, bf16 pairs
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
                        pk[i] = pack_bf16x2(e0, e1);
                        pk[i + 1] = pack_bf16x2(e2, e3);
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
                    tmem_ld64(tS, sa);
                    tmem_ld64(tS + 64, sbv);
                    if (CAU && j == qt_diag) {
                        const uint32_t ninf = f2u(-INFINITY);
#pragma unroll
                        for (int i = 0; i < 64; ++i) {
                            sa[i] = i > row ? ninf : sa[i];
                            sbv[i] = 64 + i > row ? ninf : sbv[i];
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
                        // O must hold the previous step's P V before it is rescaled: the
                        // step's S was issued ahead of that PV. It is the PV count npv +
                        // j - 1 (0-based) and at most one phase ahead of this wait.
                        ok = warp_bwait(BAR(BPV_DONE), (npv + (uint32_t)j - 1u) & 1u, abort_flag, kSiteSoftO);
                        if (!ok) break;
                        tc_fence_after();
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
                if (lane == 0) mbar_arrive(BAR(BP_FULL + b));
            }
            if (!ok) break;
            npv += (uint32_t)nseg;
            if (g.split && sched_done<CAU>(sch, p)) {
                // This CTA's last piece of a split item: finish it here instead of
                // handing it to the epilogue. Every MMA of the CTA is complete once
                // O is final, so the query tile's shared memory is free and serves
                // as staging.
                ok = warp_bwait(BAR(BO_FINAL + ob), ouse & 1u, abort_flag, kSiteSoftO);
                if (!ok) break;
                tc_fence_after();
                const Item w = decode_item(p, g.item);
                const uint32_t ua = (uint32_t)(g.item - p.sk_item0) * (uint32_t)p.n_kv;
                const int c_first = sk_cta_of(ua, p), c_last = sk_cta_of(ua + (uint32_t)p.n_kv - 1u, p);
                const int64_t dst = out_row_offset<D, RAG>(p, w.rb, w.hl, w.qt * 128 + row);
                const uint32_t stage = sQ + (warp & 3) * C::kStageWarp;
                const uint32_t pend = finish_piece<D, D % 64 ? 32 : 64, RAG>(p, g, warp & 3, row, lane, stage,
                                                                             c_first, c_last, ua, m, l, tO, dst,
                                                                             true, [] {});
                if (pend) {
                    __threadfence();
                    __syncwarp();
                    arrive_piece<D, D % 64 ? 32 : 64, RAG>(p, g, warp & 3, row, lane, stage, c_first, c_last, ua,
                                                           dst, true);
                }
                continue;
            }
            ok = warp_bwait(BAR(BL_EMPTY + ob), (ouse & 1u) ^ 1u, abort_flag, kSiteSoftL);
            if (!ok) break;
            row_ml[ob * 256 + row] = l;
            row_ml[ob * 256 + 128 + row] = m;
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(BL_FULL + ob));
        }
    } else if (wg == 2) {
        // spare warpgroup: hands its registers to the softmax and the epilogue
        setmaxnreg_dec<24>();
    } else {
        // ------------------------------------------------------------ epilogue
        setmaxnreg_inc<208>();
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
            // a CTA's last piece of a split item is finished by the softmax warpgroup
            if (g.split && sched_done<CAU>(sch, p)) continue;
            const uint32_t ob = C::kOBufs == 2 ? (it & 1u) : 0u;
            const uint32_t ouse = C::kOBufs == 2 ? (it >> 1) : it;
            const Item w = decode_item(p, g.item);
            const uint32_t ua = (uint32_t)(g.item - p.sk_item0) * (uint32_t)p.n_kv;  // a split item's first unit
            int c_first = 0, c_last = 0;
            if (g.split) {
                c_first = sk_cta_of(ua, p);
                c_last = sk_cta_of(ua + (uint32_t)p.n_kv - 1u, p);
            }
            ok = warp_bwait(BAR(BO_FINAL + ob), ouse & 1u, abort_flag, kSiteEpiO) &&
                 warp_bwait(BAR(BL_FULL + ob), ouse & 1u, abort_flag, kSiteEpiL);
            if (!ok) break;
            const float l = row_ml[ob * 256 + row];
            const float m = row_ml[ob * 256 + 128 + row];
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(BL_EMPTY + ob));
            tc_fence_after();
            const int64_t dst = out_row_offset<D, RAG>(p, w.rb, w.hl, w.qt * 128 + row);
            const uint32_t tO = tmem + lane_base + C::colO(ob);
            auto release_o = [&]() {  // O fully read: a later item may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(BO_FREE + ob));
            };
            if (g.split) {
                const uint32_t pend = finish_piece<D, 32, RAG>(p, g, wq, row, lane, stage, c_first, c_last, ua, m,
                                                               l, tO, dst, true, release_o);
                if (pend) {
                    // count this piece's arrival; the last arrival merges
                    __threadfence();
                    __syncwarp();
                    arrive_piece<D, 32, RAG>(p, g, wq, row, lane, stage, c_first, c_last, ua, dst, true);
                }
                continue;
            }
            const float inv_l = 1.0f / l;
            unsigned long long t_ready = 0, t_store = 0, g_ready = 0;
            if (TRACE) {
                t_ready = clock64_now();
                g_ready = globaltimer_ns();
            }
#pragma unroll 1
            for (int db = 0; db < D / 64; ++db) {
                uint32_t o[64];
                tmem_ld64(tO + db * 64, o);
                if (db == C::kNDB - 1) release_o();
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    stage_chunk(stage, lane, c, pack_bf16x2(u2f(o[8 * c + 0]) * inv_l, u2f(o[8 * c + 1]) * inv_l),
                                pack_bf16x2(u2f(o[8 * c + 2]) * inv_l, u2f(o[8 * c + 3]) * inv_l),
                                pack_bf16x2(u2f(o[8 * c + 4]) * inv_l, u2f(o[8 * c + 5]) * inv_l),
                                pack_bf16x2(u2f(o[8 * c + 6]) * inv_l, u2f(o[8 * c + 7]) * inv_l));
                if (TRACE && db == 0) t_store = clock64_now();
                flush_block<RAG>(p.out, stage, lane, dst, db);
            }
            if (D % 64) {  // the last 32 columns of D = 96
                uint32_t o[32];
                tmem_ld32(tO + (D / 64) * 64, o);
                release_o();
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    stage_chunk(stage, lane, c, pack_bf16x2(u2f(o[8 * c + 0]) * inv_l, u2f(o[8 * c + 1]) * inv_l),
                                pack_bf16x2(u2f(o[8 * c + 2]) * inv_l, u2f(o[8 * c + 3]) * inv_l),
                                pack_bf16x2(u2f(o[8 * c + 4]) * inv_l, u2f(o[8 * c + 5]) * inv_l),
                                pack_bf16x2(u2f(o[8 * c + 6]) * inv_l, u2f(o[8 * c + 7]) * inv_l));
                flush_block<RAG, 4>(p.out, stage, lane, dst, D / 64);
            }
            if (TRACE && lane == 0) {
                const unsigned long long t_end = clock64_now();
                unsigned long long *r = p.trace + (((size_t)blockIdx.x * p.n_dp + it) * 4 + wq) * kTraceWords;
                r[0] = t_ready;
                r[1] = t_store;
                r[2] = t_end;
                r[3] = g_ready;
                r[4] = ((unsigned long long)g.item << 8) | (uint32_t)wq;
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
#undef BAR
}

template <int D, int LD, int TRACE, bool RAG, bool CAU = false>
static cudaError_t launch_one(const OperandMaps<LD ? kSeqMaps : 1> &maps, const AttnParams &p, int grid,
                              cudaStream_t stream) {
    auto kern = attn_fwd_kernel<D, LD, TRACE, RAG, CAU>;
    // The shared-memory limit is raised once per device and instance: setting a
    // function attribute before every launch makes each launch start much later.
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<D>::kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    kern<<<grid, 512, Cfg<D>::kSmemAlloc, stream>>>(maps, p);
    e = cudaGetLastError();
    if (e == cudaErrorInvalidValue || e == cudaErrorLaunchOutOfResources) {
        // the attribute was lost (for instance by a device reset): set it again once
        configured.fetch_and(~bit, std::memory_order_acq_rel);
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)Cfg<D>::kSmemAlloc)) != cudaSuccess)
            return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
        kern<<<grid, 512, Cfg<D>::kSmemAlloc, stream>>>(maps, p);
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
#define XS_DEFINE_ATTN1_ENTRY(D)                                                                                   \
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

}  // namespace one
}  // namespace xs

