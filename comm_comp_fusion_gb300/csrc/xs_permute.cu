// xs_permute.cu -- the standalone All-to-Alls of Ulysses sequence parallelism
// on one GPU (X-Stage paper, arXiv 2607.23264v1, section 4.3, Figure 5; the
// "A2A-only" variant and the All-to-All half of "Serial" in section 5.3):
//   forward: head-partitioned [P][B][S][Hl][D] -> sequence-partitioned
//            [P][B][Sl][H][D] (the post-attention All-to-All, Figure 5 (d-e));
//   inverse: sequence-partitioned -> head-partitioned (the pre-attention
//            All-to-All, Figure 5 (a-c)).
// Every row of D elements moves whole, so each direction is an HBM-bound
// gather of 16-byte chunks: threads walk the OUTPUT in order (so stores are
// fully coalesced) and fetch each chunk from its source row. Index arithmetic
// uses precomputed multiply-shift division (Granlund and Montgomery, "Division
// by Invariant Integers using Multiplication", 1994).
#include "xs_internal.h"

namespace xs {

// Round-up magic for unsigned n / d with n < 2^31: q = (umulhi(n, m) + n) >> s.
void fastdiv_magic(uint32_t d, uint32_t *m, uint32_t *s) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    *s = l;
    *m = (uint32_t)((((1ull << l) - d) << 32) / d + 1ull);
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, uint32_t m, uint32_t s) {
    return (__umulhi(n, m) + n) >> s;
}

template <bool INV>
__device__ __forceinline__ uint32_t src_chunk_row(uint32_t orow, const PermParams &p) {
    if (INV) {
        // output row orow = ((r * B + b) * S + s) * Hl + hl
        const uint32_t t1 = fdiv(orow, p.mHl, p.sHl);
        const uint32_t hl = orow - t1 * p.Hl;
        const uint32_t t2 = fdiv(t1, p.mS, p.sS);
        const uint32_t s = t1 - t2 * p.S;
        const uint32_t r = fdiv(t2, p.mB, p.sB);
        const uint32_t b = t2 - r * p.B;
        const uint32_t rd = fdiv(s, p.mSl, p.sSl);
        const uint32_t sl = s - rd * p.Sl;
        // source row ((rd * B + b) * Sl + sl) * H + r * Hl + hl
        return ((rd * p.B + b) * p.Sl + sl) * p.H + r * p.Hl + hl;
    }
    // output row orow = ((rd * B + b) * Sl + sl) * H + h
    const uint32_t t1 = fdiv(orow, p.mH, p.sH);
    const uint32_t h = orow - t1 * p.H;
    const uint32_t t2 = fdiv(t1, p.mSl, p.sSl);
    const uint32_t sl = t1 - t2 * p.Sl;
    const uint32_t rd = fdiv(t2, p.mB, p.sB);
    const uint32_t b = t2 - rd * p.B;
    const uint32_t r = fdiv(h, p.mHl, p.sHl);
    const uint32_t hl = h - r * p.Hl;
    const uint32_t s = rd * p.Sl + sl;
    // source row ((r * B + b) * S + s) * Hl + hl
    return ((r * p.B + b) * p.S + s) * p.Hl + hl;
}

__device__ __forceinline__ uint4 ld_stream(const uint4 *ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

constexpr int kPermThreads = 256;
constexpr int kPermUnroll = 4;

// Source chunk of output chunk o: rows of 2^cpr_log2 chunks (POW2), or of
// p.cpr chunks with o below 2^31 (D = 96: 12 chunks per row).
template <bool INV, bool POW2>
__device__ __forceinline__ uint64_t src_chunk(uint64_t o, const PermParams &p) {
    if (POW2) {
        const uint32_t orow = (uint32_t)(o >> p.cpr_log2);
        return ((uint64_t)src_chunk_row<INV>(orow, p) << p.cpr_log2) | (o & ((1u << p.cpr_log2) - 1u));
    }
    const uint32_t orow = fdiv((uint32_t)o, p.mC, p.sC);
    return (uint64_t)src_chunk_row<INV>(orow, p) * p.cpr + ((uint32_t)o - orow * p.cpr);
}

template <bool INV, bool POW2>
__global__ void __launch_bounds__(kPermThreads) a2a_permute_kernel(const uint4 *__restrict__ in,
                                                                   uint4 *__restrict__ out, const PermParams p) {
    const uint64_t total = (uint64_t)p.rows * p.cpr;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (kPermUnroll - 1) * stride < total; i += kPermUnroll * stride) {
        uint4 v[kPermUnroll];
#pragma unroll
        for (int u = 0; u < kPermUnroll; ++u) v[u] = ld_stream(in + src_chunk<INV, POW2>(i + u * stride, p));
#pragma unroll
        for (int u = 0; u < kPermUnroll; ++u) out[i + u * stride] = v[u];
    }
    for (; i < total; i += stride) out[i] = ld_stream(in + src_chunk<INV, POW2>(i, p));
}

cudaError_t launch_permute(const void *in, void *out, const PermParams &p, bool inverse, int num_sms,
                           cudaStream_t stream) {
    const uint64_t total = (uint64_t)p.rows * p.cpr;
    uint64_t blocks = (total + kPermThreads - 1) / kPermThreads;
    const uint64_t cap = (uint64_t)num_sms * (2048 / kPermThreads);  // one full wave of resident threads
    if (blocks > cap) blocks = cap;
    if (blocks == 0) return cudaSuccess;
    const bool pow2 = (p.cpr & (p.cpr - 1u)) == 0u;
    auto kern = inverse ? (pow2 ? a2a_permute_kernel<true, true> : a2a_permute_kernel<true, false>)
                        : (pow2 ? a2a_permute_kernel<false, true> : a2a_permute_kernel<false, false>);
    kern<<<(unsigned)blocks, kPermThreads, 0, stream>>>(static_cast<const uint4 *>(in), static_cast<uint4 *>(out), p);
    return cudaGetLastError();
}

}  // namespace xs
