// xs_attn.cu -- host side of the attention kernel: the work schedule, the
// workspace size, dispatch to the per-head-dimension instances
// (xs_attn_d64.cu, xs_attn_d96.cu, xs_attn_d128.cu, xs_attn_d256.cu), the bounded-wait
// self-test and the device error words.
#include "xs_attn_kernel.cuh"

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

size_t attn_workspace_bytes(int n_items, int n_kv, int D, int num_sms) {
    (void)n_kv;
    const size_t rec = ((size_t)2 * num_sms * partial_record_bytes(D) + 255) & ~(size_t)255;
    // four epilogue warps' arrival counters per tile
    const size_t cnt = ((size_t)n_items * 4 * tiles_per_item(D) * sizeof(uint32_t) + 255) & ~(size_t)255;
    return rec + cnt;
}

cudaError_t launch_attention(int D, int epi, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                             cudaStream_t stream) {
    if (D == 256) return launch_attention_d256(epi, maps, p, grid, stream);
    if (D == 128) return launch_attention_d128(epi, maps, p, grid, stream);
    if (D == 96) return launch_attention_d96(epi, maps, p, grid, stream);
    if (D == 64) return launch_attention_d64(epi, maps, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attention_traced(int D, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                                    cudaStream_t stream) {
    if (D == 128 && p.kv_tail == 128) return launch_attention_traced_d128(maps, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_causal(int D, int epi, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                          cudaStream_t stream) {
    if (D == 256) return launch_causal_d256(epi, maps, p, grid, stream);
    if (D == 128) return launch_causal_d128(epi, maps, p, grid, stream);
    if (D == 96) return launch_causal_d96(epi, maps, p, grid, stream);
    if (D == 64) return launch_causal_d64(epi, maps, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_ulysses(int D, const OperandMaps<kSeqMaps> &maps, const AttnParams &p, int grid,
                           cudaStream_t stream) {
    if (D == 256) return launch_ulysses_d256(maps, p, grid, stream);
    if (D == 128) return launch_ulysses_d128(maps, p, grid, stream);
    if (D == 96) return launch_ulysses_d96(maps, p, grid, stream);
    if (D == 64) return launch_ulysses_d64(maps, p, grid, stream);
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ bounded-wait self-test

__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar_storage;
    __shared__ uint32_t abort_word;
    const uint32_t bar = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        abort_word = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on this barrier: the wait must run out and return.
        (void)wait_slow(bar, 0u, &abort_word, kSiteSelftest, limit_ns);
    }
    __syncthreads();
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

// The OR of every translation unit's error word (this one holds the
// self-test's), each cleared if `clear`.
cudaError_t read_device_error(unsigned int *value, bool clear, cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned int all = 0, w = 0;
    e = cudaMemcpyFromSymbol(&w, g_xs_error, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    all |= w;
    if (clear && w) {
        const unsigned int zero = 0;
        if ((e = cudaMemcpyToSymbol(g_xs_error, &zero, sizeof(unsigned int))) != cudaSuccess) return e;
    }
    cudaError_t (*const per_d[])(unsigned int *, bool) = {read_error_word_d64, read_error_word_d96,
                                                          read_error_word_d128, read_error_word_d256,
                                                          read_error_word_f8};
    for (auto fn : per_d) {
        if ((e = fn(&w, clear)) != cudaSuccess) return e;
        all |= w;
    }
    *value = all;
    return cudaSuccess;
}

}  // namespace xs
