// xs_attn.cu -- host side of the attention kernel: the workspace size, dispatch
// to the per-head-dimension instances (xs_attn_d64.cu, xs_attn_d96.cu,
// xs_attn_d128.cu, xs_attn_d256.cu), the bounded-wait self-test and the device
// error words. The work schedule is in xs_schedule.cpp.
#include "xs_attn_kernel.cuh"

namespace xs {

size_t attn_workspace_bytes(int n_items, int n_kv, int D, int num_sms) {
    (void)n_kv;
    const size_t rec = ((size_t)2 * num_sms * partial_record_bytes(D) + 255) & ~(size_t)255;
    // four epilogue warps' arrival counters (64-bit words) per tile
    const size_t cnt = ((size_t)n_items * 4 * tiles_per_item(D) * sizeof(unsigned long long) + 255) & ~(size_t)255;
    return rec + cnt;
}

cudaError_t launch_attention(int D, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                             cudaStream_t stream) {
    if (D == 256) return launch_attention_d256(maps, p, grid, stream);
    if (D == 128) return launch_attention_d128(maps, p, grid, stream);
    if (D == 96) return launch_attention_d96(maps, p, grid, stream);
    if (D == 64) return launch_attention_d64(maps, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attention_traced(int D, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                                    cudaStream_t stream) {
    if (D == 128 && p.kv_tail == 128) return launch_attention_traced_d128(maps, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_causal(int D, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                          cudaStream_t stream) {
    if (D == 256) return launch_causal_d256(maps, p, grid, stream);
    if (D == 128) return launch_causal_d128(maps, p, grid, stream);
    if (D == 96) return launch_causal_d96(maps, p, grid, stream);
    if (D == 64) return launch_causal_d64(maps, p, grid, stream);
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
