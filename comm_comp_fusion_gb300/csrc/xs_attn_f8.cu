// xs_attn_f8.cu -- the attention kernel's instances with E4M3 inputs, D = 128
// (F8 = 1: E4M3 queries and keys; F8 = 2: E4M3 queries, keys and values), for
// the fused scatter and the head-partitioned output, ragged and whole-tile
// sequence lengths. Its own translation unit keeps the build parallel.
#include "xs_attn_kernel.cuh"

namespace xs {

template <int F8>
static cudaError_t launch_f8(const OperandMaps<1> &maps, const AttnParams &p, int grid, cudaStream_t stream) {
    return p.kv_tail < 128 ? launch_one<128, 0, 0, true, false, F8>(maps, p, grid, stream)
                           : launch_one<128, 0, 0, false, false, F8>(maps, p, grid, stream);
}

cudaError_t launch_attention_f8_d128(int f8, const OperandMaps<1> &maps, const AttnParams &p, int grid,
                                     cudaStream_t stream) {
    if (f8 == 1) return launch_f8<1>(maps, p, grid, stream);
    if (f8 == 2) return launch_f8<2>(maps, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t read_error_word_f8(unsigned int *value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_xs_error, sizeof(unsigned int));
    if (e == cudaSuccess && clear && *value) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_xs_error, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace xs
