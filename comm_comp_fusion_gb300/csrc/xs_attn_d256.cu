// xs_attn_d256.cu -- the attention kernel's instances for head dimension 256,
// built from the single-query-tile variant (xs_attn1_kernel.cuh): fused scatter
// and head-partitioned output, sequence-partitioned loads, ragged and
// whole-tile sequence lengths, causal.
#include "xs_attn1_kernel.cuh"

namespace xs {
namespace one {
XS_DEFINE_ATTN1_ENTRY(256)
}  // namespace one

cudaError_t launch_attention_d256(const OperandMaps<1> &maps, const AttnParams &p, int grid, cudaStream_t stream) {
    return one::launch_attention_d256(maps, p, grid, stream);
}
cudaError_t launch_ulysses_d256(const OperandMaps<kSeqMaps> &maps, const AttnParams &p, int grid,
                                cudaStream_t stream) {
    return one::launch_ulysses_d256(maps, p, grid, stream);
}
cudaError_t launch_causal_d256(const OperandMaps<1> &maps, const AttnParams &p, int grid, cudaStream_t stream) {
    return one::launch_causal_d256(maps, p, grid, stream);
}
cudaError_t read_error_word_d256(unsigned int *value, bool clear) { return one::read_error_word_d256(value, clear); }

}  // namespace xs
