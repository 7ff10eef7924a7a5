// xs_attn_d128.cu -- the attention kernel's instances for head dimension 128
// (fused scatter and head-partitioned output, sequence-partitioned loads,
// ragged and whole-tile sequence lengths). The kernel itself is in
// xs_attn_kernel.cuh; one translation unit per head dimension keeps the build
// parallel.
#include "xs_attn_kernel.cuh"

namespace xs {

XS_DEFINE_ATTN_ENTRY(128)

cudaError_t launch_attention_traced_d128(const OperandMaps<1> &maps, const AttnParams &p, int grid,
                                         cudaStream_t stream) {
    return launch_one<128, 0, 1, false>(maps, p, grid, stream);
}

}  // namespace xs
