// xs_attn_d96.cu -- the attention kernel's instances for head dimension 96
// (fused scatter and head-partitioned output, sequence-partitioned loads,
// ragged and whole-tile sequence lengths). The kernel itself is in
// xs_attn_kernel.cuh; one translation unit per head dimension keeps the build
// parallel.
#include "xs_attn_kernel.cuh"

namespace xs {

XS_DEFINE_ATTN_ENTRY(96)

}  // namespace xs
