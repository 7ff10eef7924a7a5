// xs_attn_d64.cu -- the attention kernel's instances for head dimension 64
// (fused scatter and head-partitioned output, sequence-partitioned loads,
// ragged and whole-tile sequence lengths). The kernel itself is in
// xs_attn_kernel.cuh; one translation unit per head dimension keeps the build
// parallel.
#include "xs_attn_kernel.cuh"

namespace xs {

XS_DEFINE_ATTN_ENTRY(64)

}  // namespace xs
